// mnb_launch.cuh -- the description of one kernel launch, filled instead of
// launching when the C ABI is asked what a call would run
// (mnb_gemv_launch_info).
#pragma once

#include <cstddef>

namespace mnb {

struct LaunchDesc {
  const void* fn = nullptr;  // the kernel's host-side handle
  const char* name = "";     // kernel family
  int counter = -1;          // mnb_debug_counters index of the family, -1 if none
  unsigned grid = 0;         // CTAs
  unsigned threads = 0;      // threads per CTA
  unsigned cluster = 1;      // CTAs per cluster
  size_t smem = 0;           // dynamic shared memory per CTA
};

}  // namespace mnb
