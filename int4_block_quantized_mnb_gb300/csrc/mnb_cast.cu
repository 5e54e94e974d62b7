// mnb_cast.cu -- the fp16 -> bf16 narrowing as a launch of its own: the
// "staged route" of a bf16 model, where the GEMV writes an fp16 staging buffer
// and a separate kernel narrows it, against which the GEMV's direct bf16 store
// is measured.  ("perf(cuda): let the split-K decode GEMV store bf16
// directly", onnx-genai PR 1550, paragraphs 1-3: the cast_half launch per node
// that the direct store removes.)
//
// The conversion is the one the GEMV epilogue applies (mnb_narrow.cuh), so the
// staged route's result equals the direct store bit for bit.

#include "mnb.h"
#include "mnb_narrow.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <string>

namespace mnb {

int fail(int status, const std::string& detail);
int cuda_fail(cudaError_t e, const char* what);
extern std::atomic<unsigned long long> g_counters[MNB_NUM_COUNTERS];

namespace {

__device__ __forceinline__ uint32_t narrow(uint32_t h) {
  return narrow_f16_bits_to_bf16(static_cast<uint16_t>(h));
}

__device__ __forceinline__ uint32_t narrow2(uint32_t w) {
  return narrow(w & 0xFFFFu) | (narrow(w >> 16) << 16);
}

// Grid-stride narrowing; 16-byte vectors when both arrays are 16-byte aligned
// (a launch-uniform choice), the tail and unaligned arrays element by element.
__global__ void __launch_bounds__(256) cast_f16_bf16_kernel(const uint16_t* src, uint16_t* dst,
                                                            size_t n, int vec) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  size_t done = 0;
  if (vec) {
    const size_t n8 = n / 8;
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (size_t v = i0; v < n8; v += stride) {
      const uint4 a = s[v];
      d[v] = make_uint4(narrow2(a.x), narrow2(a.y), narrow2(a.z), narrow2(a.w));
    }
    done = n8 * 8;
  }
  for (size_t e = done + i0; e < n; e += stride) dst[e] = static_cast<uint16_t>(narrow(src[e]));
}

}  // namespace
}  // namespace mnb

extern "C" int mnb_cast_f16_to_bf16(const void* src, void* dst, size_t n, void* stream) {
  using namespace mnb;
  if (n == 0) return MNB_OK;
  if (!src || !dst) return fail(MNB_ERR_NULL, "src and dst are required");
  const uintptr_t s = reinterpret_cast<uintptr_t>(src), d = reinterpret_cast<uintptr_t>(dst);
  if ((s & 1u) || (d & 1u)) return fail(MNB_ERR_ALIGN, "src and dst must be 2-byte aligned");
  const uintptr_t bytes = static_cast<uintptr_t>(n) * 2;
  if (s != d && s < d + bytes && d < s + bytes)
    return fail(MNB_ERR_ALIAS, "src and dst overlap (only exact in-place narrowing is allowed)");
  const int vec = ((s | d) & 15u) == 0 ? 1 : 0;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  const size_t per_block = static_cast<size_t>(256) * (vec ? 8 : 1);
  const size_t want = (n + per_block - 1) / per_block;
  const unsigned blocks = static_cast<unsigned>(
      std::max<size_t>(1, std::min<size_t>(want, static_cast<size_t>(std::max(sms, 1)) * 8)));
  cast_f16_bf16_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), n, vec);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "cast kernel launch");
  g_counters[14].fetch_add(1, std::memory_order_relaxed);
  return MNB_OK;
}
