// mnb_narrow.cuh -- the fp16 -> bf16 narrowing shared by the GEMV epilogue and
// the separate narrowing kernel: fp16 -> fp32 exactly, round-to-nearest-even
// to bf16; a NaN becomes the quiet NaN 0x7FC0 with its sign.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace mnb {

__device__ __forceinline__ uint16_t narrow_f16_bits_to_bf16(uint16_t h) {
  if ((h & 0x7C00u) == 0x7C00u && (h & 0x03FFu) != 0)
    return static_cast<uint16_t>((h & 0x8000u) | 0x7FC0u);
  return __bfloat16_as_ushort(__float2bfloat16_rn(__half2float(__ushort_as_half(h))));
}

}  // namespace mnb
