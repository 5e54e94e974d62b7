// mnb_dequant.cuh -- the exact 4-bit dequant shared by the GEMV kernels, and
// the fp16 tensor-core fragment product their tensor-core math uses.
//
// Two codes of a 32-bit word (nibbles k and k + 4 of one 8-k group) become an
// fp16 pair by OR-ing them into the mantissa of a power of two: low nibbles
// under 1024 (0x6400), high nibbles under 64 (0x5400, ulp 1/16, so the
// nibble's <<4 position reads as q).  Subtracting (1024 + zp) or (64 + zp)
// then gives q - zp exactly, and each product with an fp16 activation is
// exact in fp32.
#pragma once

#include <cstdint>

namespace mnb {

// (a & mask) | magic in one LOP3 (the compiler splits it in two when both
// constants are immediates).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}

// (q - zp) for two codes: packed fp16 subtraction of magic-biased values.
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// c + a.lo*b.lo + a.hi*b.hi; f16 sources, f32 accumulation, exact products.
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n .reg .f16 a0, a1, b0, b1;\n .reg .f32 t;\n"
      " mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
      " fma.rn.f32.f16 t, a0, b0, %3;\n fma.rn.f32.f16 %0, a1, b1, t;\n}\n"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

// Eight activations k0..k7 (packed two per word) regrouped into the B
// fragment pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7).
__device__ __forceinline__ uint4 pair_k4(uint4 v) {
  uint4 o;
  o.x = __byte_perm(v.x, v.z, 0x5410);
  o.y = __byte_perm(v.x, v.z, 0x7632);
  o.z = __byte_perm(v.y, v.w, 0x5410);
  o.w = __byte_perm(v.y, v.w, 0x7632);
  return o;
}

// D = A * B + C for one m16n8k16 tile, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// D = A * B for one m16n8k16 tile (zero accumulator input).
__device__ __forceinline__ void mma_16816_zero(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm("{\n .reg .f32 z;\n mov.f32 z, 0f00000000;\n"
      " mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {z,z,z,z};\n}"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace mnb
