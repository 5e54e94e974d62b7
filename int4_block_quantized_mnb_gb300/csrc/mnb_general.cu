// mnb_general.cu -- the MatMulNBits decode GEMV for the other formats of the
// family: block sizes 16, 32, 64 and 128, with per-block zero-points or
// without them (symmetric: every zero-point is 8).
//
// Sources: the dequantized dot product y[m,n] = sum_k x[m,k] (q[n,k] -
// zp[n,k/B]) s[n,k/B], rounded once to fp16 and, on the bf16 arm, narrowed
// by a second rounding ("perf(cuda): let the split-K decode GEMV store bf16
// directly", first two paragraphs); the symmetric dequant with the +8 bias
// when a weight has no zero-point ("PORT-1 (offline bias+interleave) --
// measured NO-GO on the multicol asymmetric-zp GEMV", "Why the premise fails
// here", point 1).  Block sizes other than 32 take the same packed layout
// with the block size as a parameter: scales [N][K/B], zero-points
// [N][ceil(K/B/2)] with the low nibble holding the even block.
//
// Kernel shape.  A CTA of W = P * S warps takes P row groups (four rows per
// warp for M <= 2; sixteen above, see gemv_general_wide); the S warps of a group split K into S contiguous ranges
// of 32-k chunks, and lane l of a warp takes chunks l, l + 32, ... of its
// range.  A chunk of one row is 16 bytes of codes (one vector load) and its
// block's scale and zero-point (two for block 16, where a chunk spans two
// blocks), dequantized once into registers for all M batch rows.  Where each
// lane has at least four chunks, the activations (up to 96 KB) are staged
// once per CTA in shared memory, already regrouped into the pairs the
// dequant produces; otherwise they are read through the read-only cache.  Dequant is the exact one of mnb_dequant.cuh; each lane keeps
// fp32 sums per (row, m), reduced across lanes by a fixed shuffle tree and
// across the S warps through shared memory in warp order.
#include "mnb.h"
#include "mnb_launch.cuh"
#include "mnb_dequant.cuh"
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

constexpr int kGenWarps = 8;                 // warps per CTA at most

struct GenParams {
  const uint16_t* x;
  const uint8_t* q;
  const uint16_t* scales;
  const uint8_t* zp;                         // nullptr: symmetric
  void* y;
  int N, K;
  int chunks;                                // K / 32
  int blocks;                                // K / B
  int zstride;                               // zero-point bytes per row
  int bshift;                                // log2(B / 32) for B >= 32
  int split;                                 // S: warps per row group
  int pairs;                                 // P: row groups per CTA
  int out_bf16;
  int x_aligned;                             // x is 16-byte aligned
  int x_smem;                                // activations staged in shared memory
};

__device__ __forceinline__ void gen_store(void* y, size_t idx, float v, int out_bf16) {
  const __half h = __float2half_rn(v);
  if (out_bf16)
    static_cast<uint16_t*>(y)[idx] = narrow_f16_bits_to_bf16(__half_as_ushort(h));
  else
    static_cast<__half*>(y)[idx] = h;
}

__device__ __forceinline__ float f16_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// (1024 + z, 64 + z) in both halves: the bias words of zero-point z.
__device__ __forceinline__ void zp_bias(uint32_t z, uint32_t& lo, uint32_t& hi) {
  lo = z * 0x00010001u + 0x64006400u;
  hi = z * 0x00100010u + 0x54005400u;
}

// 64 bytes of activations x[m][32c .. 32c + 32), as four 8-k groups already
// regrouped into the (k, k + 4) pairs the dequant produces.
__device__ __forceinline__ void load_x_chunk(const GenParams& p, int m, int c, uint4 (&xr)[4]) {
  const uint16_t* src = p.x + static_cast<size_t>(m) * p.K + 32 * c;
  if (p.x_aligned) {
    const uint4* v = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int g = 0; g < 4; ++g) xr[g] = pair_k4(__ldg(v + g));
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint16_t* e = src + 8 * g;
      uint4 v;
      v.x = __ldg(e + 0) | (static_cast<uint32_t>(__ldg(e + 1)) << 16);
      v.y = __ldg(e + 2) | (static_cast<uint32_t>(__ldg(e + 3)) << 16);
      v.z = __ldg(e + 4) | (static_cast<uint32_t>(__ldg(e + 5)) << 16);
      v.w = __ldg(e + 6) | (static_cast<uint32_t>(__ldg(e + 7)) << 16);
      xr[g] = pair_k4(v);
    }
  }
}

// q - zp of one 8-k group word as the pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7).
__device__ __forceinline__ void dequant_word(uint32_t word, uint32_t zl, uint32_t zh,
                                             uint32_t* d) {
  const uint32_t w8 = word >> 8;
  d[0] = hsub2(and_or(word, 0x000F000Fu, 0x64006400u), zl);
  d[1] = hsub2(and_or(word, 0x00F000F0u, 0x54005400u), zh);
  d[2] = hsub2(and_or(w8, 0x000F000Fu, 0x64006400u), zl);
  d[3] = hsub2(and_or(w8, 0x00F000F0u, 0x54005400u), zh);
}

// acc + the dot product of one dequantized group with one activation group.
__device__ __forceinline__ float group_dot(const uint32_t* d, uint4 xv, float acc) {
  acc = fma2_f16_f32(xv.x, d[0], acc);
  acc = fma2_f16_f32(xv.y, d[1], acc);
  acc = fma2_f16_f32(xv.z, d[2], acc);
  acc = fma2_f16_f32(xv.w, d[3], acc);
  return acc;
}

// acc + one row's chunk (dequantized d, four groups) against one batch row's
// activations: one block sum times its scale, or two for block 16 (words 0-1
// are block 2c, words 2-3 block 2c + 1).
template <bool kB16>
__device__ __forceinline__ void chunk_dot(const uint32_t* d, const uint4 (&xr)[4], float s0,
                                          float s1, float& acc) {
  if (kB16) {
    const float b0 = group_dot(d + 4, xr[1], group_dot(d + 0, xr[0], 0.f));
    const float b1 = group_dot(d + 12, xr[3], group_dot(d + 8, xr[2], 0.f));
    acc = fmaf(b0, s0, acc);
    acc = fmaf(b1, s1, acc);
  } else {
    float b = group_dot(d + 0, xr[0], 0.f);
    b = group_dot(d + 4, xr[1], b);
    b = group_dot(d + 8, xr[2], b);
    b = group_dot(d + 12, xr[3], b);
    acc = fmaf(b, s0, acc);
  }
}

// Rows per warp: four (lanes over chunks) for M <= 2; sixteen for M > 2,
// where lane (q, rr) takes rows rr and rr + 8 and every fourth chunk, so the
// eight lanes of a quarter warp share each activation load.
constexpr int gen_rows(int M) { return M <= 2 ? 4 : 16; }

// Staged activations at most; larger batches read them from global memory.
constexpr int kGenXSmemMax = 96 * 1024;

template <int M, bool kB16>
__global__ void __launch_bounds__(kGenWarps * 32, 2) gemv_general_kernel(const GenParams p) {
  constexpr int RW = gen_rows(M);
  // staged activations, [m][group g][chunk c] of regrouped 8-k groups, so the
  // 32 lanes of a warp (consecutive chunks) read consecutive 16-byte words
  extern __shared__ uint4 xs[];
  __shared__ float red[kGenWarps][RW][M];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = warp / p.split;
  const int part = warp - grp * p.split;
  const int row0 = (blockIdx.x * p.pairs + grp) * RW;
  const int c_begin = static_cast<int>(static_cast<long long>(part) * p.chunks / p.split);
  const int c_end = static_cast<int>(static_cast<long long>(part + 1) * p.chunks / p.split);
  const int nrows = max(0, min(RW, p.N - row0));

  // programmatic dependent launch: let the next grid launch, then wait for
  // the preceding grid's writes before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (p.x_smem) {
    const int per_m = 4 * p.chunks;
    for (int e = threadIdx.x; e < M * per_m; e += blockDim.x) {
      const int m = e / per_m;
      const int rem = e - m * per_m;
      const int c = rem >> 2, g = rem & 3;
      const uint16_t* src = p.x + static_cast<size_t>(m) * p.K + 32 * c + 8 * g;
      uint4 v;
      if (p.x_aligned) {
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        v.x = __ldg(src + 0) | (static_cast<uint32_t>(__ldg(src + 1)) << 16);
        v.y = __ldg(src + 2) | (static_cast<uint32_t>(__ldg(src + 3)) << 16);
        v.z = __ldg(src + 4) | (static_cast<uint32_t>(__ldg(src + 5)) << 16);
        v.w = __ldg(src + 6) | (static_cast<uint32_t>(__ldg(src + 7)) << 16);
      }
      xs[(m * 4 + g) * p.chunks + c] = pair_k4(v);
    }
    __syncthreads();
  }

  float acc[RW][M];
#pragma unroll
  for (int i = 0; i < RW; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[i][m] = 0.f;

  if (nrows > 0) {
#pragma unroll 2
    for (int c = c_begin + lane; c < c_end; c += 32) {
      uint4 w[RW];
      float s0[RW], s1[RW];
      uint32_t zl0[RW], zh0[RW], zl1[RW], zh1[RW];
#pragma unroll
      for (int i = 0; i < RW; ++i) {
        const int r = min(row0 + i, p.N - 1);       // missing rows repeat the last one
        w[i] = __ldg(reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(r) * (p.K / 2)) + c);
        const uint16_t* srow = p.scales + static_cast<size_t>(r) * p.blocks;
        uint32_t z0 = 8, z1 = 8;
        if (kB16) {                                   // blocks 2c and 2c + 1
          s0[i] = f16_bits_to_float(__ldg(srow + 2 * c));
          s1[i] = f16_bits_to_float(__ldg(srow + 2 * c + 1));
          if (p.zp) {
            const uint32_t zb = __ldg(p.zp + static_cast<size_t>(r) * p.zstride + c);
            z0 = zb & 0xFu;
            z1 = zb >> 4;
          }
        } else {                                      // block c >> bshift
          const int b = c >> p.bshift;
          s0[i] = f16_bits_to_float(__ldg(srow + b));
          s1[i] = 0.f;
          if (p.zp) {
            const uint32_t zb = __ldg(p.zp + static_cast<size_t>(r) * p.zstride + (b >> 1));
            z0 = (b & 1) ? (zb >> 4) : (zb & 0xFu);
          }
          z1 = z0;
        }
        zp_bias(z0, zl0[i], zh0[i]);
        zp_bias(z1, zl1[i], zh1[i]);
      }
      if constexpr (M <= 2) {
        // small batch: the activations of every batch row first, then one
        // row at a time dequantized and used for all of them
        uint4 xr[M][4];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          if (p.x_smem) {
#pragma unroll
            for (int g = 0; g < 4; ++g) xr[m][g] = xs[(m * 4 + g) * p.chunks + c];
          } else {
            load_x_chunk(p, m, c, xr[m]);
          }
        }
#pragma unroll
        for (int i = 0; i < RW; ++i) {
          uint32_t d[16];
          dequant_word(w[i].x, zl0[i], zh0[i], d + 0);
          dequant_word(w[i].y, zl0[i], zh0[i], d + 4);
          dequant_word(w[i].z, zl1[i], zh1[i], d + 8);
          dequant_word(w[i].w, zl1[i], zh1[i], d + 12);
#pragma unroll
          for (int m = 0; m < M; ++m) chunk_dot<kB16>(d, xr[m], s0[i], s1[i], acc[i][m]);
        }
      } else {
        // each row's chunk is dequantized once and used for every batch row
        uint32_t d[RW][16];
#pragma unroll
        for (int i = 0; i < RW; ++i) {
          dequant_word(w[i].x, zl0[i], zh0[i], d[i] + 0);
          dequant_word(w[i].y, zl0[i], zh0[i], d[i] + 4);
          dequant_word(w[i].z, zl1[i], zh1[i], d[i] + 8);
          dequant_word(w[i].w, zl1[i], zh1[i], d[i] + 12);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          uint4 xr[4];
          if (p.x_smem) {
#pragma unroll
            for (int g = 0; g < 4; ++g) xr[g] = xs[(m * 4 + g) * p.chunks + c];
          } else {
            load_x_chunk(p, m, c, xr);
          }
#pragma unroll
          for (int i = 0; i < RW; ++i) chunk_dot<kB16>(d[i], xr, s0[i], s1[i], acc[i][m]);
        }
      }
    }
  }

  // lanes, in a fixed butterfly order
#pragma unroll
  for (int i = 0; i < RW; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[i][m];
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
      acc[i][m] = v;
    }
  if (p.split > 1) {
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < RW; ++i)
#pragma unroll
        for (int m = 0; m < M; ++m) red[warp][i][m] = acc[i][m];
    }
    __syncthreads();
    if (part != 0) return;
    // the K ranges of the group, in range order
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float v = red[warp][i][m];
        for (int j = 1; j < p.split; ++j) v += red[warp + j][i][m];
        acc[i][m] = v;
      }
  }
  // lane i * M + m stores output (row0 + i, batch row m)
#pragma unroll
  for (int i = 0; i < RW; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m)
      if (lane == i * M + m && i < nrows)
        gen_store(p.y, static_cast<size_t>(m) * p.N + row0 + i, acc[i][m], p.out_bf16);
}

// M > 2: lane (q, rr) = (lane >> 3, lane & 7) takes weight rows rr and rr + 8
// of the warp's 16 and chunks q, q + 4, ... of the warp's K range.  Each row's
// chunk is dequantized once for all M activation rows, and one activation load
// (the same address for the eight lanes of a quarter warp) serves both rows.
template <int M, bool kB16>
__global__ void __launch_bounds__(kGenWarps * 32, 2) gemv_general_wide(const GenParams p) {
  extern __shared__ uint4 xs[];
  __shared__ float red[kGenWarps][2][M][8];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rr = lane & 7;
  const int q4 = lane >> 3;
  const int grp = warp / p.split;
  const int part = warp - grp * p.split;
  const int row0 = (blockIdx.x * p.pairs + grp) * 16;
  const int c_begin = static_cast<int>(static_cast<long long>(part) * p.chunks / p.split);
  const int c_end = static_cast<int>(static_cast<long long>(part + 1) * p.chunks / p.split);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (p.x_smem) {
    const int per_m = 4 * p.chunks;
    for (int e = threadIdx.x; e < M * per_m; e += blockDim.x) {
      const int m = e / per_m;
      const int rem = e - m * per_m;
      const int c = rem >> 2, g = rem & 3;
      const uint16_t* src = p.x + static_cast<size_t>(m) * p.K + 32 * c + 8 * g;
      uint4 v;
      if (p.x_aligned) {
        v = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        v.x = __ldg(src + 0) | (static_cast<uint32_t>(__ldg(src + 1)) << 16);
        v.y = __ldg(src + 2) | (static_cast<uint32_t>(__ldg(src + 3)) << 16);
        v.z = __ldg(src + 4) | (static_cast<uint32_t>(__ldg(src + 5)) << 16);
        v.w = __ldg(src + 6) | (static_cast<uint32_t>(__ldg(src + 7)) << 16);
      }
      xs[(m * 4 + g) * p.chunks + c] = pair_k4(v);
    }
    __syncthreads();
  }

  float acc[2][M];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[i][m] = 0.f;
  const int ra = min(row0 + rr, p.N - 1), rb = min(row0 + rr + 8, p.N - 1);
  if (row0 < p.N) {
#pragma unroll 2
    for (int c = c_begin + q4; c < c_end; c += 4) {
      uint4 w[2];
      float s0[2], s1[2];
      uint32_t zl0[2], zh0[2], zl1[2], zh1[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = i ? rb : ra;
        w[i] = __ldg(reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(r) * (p.K / 2)) + c);
        const uint16_t* srow = p.scales + static_cast<size_t>(r) * p.blocks;
        uint32_t z0 = 8, z1 = 8;
        if (kB16) {
          s0[i] = f16_bits_to_float(__ldg(srow + 2 * c));
          s1[i] = f16_bits_to_float(__ldg(srow + 2 * c + 1));
          if (p.zp) {
            const uint32_t zb = __ldg(p.zp + static_cast<size_t>(r) * p.zstride + c);
            z0 = zb & 0xFu;
            z1 = zb >> 4;
          }
        } else {
          const int b = c >> p.bshift;
          s0[i] = f16_bits_to_float(__ldg(srow + b));
          s1[i] = 0.f;
          if (p.zp) {
            const uint32_t zb = __ldg(p.zp + static_cast<size_t>(r) * p.zstride + (b >> 1));
            z0 = (b & 1) ? (zb >> 4) : (zb & 0xFu);
          }
          z1 = z0;
        }
        zp_bias(z0, zl0[i], zh0[i]);
        zp_bias(z1, zl1[i], zh1[i]);
      }
      uint32_t d[2][16];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        dequant_word(w[i].x, zl0[i], zh0[i], d[i] + 0);
        dequant_word(w[i].y, zl0[i], zh0[i], d[i] + 4);
        dequant_word(w[i].z, zl1[i], zh1[i], d[i] + 8);
        dequant_word(w[i].w, zl1[i], zh1[i], d[i] + 12);
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        uint4 xr[4];
        if (p.x_smem) {
#pragma unroll
          for (int g = 0; g < 4; ++g) xr[g] = xs[(m * 4 + g) * p.chunks + c];
        } else {
          load_x_chunk(p, m, c, xr);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) chunk_dot<kB16>(d[i], xr, s0[i], s1[i], acc[i][m]);
      }
    }
  }
  // the four chunk lanes of each row, in a fixed order
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[i][m];
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
      acc[i][m] = v;
    }
  if (p.split > 1) {
    if (q4 == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int m = 0; m < M; ++m) red[warp][i][m][rr] = acc[i][m];
    }
    __syncthreads();
    if (part != 0) return;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float v = red[warp][i][m][rr];
        for (int j = 1; j < p.split; ++j) v += red[warp + j][i][m][rr];
        acc[i][m] = v;
      }
  }
  if (q4 == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = row0 + rr + 8 * i;
      if (r < p.N) {
#pragma unroll
        for (int m = 0; m < M; ++m)
          gen_store(p.y, static_cast<size_t>(m) * p.N + r, acc[i][m], p.out_bf16);
      }
    }
  }
}

using GenFn = void (*)(const GenParams);

template <bool kB16>
GenFn general_kernel_for(int M) {
  switch (M) {
    case 1: return &gemv_general_kernel<1, kB16>;
    case 2: return &gemv_general_kernel<2, kB16>;
    case 3: return &gemv_general_wide<3, kB16>;
    case 4: return &gemv_general_wide<4, kB16>;
    case 5: return &gemv_general_wide<5, kB16>;
    case 6: return &gemv_general_wide<6, kB16>;
    case 7: return &gemv_general_wide<7, kB16>;
    default: return &gemv_general_wide<8, kB16>;
  }
}

int log2_exact(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return s;
}

}  // namespace

// Warps per row group (S) without a requested split: the fewest of 1, 2, 4,
// 8 that give every SM a CTA (two are resident per SM, so this stays within
// one wave where the rows allow), and no more than leave every chunk lane of a
// warp (32 for M <= 2, 4 above) at least one chunk.  A requested split_k becomes S (at most 8).
int general_split(int M, int N, int K, int split_k, int sms) {
  if (split_k > 0) return std::min(split_k, kGenWarps);
  const int chunks = K / 32;
  const int rows_warp = gen_rows(M);
  const int chunk_lanes = M <= 2 ? 32 : 4;      // lanes of a warp that split its chunks
  int s = 1;
  while (s < kGenWarps && s * 2 * chunk_lanes <= chunks) {
    const long long rows_cta = static_cast<long long>(rows_warp) * (kGenWarps / s);
    const long long ctas = (N + rows_cta - 1) / rows_cta;
    if (ctas >= sms) break;
    s *= 2;
  }
  return s;
}

// Launches the general-format kernel; arguments are validated by the caller
// (block in {16, 32, 64, 128}, K a multiple of 32 and of the block size).
int launch_general(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                   void* y, int M, int N, int K, int block, int out_bf16, int split_k, int sms,
                   cudaStream_t stream, LaunchDesc* query) {
  GenParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.q = qweight;
  p.scales = static_cast<const uint16_t*>(scales);
  p.zp = zp;
  p.y = y;
  p.N = N;
  p.K = K;
  p.chunks = K / 32;
  p.blocks = K / block;
  p.zstride = (p.blocks + 1) / 2;
  p.bshift = block >= 32 ? log2_exact(block / 32) : 0;
  p.split = general_split(M, N, K, split_k, sms);
  p.pairs = kGenWarps / p.split;
  p.out_bf16 = out_bf16;
  p.x_aligned = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  const size_t x_bytes = static_cast<size_t>(M) * K * 2;
  // staging pays where each chunk lane of a warp has at least four chunks
  p.x_smem = x_bytes <= static_cast<size_t>(kGenXSmemMax) &&
             p.chunks / p.split >= 4 * (M <= 2 ? 32 : 4);
  const long long rows_cta = static_cast<long long>(gen_rows(M)) * p.pairs;
  const long long grid = (N + rows_cta - 1) / rows_cta;
  if (grid > 0x7FFFFFFFLL) return fail(MNB_ERR_SHAPE, "N too large");

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(p.pairs * p.split * 32));
  cfg.dynamicSmemBytes = p.x_smem ? x_bytes : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const GenFn fn = block == 16 ? general_kernel_for<true>(M) : general_kernel_for<false>(M);
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGenXSmemMax);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(general format)");
  if (query) {
    query->fn = reinterpret_cast<const void*>(fn);
    query->name = M <= 2 ? "general-format kernel (rows of a warp over chunks)"
                         : "general-format kernel (two rows per lane)";
    query->counter = 15;
    query->grid = cfg.gridDim.x;
    query->threads = cfg.blockDim.x;
    query->smem = cfg.dynamicSmemBytes;
    return MNB_OK;
  }
  void* args[1] = {&p};
  e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC(general format)");
  g_counters[15].fetch_add(1, std::memory_order_relaxed);
  return MNB_OK;
}

}  // namespace mnb
