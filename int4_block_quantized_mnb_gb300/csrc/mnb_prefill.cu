// mnb_prefill.cu -- the MatMulNBits GEMM for more than 8 activation rows
// (prefill): y[m,n] = sum_k x[m,k] (q[n,k] - zp[n,k/B]) s[n,k/B], M > 8, with
// the decode GEMV's epilogue (one rounding to fp16, and on the bf16 arm the
// narrowing of that fp16 value) -- "perf(cuda): let the split-K decode GEMV
// store bf16 directly", the paragraph on the prefill path, which lacked the
// narrowing store.  Block sizes 32, 64 and 128, with or without zero-points.
//
// Tensor-core form.  Weight rows are the M dimension of mma.sync m16n8k16
// and activation rows its N dimension: a CTA takes 128 weight rows (16 per
// warp) by 64 activation rows (8 tiles of 8 per warp).  The A operand is the
// exact fp16 q - zp of mnb_dequant.cuh: lane (g, t) holds code word t of
// chunk c for weight rows g and g + 8, whose pairs (k0,k4) (k1,k5) feed one
// fragment product and (k2,k6) (k3,k7) the next; the activations are staged
// per 256-k stage in shared memory, regrouped into the same pairs, so one
// 16-byte load gives lane (g, t) the B operand of both products for
// activation row g of a tile.  The products are exact and the fragment sums
// fp32; each quantization block's sum D starts from zero and is scaled into
// fp32 accumulators when the block ends.
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

constexpr int kPfWarps = 8;
constexpr int kPfRows = 16 * kPfWarps;         // weight rows per CTA
constexpr int kPfTiles = 8;                    // 8-row activation tiles per CTA
constexpr int kPfTok = 8 * kPfTiles;           // activation rows per CTA
constexpr int kPfStage = 8;                    // 32-k chunks per stage (256 k)
// one activation row of a stage: kPfStage chunks x 4 groups of 16 bytes, plus
// 64 bytes so that rows g and g + 1 start 16 banks apart (conflict-free loads)
constexpr int kPfPitch = kPfStage * 4 + 4;     // in 16-byte words

struct PfParams {
  const uint16_t* x;
  const uint8_t* q;
  const uint16_t* scales;
  const uint8_t* zp;                           // nullptr: symmetric
  void* y;
  int M, N, K;
  int chunks;                                  // K / 32
  int blocks;                                  // K / B
  int zstride;                                 // zero-point bytes per row
  int bshift;                                  // log2(B / 32)
  int out_bf16;
  int x_aligned;
  int ksplit;                                  // CTAs of a cluster that split K (grid z)
};

__device__ __forceinline__ void pf_store(void* y, size_t idx, float v, int out_bf16) {
  const __half h = __float2half_rn(v);
  if (out_bf16)
    static_cast<uint16_t*>(y)[idx] = narrow_f16_bits_to_bf16(__half_as_ushort(h));
  else
    static_cast<__half*>(y)[idx] = h;
}

// q - zp pairs of code word `word` (see dequant_word in the general kernel).
__device__ __forceinline__ void pf_dequant(uint32_t word, uint32_t z, uint32_t* d) {
  const uint32_t zl = z * 0x00010001u + 0x64006400u;
  const uint32_t zh = z * 0x00100010u + 0x54005400u;
  const uint32_t w8 = word >> 8;
  d[0] = hsub2(and_or(word, 0x000F000Fu, 0x64006400u), zl);
  d[1] = hsub2(and_or(word, 0x00F000F0u, 0x54005400u), zh);
  d[2] = hsub2(and_or(w8, 0x000F000Fu, 0x64006400u), zl);
  d[3] = hsub2(and_or(w8, 0x00F000F0u, 0x54005400u), zh);
}

__global__ void __launch_bounds__(kPfWarps * 32, 2) gemm_prefill_kernel(const PfParams p) {
  __shared__ uint4 xs[kPfTok * kPfPitch];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int n0 = blockIdx.x * kPfRows + warp * 16;
  const int m0 = blockIdx.y * kPfTok;
  const int r0 = n0 + g, r1 = n0 + g + 8;                   // this lane's weight rows
  const int l0 = min(r0, p.N - 1), l1 = min(r1, p.N - 1);   // rows past N read row N - 1
  const uint32_t* q0 = reinterpret_cast<const uint32_t*>(p.q + static_cast<size_t>(l0) * (p.K / 2));
  const uint32_t* q1 = reinterpret_cast<const uint32_t*>(p.q + static_cast<size_t>(l1) * (p.K / 2));
  const uint16_t* s0p = p.scales + static_cast<size_t>(l0) * p.blocks;
  const uint16_t* s1p = p.scales + static_cast<size_t>(l1) * p.blocks;
  const int bmask = (1 << p.bshift) - 1;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  float acc[kPfTiles][4], D[kPfTiles][4];
#pragma unroll
  for (int j = 0; j < kPfTiles; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = D[j][e] = 0.f;

  for (int cs = 0; cs < p.chunks; cs += kPfStage) {
    const int nch = min(kPfStage, p.chunks - cs);
    __syncthreads();                                       // the last stage is read
    // stage: activation rows m0.., chunks cs.., regrouped (zero past M)
    for (int e = threadIdx.x; e < kPfTok * nch * 4; e += kPfWarps * 32) {
      const int tt = e / (nch * 4);
      const int rem = e - tt * (nch * 4);
      const int m = m0 + tt;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < p.M) {
        const uint16_t* src = p.x + static_cast<size_t>(m) * p.K + 32 * cs + 8 * rem;
        if (p.x_aligned) {
          v = __ldg(reinterpret_cast<const uint4*>(src));
        } else {
          v.x = __ldg(src + 0) | (static_cast<uint32_t>(__ldg(src + 1)) << 16);
          v.y = __ldg(src + 2) | (static_cast<uint32_t>(__ldg(src + 3)) << 16);
          v.z = __ldg(src + 4) | (static_cast<uint32_t>(__ldg(src + 5)) << 16);
          v.w = __ldg(src + 6) | (static_cast<uint32_t>(__ldg(src + 7)) << 16);
        }
      }
      xs[tt * kPfPitch + rem] = pair_k4(v);
    }
    __syncthreads();
    for (int cc = 0; cc < nch; ++cc) {
      const int c = cs + cc;
      const int b = c >> p.bshift;
      uint32_t z0 = 8, z1 = 8;
      if (p.zp) {
        const uint32_t zb0 = __ldg(p.zp + static_cast<size_t>(l0) * p.zstride + (b >> 1));
        const uint32_t zb1 = __ldg(p.zp + static_cast<size_t>(l1) * p.zstride + (b >> 1));
        z0 = (b & 1) ? (zb0 >> 4) : (zb0 & 0xFu);
        z1 = (b & 1) ? (zb1 >> 4) : (zb1 & 0xFu);
      }
      uint32_t d0[4], d1[4];
      pf_dequant(__ldg(q0 + 4 * c + t), z0, d0);
      pf_dequant(__ldg(q1 + 4 * c + t), z1, d1);
      const uint4* xrow = xs + g * kPfPitch + cc * 4 + t;
#pragma unroll
      for (int j = 0; j < kPfTiles; ++j) {
        const uint4 xv = xrow[j * 8 * kPfPitch];
        mma_16816(D[j], d0[0], d1[0], d0[1], d1[1], xv.x, xv.y, D[j]);
        mma_16816(D[j], d0[2], d1[2], d0[3], d1[3], xv.z, xv.w, D[j]);
      }
      if ((c & bmask) == bmask) {                           // the block ends here
        const float s0 = __half2float(__ushort_as_half(__ldg(s0p + b)));
        const float s1 = __half2float(__ushort_as_half(__ldg(s1p + b)));
#pragma unroll
        for (int j = 0; j < kPfTiles; ++j) {
          acc[j][0] = fmaf(D[j][0], s0, acc[j][0]);
          acc[j][1] = fmaf(D[j][1], s0, acc[j][1]);
          acc[j][2] = fmaf(D[j][2], s1, acc[j][2]);
          acc[j][3] = fmaf(D[j][3], s1, acc[j][3]);
          D[j][0] = D[j][1] = D[j][2] = D[j][3] = 0.f;
        }
      }
    }
  }
  // D element e of tile j: weight row r0 (e < 2) or r1, activation row
  // m0 + 8 j + 2 t + (e & 1)
#pragma unroll
  for (int j = 0; j < kPfTiles; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = e < 2 ? r0 : r1;
      const int m = m0 + 8 * j + 2 * t + (e & 1);
      if (n < p.N && m < p.M)
        pf_store(p.y, static_cast<size_t>(m) * p.N + n, acc[j][e], p.out_bf16);
    }
}


// ---- pipelined form (16-byte-aligned activations) --------------------------
//
// Two stage buffers in dynamic shared memory: while a stage is multiplied, the
// next stage's raw activations and codes arrive by async copies
// (cp.async.cg, 16 bytes each) and its scales and zero-points by plain loads
// held in registers until the stage's arithmetic is done.  Activations are
// regrouped into the (k, k + 4) pairs at fragment load (four byte permutes).
constexpr int kXPitch = kPfStage * 64 + 64;    // bytes per activation row of a stage
constexpr int kCPitch = kPfStage * 16 + 16;    // bytes per weight row of a stage
constexpr int kXBuf = kPfTok * kXPitch;
constexpr int kCBuf = kPfRows * kCPitch;
constexpr int kSBuf = kPfRows * kPfStage * 2;  // at most 8 scales per row and stage
constexpr int kZBuf = kPfRows * 4;             // at most 4 zero-point bytes per row and stage
constexpr int kPfSmem = 2 * (kXBuf + kCBuf + kSBuf + kZBuf);
constexpr int kSPer = kPfRows * kPfStage / (kPfWarps * 32);   // scales per thread per stage
constexpr int kZPer = kPfRows * 4 / (kPfWarps * 32);          // zero-point bytes per thread

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// kCtas: CTAs one SM holds (2 at 128 registers a thread, 1 above).
template <int kCtas>
__global__ void __launch_bounds__(kPfWarps * 32, kCtas) gemm_prefill_pipelined(const PfParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* xb = smem;                              // [2][kXBuf]
  unsigned char* cb = xb + 2 * kXBuf;                    // [2][kCBuf]
  uint16_t* sb = reinterpret_cast<uint16_t*>(cb + 2 * kCBuf);   // [2][rows][8]
  uint8_t* zb = reinterpret_cast<uint8_t*>(sb + 2 * kSBuf / 2); // [2][rows][4]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int nb0 = blockIdx.x * kPfRows;                  // first weight row of the CTA
  const int m0 = blockIdx.y * kPfTok;
  const int lr0 = warp * 16 + g, lr1 = lr0 + 8;          // this lane's rows in the CTA
  const int bper = 1 << p.bshift;                        // chunks per block
  // this CTA's stages: a contiguous share of the K stages (whole stages, so
  // every quantization block stays inside one CTA)
  const int nstages_all = (p.chunks + kPfStage - 1) / kPfStage;
  const int st_begin = static_cast<int>(blockIdx.z) * nstages_all / p.ksplit;
  const int st_end = (static_cast<int>(blockIdx.z) + 1) * nstages_all / p.ksplit;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint16_t spre[kSPer];
  uint8_t zpre[kZPer];
  auto fill_async = [&](int st, int bi) {
    const int cs = st * kPfStage;
    const int nch = min(kPfStage, p.chunks - cs);
    const uint32_t xdst = static_cast<uint32_t>(__cvta_generic_to_shared(xb + bi * kXBuf));
    const uint32_t cdst = static_cast<uint32_t>(__cvta_generic_to_shared(cb + bi * kCBuf));
    for (int e = threadIdx.x; e < kPfTok * nch * 4; e += kPfWarps * 32) {
      const int tt = e / (nch * 4), rem = e - tt * (nch * 4);
      const int m = min(m0 + tt, p.M - 1);                // rows past M repeat row M - 1
      cp_async16(xdst + tt * kXPitch + rem * 16, p.x + static_cast<size_t>(m) * p.K + 32 * cs + 8 * rem);
    }
    for (int e = threadIdx.x; e < kPfRows * nch; e += kPfWarps * 32) {
      const int r = e / nch, cc = e - r * nch;
      const int n = min(nb0 + r, p.N - 1);                // rows past N repeat row N - 1
      cp_async16(cdst + r * kCPitch + cc * 16, p.q + static_cast<size_t>(n) * (p.K / 2) + 16 * (cs + cc));
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto load_sz = [&](int st) {
    const int b0 = (st * kPfStage) >> p.bshift;
    const int nbk = (min(kPfStage, p.chunks - st * kPfStage) + bper - 1) >> p.bshift;
    const int nzb = (nbk + 1) >> 1;
#pragma unroll
    for (int i = 0; i < kSPer; ++i) {
      const int e = threadIdx.x + i * kPfWarps * 32;
      const int r = e / kPfStage, bb = e - r * kPfStage;
      const int n = min(nb0 + r, p.N - 1);
      spre[i] = bb < nbk ? __ldg(p.scales + static_cast<size_t>(n) * p.blocks + b0 + bb) : 0;
    }
#pragma unroll
    for (int i = 0; i < kZPer; ++i) {
      const int e = threadIdx.x + i * kPfWarps * 32;
      const int r = e >> 2, zz = e & 3;
      const int n = min(nb0 + r, p.N - 1);
      zpre[i] = (p.zp && zz < nzb) ? __ldg(p.zp + static_cast<size_t>(n) * p.zstride + (b0 >> 1) + zz) : 0;
    }
  };
  auto store_sz = [&](int bi) {
#pragma unroll
    for (int i = 0; i < kSPer; ++i) sb[bi * (kSBuf / 2) + threadIdx.x + i * kPfWarps * 32] = spre[i];
#pragma unroll
    for (int i = 0; i < kZPer; ++i) zb[bi * kZBuf + threadIdx.x + i * kPfWarps * 32] = zpre[i];
  };

  float acc[kPfTiles][4], D[kPfTiles][4];
#pragma unroll
  for (int j = 0; j < kPfTiles; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = D[j][e] = 0.f;

  fill_async(st_begin, 0);
  load_sz(st_begin);
  store_sz(0);
  for (int st = st_begin; st < st_end; ++st) {
    const int bi = (st - st_begin) & 1;
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();                 // stage st landed and is visible; buffer bi ^ 1 is free
    const bool more = st + 1 < st_end;
    if (more) {
      fill_async(st + 1, bi ^ 1);
      load_sz(st + 1);
    }
    const int cs = st * kPfStage;
    const int nch = min(kPfStage, p.chunks - cs);
    const int b0 = cs >> p.bshift;
    const unsigned char* xs = xb + bi * kXBuf + g * kXPitch + t * 16;
    const unsigned char* cw = cb + bi * kCBuf + 4 * t;
    const uint16_t* ss = sb + bi * (kSBuf / 2);
    const uint8_t* zs = zb + bi * kZBuf;
    for (int cc = 0; cc < nch; ++cc) {
      const int c = cs + cc;
      const int bb = (c >> p.bshift) - b0;
      uint32_t z0 = 8, z1 = 8;
      if (p.zp) {
        const uint32_t sh = (bb & 1) * 4;
        z0 = (static_cast<uint32_t>(zs[lr0 * 4 + (bb >> 1)]) >> sh) & 0xFu;
        z1 = (static_cast<uint32_t>(zs[lr1 * 4 + (bb >> 1)]) >> sh) & 0xFu;
      }
      uint32_t d0[4], d1[4];
      pf_dequant(*reinterpret_cast<const uint32_t*>(cw + lr0 * kCPitch + cc * 16), z0, d0);
      pf_dequant(*reinterpret_cast<const uint32_t*>(cw + lr1 * kCPitch + cc * 16), z1, d1);
#pragma unroll
      for (int j = 0; j < kPfTiles; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(xs + j * 8 * kXPitch + cc * 64);
        const uint32_t x04 = __byte_perm(v.x, v.z, 0x5410), x15 = __byte_perm(v.x, v.z, 0x7632);
        const uint32_t x26 = __byte_perm(v.y, v.w, 0x5410), x37 = __byte_perm(v.y, v.w, 0x7632);
        mma_16816(D[j], d0[0], d1[0], d0[1], d1[1], x04, x15, D[j]);
        mma_16816(D[j], d0[2], d1[2], d0[3], d1[3], x26, x37, D[j]);
      }
      if ((c & (bper - 1)) == bper - 1) {                  // the block ends here
        const float s0 = __half2float(__ushort_as_half(ss[lr0 * kPfStage + bb]));
        const float s1 = __half2float(__ushort_as_half(ss[lr1 * kPfStage + bb]));
#pragma unroll
        for (int j = 0; j < kPfTiles; ++j) {
          acc[j][0] = fmaf(D[j][0], s0, acc[j][0]);
          acc[j][1] = fmaf(D[j][1], s0, acc[j][1]);
          acc[j][2] = fmaf(D[j][2], s1, acc[j][2]);
          acc[j][3] = fmaf(D[j][3], s1, acc[j][3]);
          D[j][0] = D[j][1] = D[j][2] = D[j][3] = 0.f;
        }
      }
    }
    if (more) store_sz(bi ^ 1);
  }
  const int r0 = nb0 + lr0, r1 = nb0 + lr1;
  if (p.ksplit == 1) {
#pragma unroll
    for (int j = 0; j < kPfTiles; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = e < 2 ? r0 : r1;
        const int m = m0 + 8 * j + 2 * t + (e & 1);
        if (n < p.N && m < p.M)
          pf_store(p.y, static_cast<size_t>(m) * p.N + n, acc[j][e], p.out_bf16);
      }
    return;
  }
  // K split over the cluster: each CTA leaves its fp32 tile [activation row]
  // [weight row] (rows kPartPitch words apart: lanes (g, t) of a fragment
  // store hit 32 different banks) in its shared memory; after the cluster
  // barrier, rank r sums the
  // r-th 1/S of the tile over the ranks in rank order (distributed shared
  // memory) and stores it; a second barrier keeps every tile readable until
  // all ranks are done.
  __syncthreads();                                          // stage buffers are free
  constexpr int kPartPitch = kPfRows + 4;
  static_assert(kPfTok * kPartPitch * 4 <= 2 * kXBuf, "partial tile exceeds the stage buffers");
  float* part = reinterpret_cast<float*>(xb);               // 64 x 132 fp32
#pragma unroll
  for (int j = 0; j < kPfTiles; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      part[(8 * j + 2 * t + (e & 1)) * kPartPitch + (e < 2 ? lr0 : lr1)] = acc[j][e];
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  const int share = kPfRows * kPfTok / p.ksplit;
  const uint32_t part_addr = static_cast<uint32_t>(__cvta_generic_to_shared(part));
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  for (int e = threadIdx.x; e < share; e += kPfWarps * 32) {
    const int gidx = static_cast<int>(rank) * share + e;
    const int tok = gidx / kPfRows, row = gidx - tok * kPfRows;   // y row, column
    const uint32_t local = part_addr + 4u * static_cast<uint32_t>(tok * kPartPitch + row);
    float sum = 0.f;
    for (int r = 0; r < p.ksplit; ++r) {
      uint32_t remote;
      float v;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(r));
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
      sum += v;
    }
    const int n = nb0 + row, m = m0 + tok;
    if (n < p.N && m < p.M) pf_store(p.y, static_cast<size_t>(m) * p.N + n, sum, p.out_bf16);
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

// Launches the prefill GEMM; arguments are validated by the caller (M > 8,
// block 32, 64 or 128, K a multiple of 32 and of the block size).
int launch_prefill(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                   void* y, int M, int N, int K, int block, int out_bf16, int sms,
                   cudaStream_t stream, LaunchDesc* query) {
  PfParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.q = qweight;
  p.scales = static_cast<const uint16_t*>(scales);
  p.zp = zp;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.chunks = K / 32;
  p.blocks = K / block;
  p.zstride = (p.blocks + 1) / 2;
  p.bshift = block == 128 ? 2 : block == 64 ? 1 : 0;
  p.out_bf16 = out_bf16;
  p.x_aligned = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  p.ksplit = 1;
  const long long gx = (static_cast<long long>(N) + kPfRows - 1) / kPfRows;
  const long long gy = (static_cast<long long>(M) + kPfTok - 1) / kPfTok;
  if (gx > 0x7FFFFFFFLL || gy > 65535) return fail(MNB_ERR_SHAPE, "prefill shape too large");
  // A grid of at most half the SM count splits K over a cluster of up to 8
  // CTAs, doubling while the grid is below the SM count (each keeps two
  // stages); pipelined form only.
  const int nstages = (p.chunks + kPfStage - 1) / kPfStage;
  if (p.x_aligned)
    if (gx * gy * 2 <= sms)
      while (p.ksplit < 8 && gx * gy * p.ksplit < sms && nstages >= 4 * p.ksplit) p.ksplit *= 2;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                     static_cast<unsigned>(p.ksplit));
  cfg.blockDim = dim3(kPfWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.ksplit > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = static_cast<unsigned>(p.ksplit);
    cfg.numAttrs = 2;
  }
  void* args[1] = {&p};
  const void* fn = reinterpret_cast<const void*>(&gemm_prefill_kernel);
  if (p.x_aligned) {                 // the async copies want 16-byte-aligned rows
    // two CTAs per SM only when the grid needs them: a small grid would be
    // packed two to an SM and leave SMs idle
    fn = gx * gy * p.ksplit > sms ? reinterpret_cast<const void*>(&gemm_prefill_pipelined<2>)
                       : reinterpret_cast<const void*>(&gemm_prefill_pipelined<1>);
    cfg.dynamicSmemBytes = kPfSmem;
    const cudaError_t ea =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (ea != cudaSuccess) return cuda_fail(ea, "cudaFuncSetAttribute(prefill)");
  }
  if (query) {
    query->fn = fn;
    query->name = p.x_aligned ? "prefill GEMM, mma.sync form (pipelined)"
                              : "prefill GEMM, mma.sync form (synchronous, unaligned x)";
    query->counter = 16;
    query->grid = cfg.gridDim.x * cfg.gridDim.y * cfg.gridDim.z;
    query->threads = cfg.blockDim.x;
    query->cluster = static_cast<unsigned>(p.ksplit);
    query->smem = cfg.dynamicSmemBytes;
    return MNB_OK;
  }
  const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC(prefill)");
  return MNB_OK;
}

}  // namespace mnb
