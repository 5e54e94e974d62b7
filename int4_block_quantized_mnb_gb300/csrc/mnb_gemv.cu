// mnb_gemv.cu -- sm_103a kernels and C ABI of the int4 block-quantized
// MatMulNBits decode GEMV (see include/mnb.h for the contract).
//
// The operation ("perf(cuda): let the split-K decode GEMV store bf16
// directly", onnx-genai PR 1550, paragraphs 1-2; "PORT-1 ... measured NO-GO on
// the multicol asymmetric-zp GEMV", onnx-genai PR 1002, "Why the premise fails
// here" point 1):
//
//     y[m,n] = fp16( sum_k x[m,k] * (q[n,k] - zp[n,k/32]) * s[n,k/32] )
//     optionally narrowed to bf16( that fp16 value ).
//
// Design (weight-streaming, activation-stationary):
//   * One persistent CTA per SM owns a contiguous range of output rows n.  A
//     producer warp streams those rows' packed weights, scales and
//     zero-points into a ring of shared-memory stages with bulk asynchronous
//     copies (cp.async.bulk, completion on an mbarrier transaction count).
//   * Consumer warps keep their slice of the activations in registers for the
//     whole kernel.  Lane l of consumer warp w owns KPL consecutive k values
//     (a whole 32-block or half of one); the warps of one "group" tile the
//     CTA's K range, so each stage row is read from shared memory exactly once.
//   * Dequant per 32-bit word (8 codes): the code nibbles are OR-ed into the
//     mantissa of an fp16 constant (1024 + q for low nibbles, 64 + q for high
//     nibbles), and one packed fp16 subtraction of (1024 + zp) / (64 + zp)
//     leaves the exact small integer q - zp.  Each product x * (q - zp) is
//     exact in fp32 and is accumulated by a mixed-precision fma (f16 sources,
//     f32 accumulator); the block's sum is multiplied by its fp32 scale.
//   * Split-K inside the CTA: per-lane partials are reduced across the warp
//     with a transposing butterfly (one value per (row, m) per lane group),
//     then across the group's warps through shared memory in a fixed order.
//   * Split-K across CTAs (split_k > 1): the CTAs of one thread-block cluster
//     take disjoint K ranges of the same rows; partial row sums stay in each
//     CTA's shared memory and are added in rank order through distributed
//     shared memory.  No global workspace and no atomics are involved, so
//     the fp16 and bf16 arms see the identical fp32 sum.
//   * Epilogue: fp32 -> fp16 round-to-nearest-even on the lane that owns the
//     output element; the bf16 arm narrows that fp16 value with a second
//     round-to-nearest-even (launch-uniform flag).
//   * Every wait on an mbarrier is bounded by a global-timer deadline; a wait
//     that gives up records a code in a device error word, tells the CTA to
//     stop, lets in-flight copies land and returns.

#include "mnb.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace mnb {

constexpr int kBlock = MNB_BLOCK;
constexpr int kMaxM = MNB_MAX_M;
constexpr int kMaxSplit = MNB_MAX_SPLIT_K;

// Consumer warps per CTA: 12 for M <= 2 keeps at most 4 warps (14 with the
// producer and epilogue warps) on an SM sub-partition, i.e. 128 registers per thread.
constexpr int consumer_warp_budget(int M) { return M <= 2 ? 12 : 16; }
constexpr int max_threads(int M) { return (consumer_warp_budget(M) + 2) * 32; }
constexpr int kSmemBudget = 200 * 1024;           // stages + bookkeeping
constexpr int kPartBudget = 32 * 1024;            // cluster partial sums per CTA
constexpr int kMaxStages = 16;
constexpr int kSlotsPerGroup = 4;               // reduction slots a group may have pending
constexpr int kStageCodeBytes = 32 * 1024;        // target size of a stage's code area
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

enum : unsigned {
  kErrStageData = 1,
  kErrStageFree = 2,
  kErrDrain = 3,
  kErrReduceSlot = 4,
};

__device__ unsigned int g_device_error;

struct Params {
  const uint16_t* x;
  const uint8_t* q;
  const uint16_t* scales;
  const uint8_t* zp;
  void* y;
  int M, N, K;
  int C;            // 32-blocks per row
  int Z;            // zero-point bytes per row
  int out_bf16;
  int weights_ready;  // weights may be read before the preceding grid completes
  int split;        // CTAs per cluster along K
  int groups;       // consumer groups per CTA
  int wpg;          // warps per group
  int stages;
  int rows_stage;   // rows of the weight matrix per stage (a multiple of the chunk rows)
  int q_pitch;      // bytes per row inside a stage's weight area
  int q_bytes, sc_bytes, zp_bytes, stage_bytes;
  int bar_offset;   // shared-memory offset of the mbarrier array
  int red_offset;   // offset of the cross-warp reduction slots
  int part_offset;  // offset of the cluster partial sums
  int flag_offset;  // offset of the CTA abort flag
};

// ---------------------------------------------------------------- PTX glue --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Slow path of mbar_wait: polls until the phase completes, the CTA abort flag
// is raised, or kWaitLimitNs pass (then records `code` and raises the flag).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            unsigned code) {
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicCAS(&g_device_error, 0u, code);
      return false;
    }
  }
}

// Waits for the phase of `bar` with the given parity; false if the wait gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, code);
}

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: let the next grid on the stream launch now,
// and wait until the preceding grid has completed and its writes are visible.
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

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

// Butterfly that leaves lane L holding, summed over all 32 lanes, value
// number (L >> (5 - log2(VP))) of the VP values every lane started with.
template <int VP>
__device__ __forceinline__ float transpose_reduce(float (&v)[VP], int lane) {
#pragma unroll
  for (int cnt = VP, off = 16; cnt > 1; cnt >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = upper ? v[i] : v[i + cnt / 2];
      const float keep = upper ? v[i + cnt / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = 16 / VP; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

template <int N>
struct Pow2Ceil {
  static constexpr int value = N <= 1 ? 1 : 2 * Pow2Ceil<(N + 1) / 2>::value;
};
template <>
struct Pow2Ceil<1> {
  static constexpr int value = 1;
};

// fp32 accumulator -> fp16 (RNE), optionally -> bf16 (RNE of the fp16 value).
__device__ __forceinline__ void store_output(void* y, size_t idx, float v, int out_bf16) {
  const __half h = __float2half_rn(v);
  if (out_bf16) {
    static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(__half2float(h));
  } else {
    static_cast<__half*>(y)[idx] = h;
  }
}

// Copies global bytes [src, src + n) into shared memory at dst_base + (src & 15)
// so that 16-byte-aligned global addresses land on 16-byte-aligned shared
// addresses.  The aligned middle goes through one bulk copy; the (< 16 byte)
// unaligned head and tail are copied with plain loads and stores.  Returns the
// byte count handed to the bulk copy engine.
struct RegionCopy {
  uint32_t dst;
  const uint8_t* src;
  uint32_t body;
};

__device__ __forceinline__ RegionCopy plan_region(unsigned char* dst_base, const uint8_t* src,
                                                  uint32_t n) {
  const uint32_t a = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
  unsigned char* dst = dst_base + a;
  uint32_t head = (16u - a) & 15u;
  if (head > n) head = n;
  const uint32_t body = (n - head) & ~15u;
  const uint32_t tail_start = head + body;
  for (uint32_t i = 0; i < head; ++i) dst[i] = __ldg(src + i);
  for (uint32_t i = tail_start; i < n; ++i) dst[i] = __ldg(src + i);
  return RegionCopy{smem_u32(dst + head), src + head, body};
}

// ------------------------------------------------------------------ kernel --

template <int M, int KPL, int RC>
__global__ void __launch_bounds__(max_threads(M), 1) gemv_kernel(const Params p) {
  constexpr int kWords = KPL / 8;                   // 32-bit code words per lane segment
  constexpr int kLaneBlocks = KPL >= 32 ? KPL / 32 : 1;   // 32-blocks a lane's segment touches
  constexpr int kBlockWords = KPL >= 32 ? 4 : kWords;     // words of the segment in one block
  static_assert(KPL == 16 || KPL == 32 || KPL == 64, "segment of 16, 32 or 64 codes");
  constexpr int kVals = RC * M;                     // (row, m) values per lane per stage
  constexpr int kVP = Pow2Ceil<kVals>::value;
  constexpr int kOwnerShift = 5 - (kVP == 1 ? 0 : kVP == 2 ? 1 : kVP == 4 ? 2 : kVP == 8 ? 3 : kVP == 16 ? 4 : 5);
  static_assert(kVP <= 32, "too many values per lane");

  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int consumer_warps = p.groups * p.wpg;
  const int producer_warp = consumer_warps;
  const int epilogue_warp = consumer_warps + 1;
  const int nslots = p.groups * kSlotsPerGroup;

  // mbarriers:
  //   full[s]   (stage)  1 arrival + transaction bytes: the stage's data landed
  //   empty[s]  (stage)  wpg arrivals per tile of the stage: once every tile's
  //                      K-slice warps hold their data in registers the stage
  //                      may be refilled
  //   ready[j]  (slot)   wpg arrivals: every K-slice warp filed its partial sums
  //   free[j]   (slot)   1 arrival: the epilogue has consumed the slot
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_offset);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * p.stages;
  const uint32_t ready0 = empty0 + 8u * p.stages;
  const uint32_t free0 = ready0 + 8u * nslots;
  float* red = reinterpret_cast<float*>(smem + p.red_offset);     // [slots][wpg][RC * M]
  float* part = reinterpret_cast<float*>(smem + p.part_offset);   // [cluster rows][M]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.flag_offset);

  // Row range of this CTA (of its cluster when split > 1) and its K range.
  const int split = p.split;
  const uint32_t rank = split > 1 ? cluster_rank() : 0u;
  const int unit = blockIdx.x / split;
  const int units = gridDim.x / split;
  const int row_begin = static_cast<int>((static_cast<long long>(unit) * p.N) / units);
  const int row_end = static_cast<int>((static_cast<long long>(unit + 1) * p.N) / units);
  const int nrows = row_end - row_begin;
  const int ntiles = (nrows + RC - 1) / RC;         // tiles of RC rows (one group each)
  const int RS = p.rows_stage;                      // a stage holds RS / RC whole tiles
  const int TPS = RS / RC;
  const int nstages = (nrows + RS - 1) / RS;        // stage loads this CTA makes
  // K ranges are whole multiples of the lane segment's blocks (2 when KPL = 64).
  const int seg_units = p.C / kLaneBlocks;
  const int b_begin = kLaneBlocks * static_cast<int>((static_cast<long long>(rank) * seg_units) / split);
  const int b_end = kLaneBlocks * static_cast<int>((static_cast<long long>(rank + 1) * seg_units) / split);
  const int k_begin = b_begin * kBlock;
  const int k_len = (b_end - b_begin) * kBlock;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, p.wpg * TPS);
    }
    for (int j = 0; j < nslots; ++j) {
      mbar_init(ready0 + 8u * j, p.wpg);
      mbar_init(free0 + 8u * j, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // The next GEMV on the stream may launch while this one runs; every read of
  // a caller array below waits for the preceding grid first (weights only
  // when the caller has not promised they are ready).
  allow_dependents();

  if (warp == producer_warp) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      if (!p.weights_ready) wait_prerequisites();
      int issued = 0;
      int s = 0;                                        // stage slot of load i
      uint32_t ph = 0;                                  // completed uses of slot s, mod 2
      for (int i = 0; i < nstages; ++i) {
        if (i >= p.stages && !mbar_wait(empty0 + 8u * s, ph ^ 1u, abort_flag, kErrStageFree))
          break;
        const int r0 = row_begin + i * RS;
        const int nr = min(RS, row_end - r0);
        unsigned char* st = smem + static_cast<size_t>(s) * p.stage_bytes;
        const uint32_t bar = full0 + 8u * s;
        // Scales and zero-points of these rows are contiguous in global memory.
        const RegionCopy sc = plan_region(
            st + p.q_bytes,
            reinterpret_cast<const uint8_t*>(p.scales) + static_cast<size_t>(r0) * p.C * 2,
            static_cast<uint32_t>(nr) * p.C * 2);
        const RegionCopy zc = plan_region(st + p.q_bytes + p.sc_bytes,
                                          p.zp + static_cast<size_t>(r0) * p.Z,
                                          static_cast<uint32_t>(nr) * p.Z);
        fence_proxy_async_smem();
        const uint32_t q_row_bytes = static_cast<uint32_t>(k_len / 2);
        const uint32_t tx = static_cast<uint32_t>(nr) * q_row_bytes + sc.body + zc.body;
        mbar_arrive_expect_tx(bar, tx);
        const uint8_t* qsrc = p.q + static_cast<size_t>(r0) * (p.K / 2) + k_begin / 2;
        if (split == 1) {
          bulk_copy_g2s(smem_u32(st), qsrc, static_cast<uint32_t>(nr) * q_row_bytes, bar);
        } else {
          for (int r = 0; r < nr; ++r)
            bulk_copy_g2s(smem_u32(st + static_cast<size_t>(r) * p.q_pitch),
                          qsrc + static_cast<size_t>(r) * (p.K / 2), q_row_bytes, bar);
        }
        if (sc.body) bulk_copy_g2s(sc.dst, sc.src, sc.body, bar);
        if (zc.body) bulk_copy_g2s(zc.dst, zc.src, zc.body, bar);
        issued = i + 1;
        if (++s == p.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Let every copy this thread issued land before the CTA may exit.
      for (int i = max(0, issued - p.stages); i < issued; ++i) {
        const int s = i % p.stages;
        if (!mbar_try_wait(full0 + 8u * s, (i / p.stages) & 1)) {
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(full0 + 8u * s, (i / p.stages) & 1)) {
            if (global_ns() - t0 > kWaitLimitNs) {
              atomicCAS(&g_device_error, 0u, kErrDrain);
              break;
            }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == epilogue_warp) {
    // ------------------------------------------------------------ epilogue --
    // Adds the K-slice partial sums of every row in slice order, rounds and
    // stores (or keeps them for the cluster reduction), then frees the slot.
    wait_prerequisites();
    int g = 0, t = 0;                                   // tile i belongs to group g, its t-th
    for (int i = 0; i < ntiles; ++i) {
      const int j = g * kSlotsPerGroup + t % kSlotsPerGroup;
      if (!mbar_wait(ready0 + 8u * j, (t / kSlotsPerGroup) & 1, abort_flag, kErrReduceSlot)) break;
      const int r0 = row_begin + i * RC;
      const int vals = min(RC, row_end - r0) * M;
      const float* slot = red + static_cast<size_t>(j) * p.wpg * kVals;
      if (lane < vals) {
        float sum = 0.f;
        for (int w = 0; w < p.wpg; ++w) sum += slot[w * kVals + lane];
        const int r = lane / M, m = lane % M;
        if (split == 1)
          store_output(p.y, static_cast<size_t>(m) * p.N + r0 + r, sum, p.out_bf16);
        else
          part[(r0 - row_begin + r) * M + m] = sum;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(free0 + 8u * j);
      if (++g == p.groups) {
        g = 0;
        ++t;
      }
    }
  } else {
    // ----------------------------------------------------------- consumers --
    const int g = warp / p.wpg;
    const int wg = warp % p.wpg;
    const int seg = wg * 32 + lane;
    const int kl = seg * KPL;                           // offset inside the CTA's K range
    const bool active = kl < k_len;
    // Inactive lanes (past the end of the K range) alias the range's first
    // segment so every shared-memory read stays inside the stage; their
    // activations are zero, so they contribute exact zeros.
    const int klc = active ? kl : 0;
    const int bl = (k_begin + klc) / kBlock;            // global 32-block index
    const int zshift = (bl & 1) * 4;

    // Activations for this lane's k values, paired to match the nibble order
    // produced by the dequant below: word i holds k = 8i..8i+7 of the segment
    // and pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7).
    wait_prerequisites();
    uint32_t xr[M][kWords][4];
#pragma unroll
    for (int m = 0; m < M; ++m) {
#pragma unroll
      for (int i = 0; i < kWords; ++i) {
        uint16_t h[8];
        if (active) {
          const uint16_t* src = p.x + static_cast<size_t>(m) * p.K + k_begin + kl + 8 * i;
          if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
            h[0] = v.x & 0xFFFF; h[1] = v.x >> 16; h[2] = v.y & 0xFFFF; h[3] = v.y >> 16;
            h[4] = v.z & 0xFFFF; h[5] = v.z >> 16; h[6] = v.w & 0xFFFF; h[7] = v.w >> 16;
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = __ldg(src + j);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) h[j] = 0;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          xr[m][i][j] = static_cast<uint32_t>(h[j]) | (static_cast<uint32_t>(h[j + 4]) << 16);
      }
    }

    const uintptr_t sc_mis = reinterpret_cast<uintptr_t>(p.scales) & 15u;
    const uintptr_t zp_mis = reinterpret_cast<uintptr_t>(p.zp) & 15u;
    const int q_pitch = p.q_pitch, C = p.C, Z = p.Z;
    // Tile i sits in stage load si = i / TPS at row ti * RC; the load uses
    // slot s = si % stages for the ph-th time (mod 2).  Kept incrementally:
    // no division in the loop.
    int si = g / TPS;
    int ti = g - si * TPS;
    int s = si % p.stages;
    uint32_t ph = static_cast<uint32_t>(si / p.stages) & 1u;
    int t = 0;                                          // this group's tile counter
    for (int i = g; i < ntiles; ++t) {
      if (!mbar_wait(full0 + 8u * s, ph, abort_flag, kErrStageData)) break;
      const int r0 = row_begin + i * RC;
      const int nr = min(RC, row_end - r0);
      const int rin = ti * RC;                          // tile's first row inside the stage
      const int rs0 = r0 - rin;                         // first row of the stage
      const unsigned char* st = smem + static_cast<size_t>(s) * p.stage_bytes;
      // Misalignment offsets chosen by the producer's region copies.
      const uint32_t sc_off =
          static_cast<uint32_t>((sc_mis + static_cast<uintptr_t>(rs0) * C * 2) & 15u);
      const uint32_t zp_off = static_cast<uint32_t>((zp_mis + static_cast<uintptr_t>(rs0) * Z) & 15u);
      const unsigned char* qp = st + rin * q_pitch + klc / 2;
      const uint16_t* sp = reinterpret_cast<const uint16_t*>(st + p.q_bytes + sc_off) + rin * C + bl;
      const unsigned char* zpp = st + p.q_bytes + p.sc_bytes + zp_off + rin * Z + (bl >> 1);

      // Pull this lane's codes, zero-point bytes and scales of every row into
      // registers and give the stage straight back to the producer.  Rows past
      // the end of a ragged tile re-read its last row; they are never stored.
      uint32_t words[RC][kWords];
      uint32_t zbyte[RC];
      uint32_t sbits[RC];
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        const int rr = (nr == RC) ? r : min(r, nr - 1);
        const unsigned char* qrow = qp + rr * q_pitch;
        if constexpr (kWords == 2) {
          const uint2 a = *reinterpret_cast<const uint2*>(qrow);
          words[r][0] = a.x; words[r][1] = a.y;
        } else {
#pragma unroll
          for (int h = 0; h < kWords / 4; ++h) {
            const uint4 a = *reinterpret_cast<const uint4*>(qrow + 16 * h);
            words[r][4 * h] = a.x; words[r][4 * h + 1] = a.y;
            words[r][4 * h + 2] = a.z; words[r][4 * h + 3] = a.w;
          }
        }
        zbyte[r] = zpp[rr * Z];
        if constexpr (kLaneBlocks == 2)
          sbits[r] = *reinterpret_cast<const uint32_t*>(sp + rr * C);
        else
          sbits[r] = sp[rr * C];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * s);

      float v[kVP];
#pragma unroll
      for (int j = 0; j < kVP; ++j) v[j] = 0.f;
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        uint32_t zl[kLaneBlocks], zh[kLaneBlocks];
        float scale[kLaneBlocks];
        if constexpr (kLaneBlocks == 2) {
          // Blocks bl (even, low nibble) and bl + 1 (high nibble) share one byte.
          const uint32_t tz = zbyte[r] * 0x00010001u;
          zl[0] = and_or(tz, 0x000F000Fu, 0x64006400u);         // 1024 + zp, twice
          zh[0] = and_or(tz << 4, 0x00F000F0u, 0x54005400u);    //   64 + zp, twice
          zl[1] = and_or(tz >> 4, 0x000F000Fu, 0x64006400u);
          zh[1] = and_or(tz, 0x00F000F0u, 0x54005400u);
          scale[0] = __half2float(__ushort_as_half(static_cast<unsigned short>(sbits[r] & 0xFFFFu)));
          scale[1] = __half2float(__ushort_as_half(static_cast<unsigned short>(sbits[r] >> 16)));
        } else {
          const uint32_t tz = zbyte[r] >> zshift;
          zl[0] = and_or(tz * 0x00010001u, 0x000F000Fu, 0x64006400u);
          zh[0] = and_or(tz * 0x00100010u, 0x00F000F0u, 0x54005400u);
          scale[0] = __half2float(__ushort_as_half(static_cast<unsigned short>(sbits[r])));
        }
        float res[M];
#pragma unroll
        for (int m = 0; m < M; ++m) res[m] = 0.f;
#pragma unroll
        for (int j = 0; j < kLaneBlocks; ++j) {
          float acc[M];
#pragma unroll
          for (int m = 0; m < M; ++m) acc[m] = 0.f;
#pragma unroll
          for (int w = j * kBlockWords; w < (j + 1) * kBlockWords; ++w) {
            const uint32_t word = words[r][w];
            const uint32_t w8 = word >> 8;
            const uint32_t d0 = hsub2(and_or(word, 0x000F000Fu, 0x64006400u), zl[j]);   // k0, k4
            const uint32_t d1 = hsub2(and_or(word, 0x00F000F0u, 0x54005400u), zh[j]);   // k1, k5
            const uint32_t d2 = hsub2(and_or(w8, 0x000F000Fu, 0x64006400u), zl[j]);     // k2, k6
            const uint32_t d3 = hsub2(and_or(w8, 0x00F000F0u, 0x54005400u), zh[j]);     // k3, k7
#pragma unroll
            for (int m = 0; m < M; ++m) {
              acc[m] = fma2_f16_f32(xr[m][w][0], d0, acc[m]);
              acc[m] = fma2_f16_f32(xr[m][w][1], d1, acc[m]);
              acc[m] = fma2_f16_f32(xr[m][w][2], d2, acc[m]);
              acc[m] = fma2_f16_f32(xr[m][w][3], d3, acc[m]);
            }
          }
#pragma unroll
          for (int m = 0; m < M; ++m) res[m] = fmaf(acc[m], scale[j], res[m]);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) v[r * M + m] = res[m];
      }

      // Warp sum of every (row, m) value; the owning lane files it in this K
      // slice's part of a reduction slot, which the epilogue warp finishes.
      const float total = transpose_reduce<kVP>(v, lane);
      const int idx = lane >> kOwnerShift;
      const int j = g * kSlotsPerGroup + t % kSlotsPerGroup;
      if (t >= kSlotsPerGroup &&
          !mbar_wait(free0 + 8u * j, ((t / kSlotsPerGroup) - 1) & 1, abort_flag, kErrReduceSlot))
        break;
      if ((lane & ((1 << kOwnerShift) - 1)) == 0 && idx < kVals)
        red[(static_cast<size_t>(j) * p.wpg + wg) * kVals + idx] = total;
      __syncwarp();
      if (lane == 0) mbar_arrive(ready0 + 8u * j);
      i += p.groups;
      for (ti += p.groups; ti >= TPS; ti -= TPS) {
        if (++s == p.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  }

  if (split > 1) {
    wait_prerequisites();
    cluster_sync();  // every CTA of the cluster has written its partial sums
    // Rank r finalises rows r, r + split, ...; peers are added in rank order.
    const uint32_t part_addr = smem_u32(part);
    for (int e = threadIdx.x; e < nrows * M; e += blockDim.x) {
      const int r = e / M;
      if (r % split != static_cast<int>(rank)) continue;
      float sum = 0.f;
      for (int c = 0; c < split; ++c) sum += ld_dsmem_f32(part_addr + 4u * e, c);
      store_output(p.y, static_cast<size_t>(e % M) * p.N + row_begin + r, sum, p.out_bf16);
    }
    cluster_sync();  // peers' shared memory stays alive until everyone is done
  }
}

// ------------------------------------------------------------- host side --

struct KernelShape {
  int kpl;
  int rc;
};

constexpr KernelShape shape_for(int M) {
  return M == 1 ? KernelShape{32, 8}
       : M == 2 ? KernelShape{32, 4}
       : M == 3 ? KernelShape{32, 4}
       : M == 4 ? KernelShape{16, 4}
                : KernelShape{16, 2};
}

using KernelFn = void (*)(const Params);

template <int M>
constexpr KernelFn kernel_for() {
  return &gemv_kernel<M, shape_for(M).kpl, shape_for(M).rc>;
}

// Lane segment and rows per tile: the per-M default.  (The kernel template
// also supports 64-code segments, two blocks per lane; on GB300 they measured
// slower than 32-code segments for M = 1, so they are not instantiated.)
KernelShape pick_shape(int M, int, int, const void*) { return shape_for(M); }

KernelFn pick_kernel(int M, const KernelShape&) {
  switch (M) {
    case 1: return kernel_for<1>();
    case 2: return kernel_for<2>();
    case 3: return kernel_for<3>();
    case 4: return kernel_for<4>();
    case 5: return kernel_for<5>();
    case 6: return kernel_for<6>();
    case 7: return kernel_for<7>();
    default: return kernel_for<8>();
  }
}

int max_k_per_cta(int M) { return consumer_warp_budget(M) * 32 * shape_for(M).kpl; }

thread_local std::string t_detail;

int fail(int status, const std::string& detail) {
  t_detail = detail;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  t_detail = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return MNB_ERR_CUDA;
}

std::atomic<unsigned long long> g_counters[MNB_NUM_COUNTERS];

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  size_t smem_optin = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mutex;

int device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MNB_ERR_DEVICE, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_device_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(smem)");
    d.smem_optin = static_cast<size_t>(v);
    d.ready = true;
  }
  if (d.major != 10 || d.minor != 3)
    return fail(MNB_ERR_DEVICE, "this library is built for sm_103 (GB300) only; device is sm_" +
                                    std::to_string(d.major) + std::to_string(d.minor));
  *out = d;
  return MNB_OK;
}

int check_shape(int M, int N, int K) {
  if (M < 1 || M > kMaxM) return fail(MNB_ERR_SHAPE, "M must be in 1..8");
  if (N < 1) return fail(MNB_ERR_SHAPE, "N must be >= 1");
  if (K < kBlock || K % kBlock != 0) return fail(MNB_ERR_SHAPE, "K must be a positive multiple of 32");
  const int min_split = (K + max_k_per_cta(M) - 1) / max_k_per_cta(M);
  if (min_split > kMaxSplit || min_split > K / kBlock)
    return fail(MNB_ERR_SHAPE, "K too large for this M");
  return MNB_OK;
}

int min_split(int M, int K) { return (K + max_k_per_cta(M) - 1) / max_k_per_cta(M); }

int auto_split(int M, int N, int K, int sms) {
  const int C = K / kBlock;
  const int lo = min_split(M, K);
  const int hi = std::min(kMaxSplit, C);
  const int rc = shape_for(M).rc;
  const long long tiles = (static_cast<long long>(N) + rc - 1) / rc;
  int s = lo;
  // Few row tiles: spread K over a cluster so more SMs stream weights.
  if (tiles < sms) {
    const long long want = sms / std::max<long long>(tiles, 1);
    s = static_cast<int>(std::min<long long>(std::max<long long>(want, lo), hi));
  }
  return std::max(lo, std::min(s, hi));
}

struct Plan {
  Params p;
  dim3 grid, block;
  size_t smem;
};

int make_plan(const DeviceInfo& dev, int M, int N, int K, int split, const KernelShape& ks,
              Plan* plan) {
  Params& p = plan->p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.C = K / kBlock;
  p.Z = (p.C + 1) / 2;
  p.split = split;
  const int lane_blocks = ks.kpl >= 32 ? ks.kpl / 32 : 1;
  const int seg_units = p.C / lane_blocks;
  const int blocks_cta = lane_blocks * ((seg_units + split - 1) / split);   // largest rank K range
  const int k_cta = blocks_cta * kBlock;
  const int segs = k_cta / ks.kpl;
  p.wpg = (segs + 31) / 32;                            // <= consumer_warp_budget(M) by check_shape
  p.groups = std::max(1, std::min(4, consumer_warp_budget(M) / p.wpg));
  p.q_pitch = k_cta / 2;
  // Grid: one CTA per SM; with split > 1 the units are clusters, and enough
  // of them that each cluster's partial sums fit in shared memory.
  const long long tiles = (static_cast<long long>(N) + ks.rc - 1) / ks.rc;
  long long units = std::max(1, dev.sms / split);
  units = std::min(units, tiles);
  if (split > 1) {
    const long long min_units = (static_cast<long long>(N) * M * 4 + kPartBudget - 1) / kPartBudget;
    units = std::max(units, min_units);
  }
  units = std::max<long long>(units, 1);
  const long long rows_per_unit = (N + units - 1) / units;
  const int part_bytes = split > 1 ? static_cast<int>(((rows_per_unit * M * 4) + 15) & ~15LL) : 0;

  // Shared memory: a ring of stages (codes, scales and zero-points of RC rows),
  // the groups' reduction slots, and the mbarriers.
  // A stage holds whole tiles of ks.rc rows, about kStageCodeBytes of codes
  // (large bulk copies stream best), never more rows than the CTA owns.
  const int unit_tiles = static_cast<int>((rows_per_unit + ks.rc - 1) / ks.rc);
  const int tps = std::max(1, std::min(unit_tiles, kStageCodeBytes / (ks.rc * p.q_pitch)));
  p.rows_stage = ks.rc * tps;
  p.q_bytes = p.rows_stage * p.q_pitch;
  p.sc_bytes = (p.rows_stage * p.C * 2 + 16 + 15) & ~15;
  p.zp_bytes = (p.rows_stage * p.Z + 16 + 15) & ~15;
  p.stage_bytes = p.q_bytes + p.sc_bytes + p.zp_bytes;
  const int nslots = p.groups * kSlotsPerGroup;
  const int red_bytes = ((nslots * p.wpg * ks.rc * M * 4) + 15) & ~15;
  const int fixed = red_bytes + 8 * 2 * nslots + part_bytes + 16;
  const int budget = std::min<int>(kSmemBudget, static_cast<int>(dev.smem_optin)) - fixed;
  const int stages = std::min(budget / (p.stage_bytes + 16), kMaxStages);
  if (stages < 2) return fail(MNB_ERR_SHAPE, "shape needs more shared memory than one SM has");
  p.stages = stages;
  int off = stages * p.stage_bytes;
  p.red_offset = off;
  off += red_bytes;
  p.bar_offset = off;
  off += 8 * (2 * stages + 2 * nslots);
  p.part_offset = off;
  off += part_bytes;
  p.flag_offset = off;
  off += 16;
  plan->smem = static_cast<size_t>(off);
  plan->grid = dim3(static_cast<unsigned>(units * split));
  plan->block = dim3(static_cast<unsigned>((p.groups * p.wpg + 2) * 32));
  return MNB_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(a), y0 = reinterpret_cast<uintptr_t>(b);
  return x0 < y0 + nb && y0 < x0 + na;
}

}  // namespace mnb

using namespace mnb;

extern "C" {

int mnb_abi_version(void) { return MNB_ABI_VERSION; }

const char* mnb_status_string(int status) {
  switch (status) {
    case MNB_OK: return "ok";
    case MNB_ERR_NULL: return "a required pointer is NULL";
    case MNB_ERR_SHAPE: return "shape out of range";
    case MNB_ERR_BLOCK: return "block size must be 32";
    case MNB_ERR_DTYPE: return "unknown output dtype";
    case MNB_ERR_SPLITK: return "split_k out of range";
    case MNB_ERR_ALIGN: return "pointer misaligned";
    case MNB_ERR_ALIAS: return "output overlaps an input";
    case MNB_ERR_CUDA: return "CUDA runtime error";
    case MNB_ERR_DEVICE: return "unsupported device";
    case MNB_ERR_FLAGS: return "unknown flag bits";
    default: return "unknown status";
  }
}

const char* mnb_last_error_detail(void) { return t_detail.c_str(); }

int mnb_max_split_k(int K, int* max_split) {
  if (!max_split) return fail(MNB_ERR_NULL, "max_split is NULL");
  if (K < kBlock || K % kBlock != 0) return fail(MNB_ERR_SHAPE, "K must be a positive multiple of 32");
  *max_split = std::min(kMaxSplit, K / kBlock);
  return MNB_OK;
}

int mnb_min_split_k(int M, int K, int* out) {
  if (!out) return fail(MNB_ERR_NULL, "min_split is NULL");
  int st = check_shape(M, 1, K);
  if (st != MNB_OK) return st;
  *out = min_split(M, K);
  return MNB_OK;
}

int mnb_split_k_auto(int M, int N, int K, int* split_k) {
  if (!split_k) return fail(MNB_ERR_NULL, "split_k is NULL");
  int st = check_shape(M, N, K);
  if (st != MNB_OK) return st;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != MNB_OK) return st;
  *split_k = auto_split(M, N, K, dev.sms);
  return MNB_OK;
}

int mnb_gemv(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp, void* y,
             int M, int N, int K, int block, int out_dtype, int split_k, void* stream) {
  return mnb_gemv_flags(x, qweight, scales, zp, y, M, N, K, block, out_dtype, split_k, 0u, stream);
}

int mnb_gemv_flags(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                   void* y, int M, int N, int K, int block, int out_dtype, int split_k,
                   unsigned int flags, void* stream) {
  if (flags & ~static_cast<unsigned int>(MNB_FLAG_WEIGHTS_READY))
    return fail(MNB_ERR_FLAGS, "unknown flag bits");
  if (!x || !qweight || !scales || !zp || !y) return fail(MNB_ERR_NULL, "x, qweight, scales, zp and y are required");
  if (block != kBlock) return fail(MNB_ERR_BLOCK, "only block size 32 is supported");
  int st = check_shape(M, N, K);
  if (st != MNB_OK) return st;
  if (out_dtype != MNB_OUT_F16 && out_dtype != MNB_OUT_BF16)
    return fail(MNB_ERR_DTYPE, "out_dtype must be MNB_OUT_F16 or MNB_OUT_BF16");
  if ((reinterpret_cast<uintptr_t>(qweight) & 15u) != 0)
    return fail(MNB_ERR_ALIGN, "qweight must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(x) & 1u) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(y) & 1u))
    return fail(MNB_ERR_ALIGN, "x, scales and y must be 2-byte aligned");
  const size_t C = static_cast<size_t>(K) / kBlock;
  const size_t ybytes = static_cast<size_t>(M) * N * 2;
  if (overlaps(y, ybytes, x, static_cast<size_t>(M) * K * 2) ||
      overlaps(y, ybytes, qweight, static_cast<size_t>(N) * K / 2) ||
      overlaps(y, ybytes, scales, static_cast<size_t>(N) * C * 2) ||
      overlaps(y, ybytes, zp, static_cast<size_t>(N) * ((C + 1) / 2)))
    return fail(MNB_ERR_ALIAS, "y overlaps an input array");
  const int lo = min_split(M, K);
  const int hi = std::min(kMaxSplit, K / kBlock);
  if (split_k < 0 || split_k > hi || (split_k != 0 && split_k < lo))
    return fail(MNB_ERR_SPLITK, "split_k must be 0 or in [" + std::to_string(lo) + ", " +
                                    std::to_string(hi) + "] for this M and K");
  DeviceInfo dev;
  if ((st = device_info(&dev)) != MNB_OK) return st;
  const int split = split_k == 0 ? auto_split(M, N, K, dev.sms) : split_k;

  const KernelShape ks = pick_shape(M, K / kBlock, split, scales);
  Plan plan;
  if ((st = make_plan(dev, M, N, K, split, ks, &plan)) != MNB_OK) return st;
  Params& p = plan.p;
  p.x = static_cast<const uint16_t*>(x);
  p.q = qweight;
  p.scales = static_cast<const uint16_t*>(scales);
  p.zp = zp;
  p.y = y;
  p.out_bf16 = out_dtype == MNB_OUT_BF16;
  p.weights_ready = (flags & MNB_FLAG_WEIGHTS_READY) ? 1 : 0;

  KernelFn fn = pick_kernel(M, ks);
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan.smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = plan.grid;
  cfg.blockDim = plan.block;
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (split > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(split);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, fn, p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx");
  g_counters[0].fetch_add(1, std::memory_order_relaxed);
  g_counters[p.out_bf16 ? 2 : 1].fetch_add(1, std::memory_order_relaxed);
  if (split > 1) g_counters[3].fetch_add(1, std::memory_order_relaxed);
  g_counters[4 + M - 1].fetch_add(1, std::memory_order_relaxed);
  return MNB_OK;
}

int mnb_device_error(void* stream, unsigned int* code, int clear) {
  if (!code) return fail(MNB_ERR_NULL, "code is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_device_error, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbolAsync");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  *code = v;
  if (clear && v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbolAsync");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  }
  return MNB_OK;
}

int mnb_debug_counters(uint64_t* out, int n) {
  if (!out || n <= 0) return 0;
  const int c = std::min(n, MNB_NUM_COUNTERS);
  for (int i = 0; i < c; ++i) out[i] = g_counters[i].load(std::memory_order_relaxed);
  return c;
}

void mnb_debug_counters_reset(void) {
  for (auto& c : g_counters) c.store(0, std::memory_order_relaxed);
}

}  // extern "C"
