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
#include "mnb_dequant.cuh"
#include "mnb_launch.cuh"
#include "mnb_narrow.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <type_traits>

namespace mnb {

constexpr int kBlock = MNB_BLOCK;
constexpr int kMaxM = MNB_MAX_M;
constexpr int kMaxSplit = MNB_MAX_SPLIT_K;

// Consumer warps per CTA: 12 for M <= 2 keeps at most 4 warps (14 with the
// producer and epilogue warps) on an SM sub-partition, i.e. 128 registers per thread.
constexpr int consumer_warp_budget(int M) { return M <= 2 ? 12 : 16; }
constexpr int max_threads(int M) { return (consumer_warp_budget(M) + 2) * 32; }

// Tensor-core kernel: up to 16 K-slice consumer warps (18 warps with producer
// and epilogue); the activations, pre-paired in B-fragment order, live in
// shared memory (at most kMmaXBytes).
constexpr int kMmaWarps = 16;
constexpr int kMmaXBytes = 66 * 1024;
constexpr int kMmaThreads = (kMmaWarps + 2) * 32;
constexpr int kMmaRows = 16;                      // weight rows per tile
constexpr int kMmaSeg = 256;                      // k per segment (128 code bytes)
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
  // step kernel only
  int tr;           // 16-row sub-tiles per tile
  int wk;           // K slices = 256-k segments per stage
  int steps;        // stages per tile (K / 256 / wk)
  int wtc;          // consumer warps (wk * tr)
  int nslots;       // reduction slots
  int sc_sb;        // 16-byte scale chunks per row in a stage (odd)
  int zp_zb;        // 16-byte zero-point chunks per row in a stage (odd)
  int sc_offset;    // offset of a stage's scale box
  int zp_offset;    // offset of a stage's zero-point box
  int tx_bytes;     // bytes the three tensor copies of a stage write
  int q_bytes, sc_bytes, zp_bytes, stage_bytes;
  int bar_offset;   // shared-memory offset of the mbarrier array
  int red_offset;   // offset of the cross-warp reduction slots
  int part_offset;  // offset of the cluster partial sums
  int xp_offset;    // offset of the step kernel's staged activations
  int xp_pitch;     // bytes per activation row of those fragments
  int flag_offset;  // offset of the CTA abort flag
  int blk;          // weights per quantization block (step kernel)
  int zp_async;     // step kernel, blocks 64/128: zero-points by per-thread copies
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

// try_wait that may suspend the thread until the phase completes or about
// `ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait_for(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Calls f(std::integral_constant<int, 0>) .. f(std::integral_constant<int, N - 1>):
// an unrolled loop whose index is a compile-time constant (immediate offsets).
template <int I, int N, typename F>
__device__ __forceinline__ void static_for_from(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for_from<I + 1, N>(f);
  }
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  static_for_from<0, N>(f);
}

// Shared-memory loads at 32-bit shared addresses.  They are ordered after the
// preceding mbarrier wait (both are volatile with a memory clobber), which is
// what makes the stage's bytes visible.
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
// The same at a + OFF, OFF folded into the instruction's immediate.
template <int OFF>
__device__ __forceinline__ uint4 lds_v4_at(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Slow path of mbar_wait: polls until the phase completes, the CTA abort flag
// is raised, or kWaitLimitNs pass (then records `code` and raises the flag).
// (A try_wait with a suspend-time hint sleeps instead of polling, but was
// measured 1-4 % slower end to end on GB300, for the consumers' waits and for
// the producer's and epilogue's alike: the wake-up after the phase completes
// comes late.)
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
// Up to eight plain polls (each try_wait already blocks briefly in hardware)
// before the slow path with its deadline.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned code) {
#pragma unroll 1
  for (int i = 0; i < 8; ++i)
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



__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Zero-points of a block pair (low nibble: even block, high nibble: odd
// block) as the fp16 pairs the code extraction subtracts: 1024 + z for codes
// taken from low nibbles, 64 + z for codes taken from high nibbles.  The
// 64 + z / 1024 + z forms not produced by a mask come from the other by an
// exact fp16 shift of 960.
struct ZpPairs {
  uint32_t lo_e, hi_e, lo_o, hi_o;
};

// Byte jp of a zero-point word in the low byte of both 16-bit halves.
__device__ __forceinline__ uint32_t zp_byte_pair(uint32_t zword, int jp) {
  return __byte_perm(zword, 0u, 0x4040u | static_cast<uint32_t>(jp) | (static_cast<uint32_t>(jp) << 8));
}

// fp16 number h (0 = low half, 1 = high half) of a 32-bit word, as fp32.
__device__ __forceinline__ float half_word_to_float(uint32_t w, int h) {
  float f;
  if (h)
    asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.f32.f16 %0, hi;\n}" : "=f"(f) : "r"(w));
  else
    asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.f32.f16 %0, lo;\n}" : "=f"(f) : "r"(w));
  return f;
}

// zw: the block pair's zero-point byte in the low byte of both halves.
__device__ __forceinline__ ZpPairs zp_pairs(uint32_t zw) {
  ZpPairs z;
  z.lo_e = and_or(zw, 0x000F000Fu, 0x64006400u);             // 1024 + z_even
  z.hi_o = and_or(zw, 0x00F000F0u, 0x54005400u);             // 64 + z_odd
  z.hi_e = hsub2(z.lo_e, 0x63806380u);                       // 1024 + z - 960
  z.lo_o = hadd2(z.hi_o, 0x63806380u);                       // 64 + z + 960
  return z;
}



// One 32-block of a 16-row tile for the lane holding fragment rows g (codes
// w0, zero-point pairs zl0/zh0, scale s0) and g + 8 (w1, zl1/zh1, s1), k
// group tq: the exact code differences q - zp of word tq are the A operand of
// two m16n8k16 products with the activation fragment xf, k paired as
// (k0,k4) (k1,k5) in the first and (k2,k6) (k3,k7) in the second; the fresh
// block sum is then scaled into the fp32 accumulators.
__device__ __forceinline__ void mma_block(float (&acc)[4], uint32_t w0, uint32_t w1, uint4 xf,
                                          uint32_t zl0, uint32_t zh0, uint32_t zl1,
                                          uint32_t zh1, float s0, float s1) {
  float d[4];
  mma_16816_zero(d, hsub2(and_or(w0, 0x000F000Fu, 0x64006400u), zl0),
                 hsub2(and_or(w1, 0x000F000Fu, 0x64006400u), zl1),
                 hsub2(and_or(w0, 0x00F000F0u, 0x54005400u), zh0),
                 hsub2(and_or(w1, 0x00F000F0u, 0x54005400u), zh1), xf.x, xf.y);
  const uint32_t u0 = w0 >> 8, u1 = w1 >> 8;
  mma_16816(d, hsub2(and_or(u0, 0x000F000Fu, 0x64006400u), zl0),
            hsub2(and_or(u1, 0x000F000Fu, 0x64006400u), zl1),
            hsub2(and_or(u0, 0x00F000F0u, 0x54005400u), zh0),
            hsub2(and_or(u1, 0x00F000F0u, 0x54005400u), zh1), xf.z, xf.w, d);
  acc[0] = fmaf(d[0], s0, acc[0]);                             // row g,   m = 2tq
  acc[1] = fmaf(d[1], s0, acc[1]);                             // row g,   m = 2tq + 1
  acc[2] = fmaf(d[2], s1, acc[2]);                             // row g+8, m = 2tq
  acc[3] = fmaf(d[3], s1, acc[3]);                             // row g+8, m = 2tq + 1
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
    static_cast<uint16_t*>(y)[idx] = narrow_f16_bits_to_bf16(__half_as_ushort(h));
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

// ------------------------------------------------------------ warp roles --

// Producer (one thread): streams stage loads of RS rows -- codes of the CTA's K
// range, and the rows' scales and zero-points -- into the ring, each load
// completing on its stage's mbarrier transaction count; then lets every copy
// it issued land before the CTA may exit.
__device__ __forceinline__ void run_producer(const Params& p, unsigned char* smem, uint32_t full0,
                                             uint32_t empty0, volatile int* abort_flag,
                                             int row_begin, int row_end, int RS, int nstages,
                                             int k_begin, int k_len) {
  const int split = p.split;
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

// Epilogue (one warp): for each tile of RC rows, in tile order, adds the
// K-slice partial sums of every (row, m) value in slice order, rounds and
// stores them (or keeps them for the cluster reduction), then frees the slot.
// Tile i belongs to group i % groups, its (i / groups)-th tile; each group has
// `nslots` reduction slots.
__device__ __forceinline__ void run_epilogue(const Params& p, const float* red, float* part,
                                             uint32_t ready0, uint32_t free0,
                                             volatile int* abort_flag, int row_begin,
                                             int row_end, int RC, int ntiles, int M, int lane,
                                             int nslots) {
  wait_prerequisites();
  const int vals_tile = RC * M;
  int g = 0, t = 0;
  for (int i = 0; i < ntiles; ++i) {
    const int j = g * nslots + t % nslots;
    if (!mbar_wait(ready0 + 8u * j, (t / nslots) & 1, abort_flag, kErrReduceSlot)) break;
    const int r0 = row_begin + i * RC;
    const int vals = min(RC, row_end - r0) * M;
    const float* slot = red + static_cast<size_t>(j) * p.wpg * vals_tile;
    for (int e = lane; e < vals; e += 32) {
      float sum = 0.f;
      for (int w = 0; w < p.wpg; ++w) sum += slot[w * vals_tile + e];
      const int r = e / M, m = e % M;
      if (p.split == 1)
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
}

// ------------------------------------------------------------------ kernel --

namespace {

template <int M, int KPL, int RC>
__global__ void __launch_bounds__(max_threads(M), 1) mnb_gemv_rowtile_kernel(const Params p) {
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
  //   empty[s]  (stage)  one arrival per consumer warp: every consumer warp
  //                      passes every stage load in order (so no parity wait
  //                      can alias an older phase), and arrives once it holds
  //                      the data of its group's tiles there in registers
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
      mbar_init(empty0 + 8u * s, p.groups * p.wpg);
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
    if (lane == 0)
      run_producer(p, smem, full0, empty0, abort_flag, row_begin, row_end, RS, nstages, k_begin,
                   k_len);
    __syncwarp();
  } else if (warp == epilogue_warp) {
    // ------------------------------------------------------------ epilogue --
    run_epilogue(p, red, part, ready0, free0, abort_flag, row_begin, row_end, RC, ntiles, M, lane,
                 kSlotsPerGroup);
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
    // Stage load si (slot s, its ph-th use mod 2) holds tiles
    // [si * TPS, si * TPS + TPS); this group's tiles are g, g + groups, ...
    int s = 0;
    uint32_t ph = 0;
    int i = g;                                          // this group's next tile
    int t = 0;                                          // this group's tile counter
    bool run = true;
    for (int si = 0; si < nstages && run; ++si) {
      if (!mbar_wait(full0 + 8u * s, ph, abort_flag, kErrStageData)) break;
      const int stage_end = min(ntiles, (si + 1) * TPS);
      bool held = true;
      for (; i < stage_end; i += p.groups, ++t) {
        const int ti = i - si * TPS;
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
        if (i + p.groups >= stage_end) {                  // last tile of this group here
          __syncwarp();
          if (lane == 0) mbar_arrive(empty0 + 8u * s);
          held = false;
        }

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
            !mbar_wait(free0 + 8u * j, ((t / kSlotsPerGroup) - 1) & 1, abort_flag, kErrReduceSlot)) {
          run = false;
          break;
        }
        if ((lane & ((1 << kOwnerShift) - 1)) == 0 && idx < kVals)
          red[(static_cast<size_t>(j) * p.wpg + wg) * kVals + idx] = total;
        __syncwarp();
        if (lane == 0) mbar_arrive(ready0 + 8u * j);
      }
      if (held) {                                       // no tile of this group here
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * s);
      }
      if (++s == p.stages) {
        s = 0;
        ph ^= 1u;
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

}  // namespace


// ------------------------------------------------------------- step kernel --
//
// Weight tiles stream in through TMA tensor copies; the multiply-accumulate
// runs on CUDA cores by default (see mnb_gemv_step_kernel) or, on request, on the
// tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulation):
//   A = 16 weight rows x 16 k: lane (g, t) holds code word t (k = 8t..8t+7 of
//       the block) of rows g and g+8, dequantized exactly to q - zp by the same
//       lop3 + packed subtraction as the CUDA-core kernel; the word's pairs
//       (k0,k4) (k1,k5) feed one mma and (k2,k6) (k3,k7) the next, so the two
//       mmas cover the 32-block.
//   B = the same 16 k of activation row m = g (rows g >= M re-read row M - 1;
//       their D columns are never stored), paired the same way; the whole
//       activation block is staged once per CTA in shared memory in this
//       fragment order (16 bytes per lane and block).
//   D = 16 rows x 8 activation rows, fresh per block, multiplied by the rows'
//       fp32 scales into fp32 accumulators.
// Products of fp16 codes and activations are exact in the fp32 accumulate.
//
// Work: a CTA owns a contiguous range of tiles of R = 16 * tr rows.  A tile
// is streamed in K steps; step sigma is one stage holding R rows x W_k
// consecutive 256-k segments (codes, scales, zero-points), loaded by three TMA
// tensor copies.  Consumer warp (slice ks, sub-tile rho) multiplies rows
// 16 rho .. 16 rho + 15 by segment ks of every stage, so slice ks owns
// segments ks, ks + W_k, ...; the epilogue warp sums the W_k slice partials of
// each output in slice order.  Every consumer warp uses every stage, in
// order, and arrives on its empty barrier, so a stage is refilled only after
// all of them have passed it and no parity wait can alias an older phase.
//
// Shared-memory layout of a stage:
//   codes : box {128 B, R rows, W_k segments} of the code matrix viewed as
//           (byte in segment, row, segment), 128-byte swizzle: chunk j
//           (block 8s + j) of row r of segment s lands at
//           (R s + r) * 128 + 16 * (j ^ (r & 7)), so the eight rows a
//           fragment load touches sit in eight different bank groups.
//   scales: box {8 scales, sc_sb chunks, R rows} of (scale in chunk, chunk,
//           row), no swizzle: the 8 scales of segment s of row r at
//           (r * sc_sb + s) * 16; sc_sb is odd (a chunk past the stage is
//           loaded or zero-filled) so rows land in different bank groups.
//   zeros : box {16 B, zp_zb chunks, R rows} of (byte, chunk, row), starting
//           at the chunk holding the stage's first segment: the 4 zero-point
//           bytes of global segment G of row r at
//           (r * zp_zb + G / 4 - first chunk) * 16 + 4 (G % 4); zp_zb odd.
// Rows past N are zero-filled by the copies and never stored.

// Per-thread asynchronous copies of 4 or 8 bytes, and the arrival on an
// mbarrier once all of the thread's earlier copies have landed (the barrier's
// expected count includes it: .noinc).
template <int kBytes>
__device__ __forceinline__ void cp_async_small(uint32_t dst, const void* src) {
  static_assert(kBytes == 4 || kBytes == 8, "cp.async size");
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(kBytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Weight stages the step kernel's producer keeps in flight until the
// consumers have staged the activations; afterwards the ring alone bounds it.
// The activation loads, issued when the dependency wait returns, then queue
// behind at most two stages of weights instead of a whole ring (gate-up
// 18.1 -> 17.5 us, M = 2 14.3 -> 13.4 us; one stage in flight starves the
// stream: lm-head 62 -> 72 us).
constexpr int kMaxInflight = 2;

// Producer of the step kernel (one thread): one stage per (tile, part), three
// tensor copies completing on the stage's mbarrier.
template <int kB>
__device__ __forceinline__ void run_tc_producer(const Params& p, unsigned char* smem,
                                                uint32_t full0, uint32_t empty0,
                                                volatile int* abort_flag, int t_begin,
                                                int nunits, const CUtensorMap* tm_q,
                                                const CUtensorMap* tm_sc,
                                                const CUtensorMap* tm_zp, int lane) {
  prefetch_tensor_map(tm_q);
  prefetch_tensor_map(tm_sc);
  prefetch_tensor_map(tm_zp);
  if (!p.weights_ready) wait_prerequisites();
  const int R = kMmaRows * p.tr;
  int issued = 0, s = 0, step = 0, tile = t_begin;
  uint32_t ph = 0;
  int sl = 0;                       // stage of unit i - kMaxInflight, and its phase
  uint32_t phl = 0;
  for (int i = 0; i < nunits; ++i) {
    // the producer sleeps in the barrier until the stage is released (4 us
    // at most per call) so it refills the stage as soon as it is free
    if (i >= p.stages && !mbar_try_wait_for(empty0 + 8u * s, ph ^ 1u, 4000u) &&
        !mbar_wait(empty0 + 8u * s, ph ^ 1u, abort_flag, kErrStageFree))
      break;
    if (kMaxInflight < p.stages && i >= kMaxInflight && abort_flag[1] == 0) {
      // unit i - kMaxInflight must have landed; its stage is refilled only at
      // unit i - kMaxInflight + stages > i, so the parity wait cannot alias
      if (!mbar_wait(full0 + 8u * sl, phl, abort_flag, kErrStageData)) break;
      if (++sl == p.stages) {
        sl = 0;
        phl ^= 1u;
      }
    }
    const uint32_t st = smem_u32(smem + static_cast<size_t>(s) * p.stage_bytes);
    const uint32_t bar = full0 + 8u * s;
    const int row0 = tile * R;
    const int seg0 = step * p.wk;
    if (kB == 32 || lane == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(p.tx_bytes));
      tma_load_3d(st, tm_q, 0, row0, seg0, bar);
    }
    if constexpr (kB == 32) {
      tma_load_3d(st + p.sc_offset, tm_sc, 0, seg0, row0, bar);
      if (p.zp) tma_load_3d(st + p.zp_offset, tm_zp, 0, seg0 >> 2, row0, bar);
    } else {
      // the boxes start at the 8-scale and 32-block zero-point chunks holding
      // the stage's first quantization block
      const int bs0 = seg0 * (kMmaSeg / kB);
      if (lane == 0) {
        tma_load_3d(st + p.sc_offset, tm_sc, 0, bs0 >> 3, row0, bar);
        if (p.zp && !p.zp_async) tma_load_3d(st + p.zp_offset, tm_zp, 0, bs0 >> 5, row0, bar);
      }
      if constexpr (kB >= 64) {
        if (p.zp_async) {
          // Zero-point rows of K / (2 kB) bytes that are not whole 16-byte
          // chunks (no tensor map): the whole warp copies, row by row, the
          // 8-byte (kB = 64) or 4-byte (kB = 128) words holding the stage's
          // zero-point bytes to the places the tensor copy would use (row r's
          // box starts at byte b_lo of the row); each lane then arrives on
          // the stage's full barrier once its copies have landed.
          constexpr int kW = kB == 64 ? 8 : 4;
          const int rowbytes = p.K / (2 * kB);
          const int b_lo = 16 * (bs0 >> 5);
          const int need_lo = (bs0 >> 1) / kW * kW;
          const int need_hi = min(rowbytes, ((bs0 + p.wk * (kMmaSeg / kB)) / 2 + kW - 1) / kW * kW);
          const int words = (need_hi - need_lo) / kW;
          const int rows = min(R, p.N - row0);
          const uint32_t dst0 = st + p.zp_offset + (need_lo - b_lo);
          const uint8_t* src0 = p.zp + need_lo;
          for (int r = lane; r < rows; r += 32)
            for (int w = 0; w < words; ++w)
              cp_async_small<kW>(dst0 + r * p.zp_zb * 16 + w * kW,
                                 src0 + static_cast<size_t>(row0 + r) * rowbytes + w * kW);
          cp_async_arrive_noinc(bar);
        }
      }
    }
    issued = i + 1;
    if (++step == p.steps) {
      step = 0;
      ++tile;
    }
    if (++s == p.stages) {
      s = 0;
      ph ^= 1u;
    }
  }
  if constexpr (kB >= 64) {
    if (p.zp_async) cp_async_wait_all();
  }
  for (int i = max(0, issued - p.stages); i < issued; ++i) {
    const int si = i % p.stages;
    if (!mbar_try_wait(full0 + 8u * si, (i / p.stages) & 1)) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(full0 + 8u * si, (i / p.stages) & 1)) {
        if (global_ns() - t0 > kWaitLimitNs) {
          atomicCAS(&g_device_error, 0u, kErrDrain);
          break;
        }
      }
    }
  }
}

// Math of the step kernel: CUDA-core with four rows per lane (M = 2, 3),
// CUDA-core with two rows per lane and shared activation loads (M = 1 and
// M >= 4, and every M for blocks 16, 64 and 128), or tensor-core (on
// request).
enum StepMath : int { kMathFma = 0, kMathWide = 1, kMathMma = 2 };

namespace {

template <int M, int kMath, int kB = 32>
__global__ void __launch_bounds__(kMmaThreads, 1)
    mnb_gemv_step_kernel(const Params p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_sc,
                    const __grid_constant__ CUtensorMap tm_zp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle is a function of address bits 7-9: align to 1 KB
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int W = p.wtc;                                 // consumer warps
  const int producer_warp = W;
  const int epilogue_warp = W + 1;
  const int nslots = p.nslots;
  const int R = kMmaRows * p.tr;                       // rows per tile
  const int vals = R * M;                              // outputs per tile

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_offset);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * p.stages;
  const uint32_t ready0 = empty0 + 8u * p.stages;
  const uint32_t free0 = ready0 + 8u * nslots;
  float* red = reinterpret_cast<float*>(smem + p.red_offset);     // [slots][slices][R * M]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.flag_offset);

  const int tiles = (p.N + R - 1) / R;
  const int t_begin = static_cast<int>((static_cast<long long>(blockIdx.x) * tiles) / gridDim.x);
  const int t_end = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * tiles) / gridDim.x);
  const int ntiles = t_end - t_begin;
  const int row_begin = t_begin * R;
  const int row_end = min(p.N, t_end * R);

  if (threadIdx.x == 0) {
    // full: the producer's expect_tx arrival, plus one per producer lane
    // when the zero-points come by per-thread copies
    const uint32_t full_count = kB >= 64 && p.zp_async ? 33u : 1u;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8u * s, full_count);
      mbar_init(empty0 + 8u * s, W);
    }
    for (int j = 0; j < nslots; ++j) {
      mbar_init(ready0 + 8u * j, W);
      mbar_init(free0 + 8u * j, 1);
    }
    *abort_flag = 0;
    abort_flag[1] = 0;                                   // activations staged
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  allow_dependents();

  if (warp == producer_warp) {
    if (lane == 0 || (kB >= 64 && p.zp_async))
      run_tc_producer<kB>(p, smem, full0, empty0, abort_flag, t_begin, ntiles * p.steps, &tm_q,
                          &tm_sc, &tm_zp, lane);
    __syncwarp();
    return;
  }
  if (warp == epilogue_warp) {
    // p.wpg is the number of K-slice partials per output here
    run_epilogue(p, red, nullptr, ready0, free0, abort_flag, row_begin, row_end, R, ntiles, M,
                 lane, p.nslots);
    return;
  }

  // ------------------------------------------------------------- consumers --
  const int ks = warp / p.tr;                               // K slice (segment in a stage)
  const int rho = warp - ks * p.tr;                         // 16-row sub-tile

  // Activations, staged once per CTA by the consumer warps: row m, block b,
  // k group tq -> 16 bytes holding x[m][32b + 8tq + {0..7}] paired (0,4)
  // (1,5) (2,6) (3,7), at xp + m * xp_pitch + b * 64 + tq * 16 (the B
  // fragments of the tensor-core math) or xp + b * (64 M + 16) + (tq * M + m)
  // * 16 (CUDA-core math: a lane's block holds all M rows at offsets fixed at
  // compile time, and the 16-byte pad puts the 8 blocks a quarter warp reads
  // at once (four rows per lane) or the 4 blocks a warp reads (two rows per
  // lane) in different bank groups).
  // Each math's consumers compute their lane constants first and then stage
  // the activations: the constants' parameter loads overlap the dependency
  // wait instead of following the staging barrier.
  unsigned char* xp = smem + p.xp_offset;
  auto x_at = [&](int m, int rem) {
    return kMath == kMathMma ? m * p.xp_pitch + rem * 16
                             : (rem >> 2) * (64 * M + 16) + ((rem & 3) * M + m) * 16;
  };
  auto stage_activations = [&]() {
    if (p.zp == nullptr) {
      // symmetric format: the producer copies no zero-points; every stage's
      // zero-point bytes hold 0x88 (zero-point 8 in both nibbles) for the
      // whole launch, written before the dependency wait (they depend on no
      // earlier grid) and before the barrier below, so before any consumer
      // reads a stage
      for (int s = 0; s < p.stages; ++s)
        for (int i = threadIdx.x; i < p.zp_bytes / 16; i += W * 32)
          *reinterpret_cast<uint4*>(smem + static_cast<size_t>(s) * p.stage_bytes + p.zp_offset +
                                    16 * i) = make_uint4(0x88888888u, 0x88888888u, 0x88888888u,
                                                         0x88888888u);
    }
    wait_prerequisites();
    // 8 activations (one k group of a block) per element; K is a multiple of
    // 1024, so every row starts 16-byte aligned when x does.
    const int per_row = p.C * 4;
    if ((reinterpret_cast<uintptr_t>(p.x) & 15u) == 0) {
      // The rows are contiguous: element e is row e / per_row.  A thread
      // issues up to four loads before its first store, so the vector
      // arrives in one round trip behind the weight stream, not several.
      const uint4* xg = reinterpret_cast<const uint4*>(p.x);
      const int total = M * per_row;
      const int nthr = W * 32;
      for (int e0 = threadIdx.x; e0 < total; e0 += 4 * nthr) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (e0 + u * nthr < total) v[u] = __ldg(xg + e0 + u * nthr);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = e0 + u * nthr;
          if (e < total) {
            const int m = M == 1 ? 0 : e / per_row;
            *reinterpret_cast<uint4*>(xp + x_at(m, e - m * per_row)) = pair_k4(v[u]);
          }
        }
      }
    } else {
      for (int m = 0; m < M; ++m)
        for (int rem = threadIdx.x; rem < per_row; rem += W * 32) {
          const uint16_t* src = p.x + static_cast<size_t>(m) * p.K + 8 * rem;
          uint4 v;
          v.x = __ldg(src + 0) | (static_cast<uint32_t>(__ldg(src + 1)) << 16);
          v.y = __ldg(src + 2) | (static_cast<uint32_t>(__ldg(src + 3)) << 16);
          v.z = __ldg(src + 4) | (static_cast<uint32_t>(__ldg(src + 5)) << 16);
          v.w = __ldg(src + 6) | (static_cast<uint32_t>(__ldg(src + 7)) << 16);
          *reinterpret_cast<uint4*>(xp + x_at(m, rem)) = pair_k4(v);
        }
    }
    // all consumer warps (named barrier 1; producer and epilogue do not take part)
    asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");
    if (threadIdx.x == 0) abort_flag[1] = 1;
  };
  if constexpr (kMath == kMathMma) {
    const int gq = lane >> 2;                               // fragment row group
    const int tq = lane & 3;                                // fragment k group
    const int row_l = rho * kMmaRows + gq;                  // fragment row in the tile
    // Lanes of activation rows gq >= M read row M - 1: their D columns are
    // never stored.
    const unsigned char* xfrag = xp + min(gq, M - 1) * p.xp_pitch + ks * 512 + tq * 16;

    // Lane offsets inside a stage, the same for every stage.  Codes: row row_l
    // of segment ks, chunk j at (R ks + row_l) * 128 + 16 * (j ^ gq) + 4 tq;
    // row row_l + 8 is 1024 bytes on.
    uint32_t qoff[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) qoff[j] = (R * ks + row_l) * 128 + 16 * (j ^ gq) + 4 * tq;
    const int sc_lane = p.sc_offset + (row_l * p.sc_sb + ks) * 16;
    const int sc_hi = 8 * p.sc_sb * 16;                      // row row_l + 8
    const int zp_lane = p.zp_offset + row_l * p.zp_zb * 16;
    const int zp_hi = 8 * p.zp_zb * 16;
    stage_activations();

    int s = 0;                                               // stage of the next unit
    uint32_t ph = 0;
    bool run = true;
    for (int t = 0; t < ntiles && run; ++t) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const unsigned char* xs = xfrag;
      for (int step = 0; step < p.steps; ++step, xs += p.wk * 512) {
        if (!mbar_wait(full0 + 8u * s, ph, abort_flag, kErrStageData)) {
          run = false;
          break;
        }
        const unsigned char* st = smem + static_cast<size_t>(s) * p.stage_bytes;
        const uint4 sca = *reinterpret_cast<const uint4*>(st + sc_lane);
        const uint4 scb = *reinterpret_cast<const uint4*>(st + sc_lane + sc_hi);
        const int seg0 = step * p.wk;                        // the stage's first segment
        const int G = seg0 + ks;                             // this warp's segment
        const int zo = zp_lane + ((G >> 2) - (seg0 >> 2)) * 16 + (G & 3) * 4;
        const uint32_t zwa = *reinterpret_cast<const uint32_t*>(st + zo);
        const uint32_t zwb = *reinterpret_cast<const uint32_t*>(st + zo + zp_hi);
        const uint32_t scw_a[4] = {sca.x, sca.y, sca.z, sca.w};
        const uint32_t scw_b[4] = {scb.x, scb.y, scb.z, scb.w};
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {                     // block pair (2 jp, 2 jp + 1)
          const ZpPairs z0 = zp_pairs(zp_byte_pair(zwa, jp));
          const ZpPairs z1 = zp_pairs(zp_byte_pair(zwb, jp));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = 2 * jp + h;
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(st + qoff[j]);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(st + qoff[j] + 1024);
            const uint4 xf = *reinterpret_cast<const uint4*>(xs + 64 * j);
            const float sa = half_word_to_float(scw_a[jp], h);
            const float sb = half_word_to_float(scw_b[jp], h);
            if (h == 0)
              mma_block(acc, w0, w1, xf, z0.lo_e, z0.hi_e, z1.lo_e, z1.hi_e, sa, sb);
            else
              mma_block(acc, w0, w1, xf, z0.lo_o, z0.hi_o, z1.lo_o, z1.hi_o, sa, sb);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * s);
        if (++s == p.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!run) break;

      const int j = t % nslots;
      if (t >= nslots && !mbar_wait(free0 + 8u * j, ((t / nslots) - 1) & 1, abort_flag,
                                    kErrReduceSlot))
        break;
      float* slot = red + (static_cast<size_t>(j) * p.wpg + ks) * vals;
      const int m0 = 2 * tq;
      if (m0 < M) {
        slot[row_l * M + m0] = acc[0];
        slot[(row_l + 8) * M + m0] = acc[2];
      }
      if (m0 + 1 < M) {
        slot[row_l * M + m0 + 1] = acc[1];
        slot[(row_l + 8) * M + m0 + 1] = acc[3];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ready0 + 8u * j);
    }
  } else if constexpr (kMath == kMathFma) {
    // CUDA-core math.  Lane (rg, j) = (lane >> 3, lane & 7) takes block j of
    // the warp's segment of every stage for rows 16 rho + rg + 4 i, i = 0..3:
    // one 16-byte code load per row, exact q - zp pairs, and fp32 accumulation
    // of the fp16 products (fma.rn.f32.f16); each block sum is scaled into the
    // row's accumulator.  A tile ends with a butterfly over the eight lanes of
    // a row and one partial per (row, m) for the epilogue.
    //
    // Every shared-memory address is a 32-bit offset fixed per lane except
    // for the stage base (advanced by a whole stage) and the activation base
    // (advanced by W_k segments per step); the four rows' products form four
    // independent fp32 chains, interleaved k group by k group.
    const int j = lane & 7;
    const int rg = lane >> 3;
    const int r0 = rho * kMmaRows + rg;                   // rows r0 + 4 i
    const uint32_t zsh = (j & 1) * 4;                     // this block's nibble in its zp byte
    // rows i and i + 2 share their swizzle: row i + 2 is 1024 bytes on
    const uint32_t q_lane0 = (R * ks + r0) * 128 + 16 * (j ^ (r0 & 7));
    const uint32_t q_lane1 = (R * ks + r0 + 4) * 128 + 16 * (j ^ ((r0 + 4) & 7));
    const uint32_t sc_lane = p.sc_offset + (r0 * p.sc_sb + ks) * 16 + 2 * j;
    const uint32_t sc_row4 = 4 * p.sc_sb * 16;            // scale offset of row + 4
    const uint32_t zp_lane = p.zp_offset + r0 * p.zp_zb * 16 + (j >> 1);
    const uint32_t zp_row4 = 4 * p.zp_zb * 16;            // zero-point offset of row + 4
    const uint32_t ring0 = smem_u32(smem);
    const uint32_t stage_bytes = p.stage_bytes;
    const int stages = p.stages;
    const int steps = p.steps;
    const int wk = p.wk;
    constexpr uint32_t kXBlock = 64 * M + 16;            // bytes per activation block
    const uint32_t x_lane = smem_u32(xp) + (8 * ks + j) * kXBlock;   // block 8 ks + j of step 0
    const uint32_t x_step = wk * 8 * kXBlock;
    stage_activations();
    uint32_t sb = ring0, fb = full0, eb = empty0;         // stage s: data, full and empty barriers
    int s = 0;
    uint32_t ph = 0;
    bool run = true;
    int js = 0;                                          // reduction slot of tile t
    uint32_t jround = 0;                                 // and t / nslots
    for (int t = 0; t < ntiles && run; ++t) {
      float acc[4][M];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[i][m] = 0.f;
      uint32_t xa = x_lane;
      uint32_t zr = 0;                                    // first segment of the stage, mod 4
      for (int step = 0; step < steps; ++step) {
        if (!mbar_wait(fb, ph, abort_flag, kErrStageData)) {
          run = false;
          break;
        }
        // zero-point bytes of segment G = seg0 + ks sit 4 (seg0 % 4 + ks) bytes into
        // the row's box, which starts at the 16-byte chunk holding seg0
        const uint32_t zrow = sb + zp_lane + 4 * (zr + ks);
        uint4 xr[M][4];
        static_for<M * 4>([&](auto c) {
          constexpr int m = decltype(c)::value % M, g = decltype(c)::value / M;
          xr[m][g] = lds_v4_at<(g * M + m) * 16>(xa);
        });
        uint4 w[4];
        uint32_t zl[4], zh[4];
        float sc[4];
        const uint32_t qa0 = sb + q_lane0, qa1 = sb + q_lane1;
        w[0] = lds_v4_at<0>(qa0);
        w[1] = lds_v4_at<0>(qa1);
        w[2] = lds_v4_at<1024>(qa0);
        w[3] = lds_v4_at<1024>(qa1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t z = (lds_u8(zrow + i * zp_row4) >> zsh) & 0xFu;
          // the bias words need no masking: z < 16 fills bits the magic leaves clear
          zl[i] = z * 0x00010001u + 0x64006400u;                                   // 1024 + zp
          zh[i] = z * 0x00100010u + 0x54005400u;                                   //   64 + zp
          sc[i] = half_word_to_float(lds_u16(sb + sc_lane + i * sc_row4), 0);
        }
        float bs[4][M];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int m = 0; m < M; ++m) bs[i][m] = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t word = g == 0 ? w[i].x : g == 1 ? w[i].y : g == 2 ? w[i].z : w[i].w;
            const uint32_t w8 = word >> 8;
            const uint32_t d0 = hsub2(and_or(word, 0x000F000Fu, 0x64006400u), zl[i]);   // k0, k4
            const uint32_t d1 = hsub2(and_or(word, 0x00F000F0u, 0x54005400u), zh[i]);   // k1, k5
            const uint32_t d2 = hsub2(and_or(w8, 0x000F000Fu, 0x64006400u), zl[i]);     // k2, k6
            const uint32_t d3 = hsub2(and_or(w8, 0x00F000F0u, 0x54005400u), zh[i]);     // k3, k7
#pragma unroll
            for (int m = 0; m < M; ++m) {
              bs[i][m] = fma2_f16_f32(xr[m][g].x, d0, bs[i][m]);
              bs[i][m] = fma2_f16_f32(xr[m][g].y, d1, bs[i][m]);
              bs[i][m] = fma2_f16_f32(xr[m][g].z, d2, bs[i][m]);
              bs[i][m] = fma2_f16_f32(xr[m][g].w, d3, bs[i][m]);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int m = 0; m < M; ++m) acc[i][m] = fmaf(bs[i][m], sc[i], acc[i][m]);
        __syncwarp();
        if (lane == 0) mbar_arrive(eb);
        if (++s == stages) {
          s = 0;
          sb = ring0;
          fb = full0;
          eb = empty0;
          ph ^= 1u;
        } else {
          sb += stage_bytes;
          fb += 8u;
          eb += 8u;
        }
        xa += x_step;
        zr = (zr + wk) & 3u;
      }
      if (!run) break;
      // the eight blocks of each row's segment, in a fixed butterfly order
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = acc[i][m];
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
          acc[i][m] = v;
        }
      if (jround > 0 && !mbar_wait(free0 + 8u * js, (jround - 1) & 1u, abort_flag,
                                    kErrReduceSlot))
        break;
      if (j == 0) {
        float* slot = red + (static_cast<size_t>(js) * p.wpg + ks) * vals;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int m = 0; m < M; ++m) slot[(r0 + 4 * i) * M + m] = acc[i][m];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ready0 + 8u * js);
      if (++js == nslots) {
        js = 0;
        ++jround;
      }
    }
  } else {
    if constexpr (kB == 32) {
      // CUDA-core math, two rows per lane (M = 1 and M >= 4).  Lane (q, rr) =
      // (lane >> 3, lane & 7) takes rows 16 rho + rr and 16 rho + rr + 8 and the
      // block pair (2q, 2q + 1) of the warp's segment of every stage.  An
      // activation load (16 bytes of one 8-k group, shared by the eight lanes
      // of a quarter warp) feeds both rows,
      // which balances shared-memory bandwidth against the FMA pipe; a lane holds
      // 2M accumulators, 2M block sums and one group's 4M activation registers.
      // Activation offsets inside a block are compile-time constants; only the
      // block base moves (by W_k segments a step).
      const int rr = lane & 7;
      const int q = lane >> 3;
      const int r0 = rho * kMmaRows + rr;                  // rows r0 and r0 + 8 (both rr mod 8)
      // block 2q + e of row r0; row r0 + 8 is 1024 bytes on
      const uint32_t q_lane0 = (R * ks + r0) * 128 + 16 * ((2 * q) ^ rr);
      const uint32_t q_lane1 = (R * ks + r0) * 128 + 16 * ((2 * q + 1) ^ rr);
      const uint32_t sc_lane = p.sc_offset + (r0 * p.sc_sb + ks) * 16 + 4 * q;   // scales of the pair
      const uint32_t sc_row8 = 8 * p.sc_sb * 16;
      const uint32_t zp_lane = p.zp_offset + r0 * p.zp_zb * 16 + q;            // its zero-point byte
      const uint32_t zp_row8 = 8 * p.zp_zb * 16;
      constexpr uint32_t kXBlock = 64 * M + 16;                            // bytes per activation block
      const uint32_t ring0 = smem_u32(smem);
      const uint32_t stage_bytes = p.stage_bytes;
      const int stages = p.stages;
      const int steps = p.steps;
      const int wk = p.wk;
      const uint32_t x_lane = smem_u32(xp) + (8 * ks + 2 * q) * kXBlock;     // block 8 ks + 2 q
      const uint32_t x_step = wk * 8 * kXBlock;
      stage_activations();
      uint32_t sb = ring0, fb = full0, eb = empty0;
      int s = 0;
      uint32_t ph = 0;
      bool run = true;
      int js = 0;                                          // reduction slot of tile t
      uint32_t jround = 0;                                 // and t / nslots
      for (int t = 0; t < ntiles && run; ++t) {
        float acc[2][M];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int m = 0; m < M; ++m) acc[i][m] = 0.f;
        uint32_t xa = x_lane;
        uint32_t zr = 0;                                    // first segment of the stage, mod 4
        // two stages per loop pass and a branch-free ring advance: the
        // compiler overlaps one stage's loads and waits with the previous
        // stage's arithmetic (lm-head 62.4 -> 60.5 us, gate-up 17.4 -> 17.0)
#pragma unroll 2
        for (int step = 0; step < steps; ++step) {
          if (!mbar_wait(fb, ph, abort_flag, kErrStageData)) {
            run = false;
            break;
          }
          const uint32_t zrow = sb + zp_lane + 4 * (zr + ks);
          uint32_t sw[2], zw[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            sw[i] = lds_u32(sb + sc_lane + i * sc_row8);
            zw[i] = lds_u8(zrow + i * zp_row8) * 0x00010001u;   // the pair's zp byte, both halves
          }
          static_for<2>([&](auto ec) {                      // block 2q + e
            constexpr int e = decltype(ec)::value;
            // this block's codes and bias words for both rows (one block at a
            // time keeps the wide M within the register budget)
            const uint32_t qa = sb + (e ? q_lane1 : q_lane0);
            uint4 w[2];
            uint32_t zl[2], zh[2];
            w[0] = lds_v4_at<0>(qa);
            w[1] = lds_v4_at<1024>(qa);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if (e == 0) {
                zl[i] = and_or(zw[i], 0x000F000Fu, 0x64006400u);        // 1024 + z_even
                zh[i] = hsub2(zl[i], 0x63806380u);                       //   64 + z_even
              } else {
                zh[i] = and_or(zw[i], 0x00F000F0u, 0x54005400u);        //   64 + z_odd
                zl[i] = hadd2(zh[i], 0x63806380u);                       // 1024 + z_odd
              }
            }
            float bs[2][M];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int m = 0; m < M; ++m) bs[i][m] = 0.f;
            static_for<4>([&](auto gc) {
              constexpr int g = decltype(gc)::value;
              // both rows' q - zp pairs of this 8-k group, then one activation
              // row at a time
              uint32_t d[2][4];
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const uint4 wv = w[i];
                const uint32_t word = g == 0 ? wv.x : g == 1 ? wv.y : g == 2 ? wv.z : wv.w;
                const uint32_t w8 = word >> 8;
                d[i][0] = hsub2(and_or(word, 0x000F000Fu, 0x64006400u), zl[i]);   // k0, k4
                d[i][1] = hsub2(and_or(word, 0x00F000F0u, 0x54005400u), zh[i]);   // k1, k5
                d[i][2] = hsub2(and_or(w8, 0x000F000Fu, 0x64006400u), zl[i]);     // k2, k6
                d[i][3] = hsub2(and_or(w8, 0x00F000F0u, 0x54005400u), zh[i]);     // k3, k7
              }
              static_for<M>([&](auto mc) {
                constexpr int m = decltype(mc)::value;
                const uint4 xv = lds_v4_at<e * kXBlock + (g * M + m) * 16>(xa);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  bs[i][m] = fma2_f16_f32(xv.x, d[i][0], bs[i][m]);
                  bs[i][m] = fma2_f16_f32(xv.y, d[i][1], bs[i][m]);
                  bs[i][m] = fma2_f16_f32(xv.z, d[i][2], bs[i][m]);
                  bs[i][m] = fma2_f16_f32(xv.w, d[i][3], bs[i][m]);
                }
              });
            });
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float sc = half_word_to_float(sw[i], e);
#pragma unroll
              for (int m = 0; m < M; ++m) acc[i][m] = fmaf(bs[i][m], sc, acc[i][m]);
            }
          });
          __syncwarp();
          if (lane == 0) mbar_arrive(eb);
          {
            const bool wrap = ++s == stages;
            s = wrap ? 0 : s;
            sb = wrap ? ring0 : sb + stage_bytes;
            fb = wrap ? full0 : fb + 8u;
            eb = wrap ? empty0 : eb + 8u;
            ph ^= wrap ? 1u : 0u;
          }
          xa += x_step;
          zr = (zr + wk) & 3u;
        }
        if (!run) break;
        // the four block pairs of each row's segment, in a fixed butterfly order
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int m = 0; m < M; ++m) {
            float v = acc[i][m];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
            acc[i][m] = v;
          }
        if (jround > 0 && !mbar_wait(free0 + 8u * js, (jround - 1) & 1u, abort_flag,
                                      kErrReduceSlot))
          break;
        if (q == 0) {
          float* slot = red + (static_cast<size_t>(js) * p.wpg + ks) * vals;
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int m = 0; m < M; ++m) slot[(r0 + 8 * i) * M + m] = acc[i][m];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ready0 + 8u * js);
        if (++js == nslots) {
          js = 0;
          ++jround;
        }
      }
    } else {
      // Blocks of kB = 16, 64 or 128 weights: the lane layout of
      // block 32 above, with a segment holding kNbs blocks and the lane's
      // 64 k starting at block lane_blk of the warp's segment.  A stage's
      // scale box starts at the 8-scale chunk holding its first block bs0,
      // its zero-point box at the 32-block chunk holding it: a lane's scale
      // sits 2 (bs0 % 8 + ks kNbs + lane_blk) bytes into its row of the box,
      // its zero-point byte (bs0 % 32 + ks kNbs + lane_blk) / 2 bytes in.
      // kB >= 64: one block covers both 32-k units (one sum, one scale, one
      // nibble); kB = 16: each unit holds two blocks (words 0-1 and 2-3), so
      // two sums, two scales and both nibbles of one zero-point byte.
      static_assert(kB == 16 || kB == 64 || kB == 128, "block size");
      constexpr int kNbs = 256 / kB;
      const int rr = lane & 7;
      const int q = lane >> 3;
      const int r0 = rho * kMmaRows + rr;                  // rows r0 and r0 + 8
      const int lane_blk = (64 * q) / kB;
      const uint32_t q_lane0 = (R * ks + r0) * 128 + 16 * ((2 * q) ^ rr);
      const uint32_t q_lane1 = (R * ks + r0) * 128 + 16 * ((2 * q + 1) ^ rr);
      const uint32_t sc_lane = p.sc_offset + r0 * p.sc_sb * 16 + 2 * (ks * kNbs + lane_blk);
      const uint32_t sc_row8 = 8 * p.sc_sb * 16;
      const uint32_t zp_lane = p.zp_offset + r0 * p.zp_zb * 16 + (ks * kNbs + lane_blk) / 2;
      const uint32_t zp_row8 = 8 * p.zp_zb * 16;
      const uint32_t zsh = 4 * (lane_blk & 1);             // kB >= 64: the block's nibble
      constexpr uint32_t kXBlock = 64 * M + 16;
      const uint32_t ring0 = smem_u32(smem);
      const uint32_t stage_bytes = p.stage_bytes;
      const int stages = p.stages;
      const int steps = p.steps;
      const int wk = p.wk;
      const uint32_t x_lane = smem_u32(xp) + (8 * ks + 2 * q) * kXBlock;
      const uint32_t x_step = wk * 8 * kXBlock;
      stage_activations();
      uint32_t sb = ring0, fb = full0, eb = empty0;
      int s = 0;
      uint32_t ph = 0;
      bool run = true;
      int js = 0;                                          // reduction slot of tile t
      uint32_t jround = 0;                                 // and t / nslots
      for (int t = 0; t < ntiles && run; ++t) {
        float acc[2][M];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int m = 0; m < M; ++m) acc[i][m] = 0.f;
        uint32_t xa = x_lane;
        uint32_t bsm = 0;                                 // first block of the stage, mod 32
        // two stages per pass, branch-free ring advance (as for block 32)
#pragma unroll 2
        for (int step = 0; step < steps; ++step) {
          if (!mbar_wait(fb, ph, abort_flag, kErrStageData)) {
            run = false;
            break;
          }
          const uint32_t sca = sb + sc_lane + 2 * (bsm & 7u);
          const uint32_t zpa = sb + zp_lane + (bsm >> 1);
          // per row: kB >= 64 one scale and the block's zero-point nibble;
          // kB = 16 four scales (two words) and two zero-point bytes
          uint32_t sw[2], zw[2], sw2[2], zw2[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if constexpr (kB == 16) {
              const uint2 v = lds_v2(sca + i * sc_row8);
              sw[i] = v.x;                                  // blocks 4q, 4q + 1
              sw2[i] = v.y;                                 // blocks 4q + 2, 4q + 3
              const uint32_t zz = lds_u16(zpa + i * zp_row8);
              zw[i] = (zz & 0xFFu) * 0x00010001u;
              zw2[i] = (zz >> 8) * 0x00010001u;
            } else {
              sw[i] = lds_u16(sca + i * sc_row8);
              zw[i] = ((lds_u8(zpa + i * zp_row8) >> zsh) & 0xFu) * 0x00010001u;
            }
          }
          float bsw[2][M];                                // kB >= 64: the block's sum
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int m = 0; m < M; ++m) bsw[i][m] = 0.f;
          static_for<2>([&](auto ec) {                    // 32-k unit 2q + e
            constexpr int e = decltype(ec)::value;
            const uint32_t qa = sb + (e ? q_lane1 : q_lane0);
            uint4 w[2];
            uint32_t zl[2], zh[2], zl2[2], zh2[2];
            w[0] = lds_v4_at<0>(qa);
            w[1] = lds_v4_at<1024>(qa);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if constexpr (kB == 16) {
                const uint32_t zb = e ? zw2[i] : zw[i];
                zl[i] = and_or(zb, 0x000F000Fu, 0x64006400u);    // first block: 1024 + z
                zh[i] = hsub2(zl[i], 0x63806380u);                //                64 + z
                zh2[i] = and_or(zb, 0x00F000F0u, 0x54005400u);   // second block:  64 + z
                zl2[i] = hadd2(zh2[i], 0x63806380u);              //              1024 + z
              } else {
                zl[i] = zw[i] | 0x64006400u;                      // 1024 + z
                zh[i] = hsub2(zl[i], 0x63806380u);                //   64 + z
              }
            }
            float bs[2][M], bs2[2][M];                    // kB = 16: the unit's two sums
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int m = 0; m < M; ++m) bs[i][m] = bs2[i][m] = 0.f;
            static_for<4>([&](auto gc) {
              constexpr int g = decltype(gc)::value;
              constexpr bool second = kB == 16 && g >= 2;
              uint32_t d[2][4];
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const uint4 wv = w[i];
                const uint32_t word = g == 0 ? wv.x : g == 1 ? wv.y : g == 2 ? wv.z : wv.w;
                const uint32_t w8 = word >> 8;
                const uint32_t l = second ? zl2[i] : zl[i], h = second ? zh2[i] : zh[i];
                d[i][0] = hsub2(and_or(word, 0x000F000Fu, 0x64006400u), l);   // k0, k4
                d[i][1] = hsub2(and_or(word, 0x00F000F0u, 0x54005400u), h);   // k1, k5
                d[i][2] = hsub2(and_or(w8, 0x000F000Fu, 0x64006400u), l);     // k2, k6
                d[i][3] = hsub2(and_or(w8, 0x00F000F0u, 0x54005400u), h);     // k3, k7
              }
              static_for<M>([&](auto mc) {
                constexpr int m = decltype(mc)::value;
                const uint4 xv = lds_v4_at<e * kXBlock + (g * M + m) * 16>(xa);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  float& b = kB >= 64 ? bsw[i][m] : second ? bs2[i][m] : bs[i][m];
                  b = fma2_f16_f32(xv.x, d[i][0], b);
                  b = fma2_f16_f32(xv.y, d[i][1], b);
                  b = fma2_f16_f32(xv.z, d[i][2], b);
                  b = fma2_f16_f32(xv.w, d[i][3], b);
                }
              });
            });
            if constexpr (kB == 16) {
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const uint32_t sp = e ? sw2[i] : sw[i];
                const float sa = half_word_to_float(sp, 0), sc2 = half_word_to_float(sp, 1);
#pragma unroll
                for (int m = 0; m < M; ++m) {
                  acc[i][m] = fmaf(bs[i][m], sa, acc[i][m]);
                  acc[i][m] = fmaf(bs2[i][m], sc2, acc[i][m]);
                }
              }
            }
          });
          if constexpr (kB >= 64) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float sc = half_word_to_float(sw[i], 0);
#pragma unroll
              for (int m = 0; m < M; ++m) acc[i][m] = fmaf(bsw[i][m], sc, acc[i][m]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(eb);
          {
            const bool wrap = ++s == stages;
            s = wrap ? 0 : s;
            sb = wrap ? ring0 : sb + stage_bytes;
            fb = wrap ? full0 : fb + 8u;
            eb = wrap ? empty0 : eb + 8u;
            ph ^= wrap ? 1u : 0u;
          }
          xa += x_step;
          bsm = (bsm + wk * kNbs) & 31u;
        }
        if (!run) break;
        // the four 64-k pieces of each row's segment, in a fixed butterfly order
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int m = 0; m < M; ++m) {
            float v = acc[i][m];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
            acc[i][m] = v;
          }
        if (jround > 0 && !mbar_wait(free0 + 8u * js, (jround - 1) & 1u, abort_flag,
                                      kErrReduceSlot))
          break;
        if (q == 0) {
          float* slot = red + (static_cast<size_t>(js) * p.wpg + ks) * vals;
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int m = 0; m < M; ++m) slot[(r0 + 8 * i) * M + m] = acc[i][m];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ready0 + 8u * js);
        if (++js == nslots) {
          js = 0;
          ++jround;
        }
      }
    }
  }
}

}  // namespace

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
  return &mnb_gemv_rowtile_kernel<M, shape_for(M).kpl, shape_for(M).rc>;
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

// mnb_prefill_tc.cu: the prefill GEMM on tcgen05 (the default form).
int launch_prefill_tc(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                      void* y, int M, int N, int K, int block, int out_bf16, unsigned int* err,
                      int sms, cudaStream_t stream, LaunchDesc* query);

// mnb_prefill.cu: more than MNB_MAX_M activation rows.
int launch_prefill(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                   void* y, int M, int N, int K, int block, int out_bf16, int sms,
                   cudaStream_t stream, LaunchDesc* query);

// mnb_general.cu: block sizes other than 32 and the symmetric format.
int launch_general(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                   void* y, int M, int N, int K, int block, int out_bf16, int split_k, int sms,
                   cudaStream_t stream, LaunchDesc* query);

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  size_t smem_optin = 0;
  unsigned int* err = nullptr;   // this device's g_device_error
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
    void* err = nullptr;
    if ((e = cudaGetSymbolAddress(&err, g_device_error)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(device error)");
    d.err = static_cast<unsigned int*>(err);
    d.ready = true;
  }
  if (d.major != 10 || d.minor != 3)
    return fail(MNB_ERR_DEVICE, "this library is built for sm_103 (GB300) only; device is sm_" +
                                    std::to_string(d.major) + std::to_string(d.minor));
  *out = d;
  return MNB_OK;
}

int check_shape(int M, int N, int K) {
  if (M < 1 || M > kMaxM) return fail(MNB_ERR_SHAPE, "M must be in 1..4194240");
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

// Staged activations of the step kernel: 64 bytes per block and row; a row
// pitch of 64 mod 128 bytes puts two activation rows (4 lanes x 16 bytes
// each) in one shared-memory wavefront of the tensor-core fragment loads.
int mma_x_pitch(int C) { return C * 64 + ((C & 1) ? 0 : 64); }
int mma_x_bytes(int M, int C) { return M * mma_x_pitch(C); }
// CUDA-core maths: blocks of all M rows, 64 M + 16 bytes each
int wide_x_bytes(int M, int C) { return C * (64 * M + 16); }

// The step kernel takes a launch without a K split (split_k 0 or 1) when K
// is a multiple of 1024 (whole 256-k segments and 16-byte zero-point rows for
// the tensor copies), scales and zero-points are 16-byte aligned and the
// staged activations fit.  Math: tensor-core on request; otherwise CUDA-core
// with four rows and one block per lane for M = 2 and 3, and two rows and a
// block pair per lane for M = 1 (one zero-point byte and one scale word per
// row serve both blocks: 1.7 % faster than four rows at the lm_head shape)
// and M >= 4 (one activation load feeds both rows).  The two-row layout
// accepts more activations (M = 8 at K = 8192) and then runs with two
// reduction slots and as few as two stages, enough for a launch that is bound
// by its FMAs.
constexpr int kStepFmaMinM = 2;
constexpr int kStepFmaMaxM = 3;
constexpr int kWideXBytes = 136 * 1024;

int step_math(int M, bool tensor_cores) {
  return tensor_cores ? kMathMma
                      : (M >= kStepFmaMinM && M <= kStepFmaMaxM ? kMathFma : kMathWide);
}

int step_x_bytes(int M, int C, int math) {
  return math == kMathMma ? mma_x_bytes(M, C) : wide_x_bytes(M, C);
}

bool step_shape(int M, int K, bool tensor_cores) {
  const int math = step_math(M, tensor_cores);
  const int limit = math == kMathMma ? kMmaXBytes : kWideXBytes;
  return K % 1024 == 0 && K <= 65536 && step_x_bytes(M, K / kBlock, math) <= limit;
}

// Formats the step kernel takes besides block 32: blocks 16, 64 and 128 on
// the CUDA-core math with two rows per lane (for every M).  Their zero-point
// rows (K / (2 block) bytes) come by tensor copies where they are whole
// 16-byte chunks (always for block 16) and by per-thread copies otherwise.
bool step_takes_block(int block) { return block == 16 || block == 64 || block == 128; }
bool zp_by_thread_copies(int block, int K, const void* zp) {
  return zp != nullptr && block >= 64 && K % (32 * block) != 0;
}

bool use_step(int M, int K, int split_k, const void* scales, const void* zp,
              bool tensor_cores) {
  return (split_k == 0 || split_k == 1) && step_shape(M, K, tensor_cores) &&
         (reinterpret_cast<uintptr_t>(scales) & 15u) == 0 &&
         (reinterpret_cast<uintptr_t>(zp) & 15u) == 0;
}

using MmaFn = void (*)(const Params, const CUtensorMap, const CUtensorMap, const CUtensorMap);

template <int kMath, int kB = kBlock>
MmaFn step_kernel_for(int M) {
  switch (M) {
    case 1: return &mnb_gemv_step_kernel<1, kMath, kB>;
    case 2: return &mnb_gemv_step_kernel<2, kMath, kB>;
    case 3: return &mnb_gemv_step_kernel<3, kMath, kB>;
    case 4: return &mnb_gemv_step_kernel<4, kMath, kB>;
    case 5: return &mnb_gemv_step_kernel<5, kMath, kB>;
    case 6: return &mnb_gemv_step_kernel<6, kMath, kB>;
    case 7: return &mnb_gemv_step_kernel<7, kMath, kB>;
    default: return &mnb_gemv_step_kernel<8, kMath, kB>;
  }
}

MmaFn pick_step_kernel(int M, int math, int block) {
  if (block != kBlock) {  // two rows per lane (step_takes_block)
    switch (block) {
      case 16: return step_kernel_for<kMathWide, 16>(M);
      case 64: return step_kernel_for<kMathWide, 64>(M);
      default: return step_kernel_for<kMathWide, 128>(M);
    }
  }
  if (math == kMathMma) return step_kernel_for<kMathMma>(M);
  if (math == kMathWide) return step_kernel_for<kMathWide>(M);
  switch (M) {            // four rows per lane: kStepFmaMinM <= M <= kStepFmaMaxM
    case 2: return &mnb_gemv_step_kernel<2, kMathFma>;
    default: return &mnb_gemv_step_kernel<3, kMathFma>;
  }
}

int round_up(int v, int a) { return (v + a - 1) / a * a; }
int odd_at_least(int v) { return v | 1; }

// Tile shape and stage layout of the step kernel.  Sub-tiles per tile
// (tr): the largest whose makespan, in 16-row tiles per CTA, is within 5% of
// the best and that keeps as many SMs busy; K slices: the largest divisor of
// K / 256 up to 16 / tr (at least 4 where K allows, so a stage's zero-point
// chunk is never re-read).  A stage always holds about 32 KB of codes.
int make_mma_plan(const DeviceInfo& dev, int M, int N, int K, int math, int block, Plan* plan) {
  Params& p = plan->p;
  p.blk = block;
  p.M = M;
  p.N = N;
  p.K = K;
  p.C = K / kBlock;
  p.Z = (p.C + 1) / 2;
  p.split = 1;
  p.groups = 1;
  const int S = K / kMmaSeg;
  p.xp_pitch = mma_x_pitch(p.C);
  const int x_bytes = step_x_bytes(M, p.C, math);
  const int budget = static_cast<int>(dev.smem_optin) - 1024;   // 1 KB for the alignment
  const long long tiles16 = (static_cast<long long>(N) + kMmaRows - 1) / kMmaRows;
  const long long sms = std::max(1, dev.sms);
  auto makespan = [&](int tr) {
    const long long ct = (tiles16 + tr - 1) / tr;
    return ((ct + sms - 1) / sms) * tr;
  };
  long long best = makespan(1);
  for (int tr = 2; tr <= 4; tr *= 2) best = std::min(best, makespan(tr));
  int tr = 1;
  long long used_best = -1;
  for (int c = 4; c >= 1; c /= 2) {
    if (makespan(c) * 100 > best * 105) continue;
    const long long used = std::min(sms, (tiles16 + c - 1) / c);
    if (used > used_best) {
      used_best = used;
      tr = c;
    }
  }
  const int R = kMmaRows * tr;
  // K slices: the largest divisor of S up to 16 / tr; where the stages then
  // do not fit twice beside the activations (block 16's large scale boxes
  // at large M K), the next smaller divisor
  int nslots = kSlotsPerGroup, red_bytes = 0;
  for (int wk = std::min(kMmaWarps / tr, S); wk >= 1; --wk) {
    if (S % wk) continue;
    // 8-scale and 32-block zero-point chunks one stage spans
    const int nbs = kMmaSeg / block;
    int sspan = 1, zspan = 1;
    for (int st = 0; st < S / wk; ++st) {
      const int b0 = st * wk * nbs, b1 = (st + 1) * wk * nbs - 1;
      sspan = std::max(sspan, (b1 >> 3) - (b0 >> 3) + 1);
      zspan = std::max(zspan, (b1 >> 5) - (b0 >> 5) + 1);
    }
    p.tr = tr;
    p.wk = wk;
    p.steps = S / wk;
    p.wtc = wk * tr;
    p.wpg = wk;                                      // partials per output for the epilogue
    p.sc_sb = odd_at_least(sspan);
    p.zp_zb = odd_at_least(zspan);
    p.q_bytes = R * wk * 128;
    p.sc_bytes = round_up(R * p.sc_sb * 16, 128);
    p.zp_bytes = round_up(R * p.zp_zb * 16, 128);
    p.sc_offset = p.q_bytes;
    p.zp_offset = p.q_bytes + p.sc_bytes;
    p.tx_bytes = R * (wk * 128 + p.sc_sb * 16 + p.zp_zb * 16);
    p.stage_bytes = round_up(p.q_bytes + p.sc_bytes + p.zp_bytes, 1024);
    // four reduction slots, or two when four would leave fewer than three stages
    nslots = kSlotsPerGroup;
    for (;;) {
      red_bytes = round_up(nslots * wk * R * M * 4, 16);
      const int fixed = x_bytes + red_bytes + 8 * 2 * nslots + 16;
      p.stages = std::min(kMaxStages, (budget - fixed) / (p.stage_bytes + 16));
      if (p.stages >= 3 || nslots == 2) break;
      nslots = 2;
    }
    p.nslots = nslots;
    if (p.stages >= 2) break;
  }
  if (p.stages < 2) return fail(MNB_ERR_SHAPE, "shape needs more shared memory than one SM has");
  int off = p.stages * p.stage_bytes;
  p.xp_offset = off;
  off += x_bytes;
  p.red_offset = off;
  off += red_bytes;
  p.bar_offset = off;
  off += 8 * (2 * p.stages + 2 * nslots);
  p.part_offset = off;
  p.flag_offset = off;
  off += 16;
  const long long tiles = (static_cast<long long>(N) + R - 1) / R;
  plan->smem = static_cast<size_t>(off) + 1024;
  plan->grid = dim3(static_cast<unsigned>(std::max<long long>(1, std::min<long long>(sms, tiles))));
  plan->block = dim3(static_cast<unsigned>((p.wtc + 2) * 32));
  return MNB_OK;
}

// ---------------------------------------------------------- tensor maps --
//
// The three views the step kernel copies from (see its layout notes),
// encoded with the driver's cuTensorMapEncodeTiled (fetched once through the
// runtime, no link-time dependence on libcuda).  A map depends only on the
// array's address, N, K and the tile shape (tr, wk), so encoded maps are kept in a
// small cache: static weights are encoded once.

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct MapEntry {
  const void* ptr = nullptr;
  int kind = -1, N = 0, K = 0, tr = 0, wk = 0, blk = 0;
  CUtensorMap map;
};

constexpr int kMapCache = 96;
MapEntry g_maps[kMapCache];
int g_map_next = 0;
std::mutex g_map_mutex;
EncodeTiledFn g_encode = nullptr;

enum MapKind { kMapCodes = 0, kMapScales = 1, kMapZeros = 2 };

int encode_map(MapKind kind, const void* ptr, const Params& p, CUtensorMap* out) {
  const cuuint64_t N = static_cast<cuuint64_t>(p.N);
  const cuuint64_t K = static_cast<cuuint64_t>(p.K);
  const cuuint32_t ones[3] = {1, 1, 1};
  void* base = const_cast<void*>(ptr);
  CUresult r;
  if (kind == kMapCodes) {
    // (byte in segment, row, segment): rows K/2 bytes apart, segments 128
    const cuuint64_t dims[3] = {128, N, K / kMmaSeg};
    const cuuint64_t strides[2] = {K / 2, 128};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(kMmaRows * p.tr),
                               static_cast<cuuint32_t>(p.wk)};
    r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, ones,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (kind == kMapScales) {
    // (scale in 8-scale chunk, chunk, row): rows 2 K / blk bytes apart
    const cuuint64_t B = static_cast<cuuint64_t>(p.blk);
    const cuuint64_t dims[3] = {8, K / (8 * B), N};
    const cuuint64_t strides[2] = {16, 2 * K / B};
    const cuuint32_t box[3] = {8, static_cast<cuuint32_t>(p.sc_sb),
                               static_cast<cuuint32_t>(kMmaRows * p.tr)};
    r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, base, dims, strides, box, ones,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // (byte in 16-byte chunk, chunk, row): rows K / (2 blk) bytes apart, a
    // multiple of 16 where the step kernel takes the format
    const cuuint64_t B = static_cast<cuuint64_t>(p.blk);
    const cuuint64_t dims[3] = {16, K / (32 * B), N};
    const cuuint64_t strides[2] = {16, K / (2 * B)};
    const cuuint32_t box[3] = {16, static_cast<cuuint32_t>(p.zp_zb),
                               static_cast<cuuint32_t>(kMmaRows * p.tr)};
    r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, ones,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS)
    return fail(MNB_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult " + std::to_string(r) + ")");
  return MNB_OK;
}

int tensor_map(MapKind kind, const void* ptr, const Params& p, CUtensorMap* out) {
  std::lock_guard<std::mutex> lock(g_map_mutex);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(MNB_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  for (const MapEntry& m : g_maps)
    if (m.ptr == ptr && m.kind == kind && m.N == p.N && m.K == p.K && m.tr == p.tr &&
        m.wk == p.wk && m.blk == p.blk) {
      *out = m.map;
      return MNB_OK;
    }
  MapEntry& slot = g_maps[g_map_next];
  const int st = encode_map(kind, ptr, p, &slot.map);
  if (st != MNB_OK) {
    slot.ptr = nullptr;
    return st;
  }
  slot.ptr = ptr;
  slot.kind = kind;
  slot.N = p.N;
  slot.K = p.K;
  slot.tr = p.tr;
  slot.wk = p.wk;
  slot.blk = p.blk;
  g_map_next = (g_map_next + 1) % kMapCache;
  *out = slot.map;
  return MNB_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(a), y0 = reinterpret_cast<uintptr_t>(b);
  return x0 < y0 + nb && y0 < x0 + na;
}

// The prefill path (M > MNB_MAX_M): its own checks, then one launch.
int gemm_prefill(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                 void* y, int M, int N, int K, int block, int out_dtype, int split_k,
                 unsigned int flags, void* stream, LaunchDesc* query) {
  if (block == 16) return fail(MNB_ERR_BLOCK, "the prefill path takes block 32, 64 or 128");
  if (N < 1) return fail(MNB_ERR_SHAPE, "N must be >= 1");
  if (K < kBlock || K % kBlock != 0 || K % block != 0)
    return fail(MNB_ERR_SHAPE, "K must be a positive multiple of 32 and of the block size");
  if (out_dtype != MNB_OUT_F16 && out_dtype != MNB_OUT_BF16)
    return fail(MNB_ERR_DTYPE, "out_dtype must be MNB_OUT_F16 or MNB_OUT_BF16");
  if ((reinterpret_cast<uintptr_t>(qweight) & 15u) != 0)
    return fail(MNB_ERR_ALIGN, "qweight must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(x) & 1u) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(y) & 1u))
    return fail(MNB_ERR_ALIGN, "x, scales and y must be 2-byte aligned");
  const size_t C = static_cast<size_t>(K) / block;
  const size_t ybytes = static_cast<size_t>(M) * N * 2;
  if (overlaps(y, ybytes, x, static_cast<size_t>(M) * K * 2) ||
      overlaps(y, ybytes, qweight, static_cast<size_t>(N) * K / 2) ||
      overlaps(y, ybytes, scales, static_cast<size_t>(N) * C * 2) ||
      (zp && overlaps(y, ybytes, zp, static_cast<size_t>(N) * ((C + 1) / 2))))
    return fail(MNB_ERR_ALIAS, "y overlaps an input array");
  if (split_k != 0 && split_k != 1)
    return fail(MNB_ERR_SPLITK, "split_k must be 0 or 1 on the prefill path");
  DeviceInfo dev;
  int st = device_info(&dev);
  if (st != MNB_OK) return st;
  // the tcgen05 form where the activations are 16-byte aligned (its tensor
  // copies need it) unless the mma.sync form is requested
  const bool tc = !(flags & MNB_FLAG_PREFILL_MMA_SYNC) && (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  if (tc)
    st = launch_prefill_tc(x, qweight, scales, zp, y, M, N, K, block, out_dtype == MNB_OUT_BF16,
                           dev.err, dev.sms, static_cast<cudaStream_t>(stream), query);
  else
    st = launch_prefill(x, qweight, scales, zp, y, M, N, K, block, out_dtype == MNB_OUT_BF16,
                        dev.sms, static_cast<cudaStream_t>(stream), query);
  if (st != MNB_OK || query) return st;
  g_counters[16].fetch_add(1, std::memory_order_relaxed);
  if (tc) g_counters[17].fetch_add(1, std::memory_order_relaxed);
  g_counters[0].fetch_add(1, std::memory_order_relaxed);
  g_counters[out_dtype == MNB_OUT_BF16 ? 2 : 1].fetch_add(1, std::memory_order_relaxed);
  return MNB_OK;
}

// Validates a call, picks its kernel and launch shape, and launches it; with
// `query` non-null it fills *query instead and launches nothing.
int dispatch(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
             void* y, int M, int N, int K, int block, int out_dtype, int split_k,
             unsigned int flags, void* stream, LaunchDesc* query) {
  if (flags & ~static_cast<unsigned int>(MNB_FLAG_WEIGHTS_READY | MNB_FLAG_TENSOR_CORES |
                                          MNB_FLAG_PREFILL_MMA_SYNC))
    return fail(MNB_ERR_FLAGS, "unknown flag bits");
  if (!x || !qweight || !scales || !y) return fail(MNB_ERR_NULL, "x, qweight, scales and y are required");
  if (block != 16 && block != 32 && block != 64 && block != 128)
    return fail(MNB_ERR_BLOCK, "block size must be 16, 32, 64 or 128");
  if (M > kMaxM && M <= MNB_MAX_PREFILL_M)
    return gemm_prefill(x, qweight, scales, zp, y, M, N, K, block, out_dtype, split_k, flags,
                        stream, query);
  int st = check_shape(M, N, K);
  if (st != MNB_OK) return st;
  if (K % block != 0) return fail(MNB_ERR_SHAPE, "K must be a multiple of the block size");
  if (out_dtype != MNB_OUT_F16 && out_dtype != MNB_OUT_BF16)
    return fail(MNB_ERR_DTYPE, "out_dtype must be MNB_OUT_F16 or MNB_OUT_BF16");
  if ((reinterpret_cast<uintptr_t>(qweight) & 15u) != 0)
    return fail(MNB_ERR_ALIGN, "qweight must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(x) & 1u) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(y) & 1u))
    return fail(MNB_ERR_ALIGN, "x, scales and y must be 2-byte aligned");
  const size_t C = static_cast<size_t>(K) / block;
  const size_t ybytes = static_cast<size_t>(M) * N * 2;
  if (overlaps(y, ybytes, x, static_cast<size_t>(M) * K * 2) ||
      overlaps(y, ybytes, qweight, static_cast<size_t>(N) * K / 2) ||
      overlaps(y, ybytes, scales, static_cast<size_t>(N) * C * 2) ||
      (zp && overlaps(y, ybytes, zp, static_cast<size_t>(N) * ((C + 1) / 2))))
    return fail(MNB_ERR_ALIAS, "y overlaps an input array");
  const int lo = min_split(M, K);
  const int hi = std::min(kMaxSplit, K / kBlock);
  if (split_k < 0 || split_k > hi || (split_k != 0 && split_k < lo))
    return fail(MNB_ERR_SPLITK, "split_k must be 0 or in [" + std::to_string(lo) + ", " +
                                    std::to_string(hi) + "] for this M and K");
  DeviceInfo dev;
  if ((st = device_info(&dev)) != MNB_OK) return st;
  const bool tc = (flags & MNB_FLAG_TENSOR_CORES) != 0;
  const int math = block == kBlock ? step_math(M, tc) : kMathWide;
  const bool step_format = block == kBlock || (!tc && step_takes_block(block));
  bool step = step_format && use_step(M, K, split_k, scales, zp, tc);
  Plan plan{};
  if (step && make_mma_plan(dev, M, N, K, math, block, &plan) != MNB_OK) {
    step = false;                                 // no stage layout fits: row-tile kernel
    plan = Plan{};
  }
  // the step kernel takes block 32 with or without zero-points (its stages
  // then hold constant zero-points of 8) and blocks 16, 64 and 128 (two rows
  // per lane for every M); where it does not apply, the other formats and the
  // symmetric format run one CUDA-core kernel for all of them
  if (!step && (block != kBlock || zp == nullptr)) {
    // the other formats of the family: one CUDA-core kernel for all of them
    if ((st = launch_general(x, qweight, scales, zp, y, M, N, K, block, out_dtype == MNB_OUT_BF16,
                             split_k, dev.sms, static_cast<cudaStream_t>(stream), query)) != MNB_OK ||
        query)
      return st;
    g_counters[0].fetch_add(1, std::memory_order_relaxed);
    g_counters[out_dtype == MNB_OUT_BF16 ? 2 : 1].fetch_add(1, std::memory_order_relaxed);
    g_counters[4 + M - 1].fetch_add(1, std::memory_order_relaxed);
    return MNB_OK;
  }
  const bool mma = step && math == kMathMma;
  const int split = step ? 1 : (split_k == 0 ? auto_split(M, N, K, dev.sms) : split_k);
  const KernelShape ks = pick_shape(M, K / kBlock, split, scales);
  if (!step && (st = make_plan(dev, M, N, K, split, ks, &plan)) != MNB_OK) return st;
  Params& p = plan.p;
  p.x = static_cast<const uint16_t*>(x);
  p.q = qweight;
  p.scales = static_cast<const uint16_t*>(scales);
  p.zp = zp;
  p.y = y;
  p.out_bf16 = out_dtype == MNB_OUT_BF16;
  p.weights_ready = (flags & MNB_FLAG_WEIGHTS_READY) ? 1 : 0;
  p.zp_async = step && zp_by_thread_copies(block, K, zp) ? 1 : 0;

  const void* fn = step ? reinterpret_cast<const void*>(pick_step_kernel(M, math, block))
                        : reinterpret_cast<const void*>(pick_kernel(M, ks));
  if (query) {
    query->fn = fn;
    query->name = !step ? (split > 1 ? "row-tile kernel (K split over a cluster)" : "row-tile kernel")
                  : math == kMathMma  ? "step kernel (tensor-core math)"
                  : math == kMathWide ? "step kernel (CUDA-core, two rows per lane)"
                                      : "step kernel (CUDA-core, four rows per lane)";
    query->counter = step ? 13 : -1;
    query->grid = plan.grid.x;
    query->threads = plan.block.x;
    query->cluster = static_cast<unsigned>(split);
    query->smem = plan.smem;
    return MNB_OK;
  }
  CUtensorMap maps[3];
  if (step) {
    if ((st = tensor_map(kMapCodes, qweight, p, &maps[0])) != MNB_OK ||
        (st = tensor_map(kMapScales, scales, p, &maps[1])) != MNB_OK)
      return st;
    if (zp && !p.zp_async) {
      if ((st = tensor_map(kMapZeros, zp, p, &maps[2])) != MNB_OK) return st;
    } else {
      // never copied from: no zero-points, or zero-points by per-thread copies
      maps[2] = maps[1];
      p.tx_bytes -= kMmaRows * p.tr * p.zp_zb * 16;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(fn,
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
  void* args[4] = {&p, &maps[0], &maps[1], &maps[2]};
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC");
  g_counters[0].fetch_add(1, std::memory_order_relaxed);
  g_counters[p.out_bf16 ? 2 : 1].fetch_add(1, std::memory_order_relaxed);
  if (split > 1) g_counters[3].fetch_add(1, std::memory_order_relaxed);
  g_counters[4 + M - 1].fetch_add(1, std::memory_order_relaxed);
  if (mma) g_counters[12].fetch_add(1, std::memory_order_relaxed);
  if (step) g_counters[13].fetch_add(1, std::memory_order_relaxed);
  return MNB_OK;
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
    case MNB_ERR_BLOCK: return "block size must be 16, 32, 64 or 128";
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

const char* mnb_last_cuda_error(void) { return t_detail.c_str(); }

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
  *split_k = step_shape(M, K, false) ? 1 : auto_split(M, N, K, dev.sms);
  return MNB_OK;
}

int mnb_gemv(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp, void* y,
             int M, int N, int K, int block, int out_dtype, int split_k, void* stream) {
  return mnb_gemv_flags(x, qweight, scales, zp, y, M, N, K, block, out_dtype, split_k, 0u, stream);
}

int mnb_gemv_flags(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                   void* y, int M, int N, int K, int block, int out_dtype, int split_k,
                   unsigned int flags, void* stream) {
  return dispatch(x, qweight, scales, zp, y, M, N, K, block, out_dtype, split_k, flags, stream,
                  nullptr);
}

int mnb_gemv_launch_info(const void* x, const uint8_t* qweight, const void* scales,
                         const uint8_t* zp, const void* y, int M, int N, int K, int block,
                         int out_dtype, int split_k, unsigned int flags, mnb_launch_info* info) {
  if (!info) return fail(MNB_ERR_NULL, "info is NULL");
  LaunchDesc d;
  int st = dispatch(x, qweight, scales, zp, const_cast<void*>(y), M, N, K, block, out_dtype,
                    split_k, flags, nullptr, &d);
  if (st != MNB_OK) return st;
  cudaError_t e = cudaFuncSetAttribute(d.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(d.smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  cudaFuncAttributes fa{};
  if ((e = cudaFuncGetAttributes(&fa, d.fn)) != cudaSuccess)
    return cuda_fail(e, "cudaFuncGetAttributes");
  int ctas = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas, d.fn, static_cast<int>(d.threads),
                                                         d.smem)) != cudaSuccess)
    return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  int dev = 0, max_threads = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if ((e = cudaDeviceGetAttribute(&max_threads, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) !=
      cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(max threads per SM)");
  std::memset(info, 0, sizeof(*info));
  std::snprintf(info->kernel, sizeof(info->kernel), "%s", d.name);
  info->counter = d.counter;
  info->grid = static_cast<int>(d.grid);
  info->threads = static_cast<int>(d.threads);
  info->cluster = static_cast<int>(d.cluster);
  info->dynamic_smem = static_cast<int>(d.smem);
  info->static_smem = static_cast<int>(fa.sharedSizeBytes);
  info->registers_per_thread = fa.numRegs;
  info->ctas_per_sm = ctas;
  info->max_threads_per_sm = max_threads;
  info->theoretical_occupancy =
      max_threads > 0 ? static_cast<double>(ctas) * d.threads / max_threads : 0.0;
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
