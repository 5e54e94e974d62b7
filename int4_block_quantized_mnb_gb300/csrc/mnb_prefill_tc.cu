// mnb_prefill_tc.cu -- the prefill GEMM (M > 8) on the fifth-generation tensor
// cores: tcgen05.mma with fp32 accumulators in tensor memory (TMEM).
//
// Exactness.  Each dequantized weight, taken as v = w / 16 = ((q - zp) / 16) s,
// has at most 15 significant bits (4 of q - zp, 11 of the fp16 scale) and
// |v| <= (15 / 16) 65504 < 65504, so it splits into hi = fp16(v), which never
// overflows, and lo = v - hi, where lo' = lo 2^11 is an fp16 value as well (at
// most 4 significant bits, on a grid no finer than 2^-17).  The split is exact
// for every finite fp16 scale and every code difference (checked exhaustively
// on the host).  Two fp16 GEMMs then give exact products x hi and x lo' with
// fp32 sums: y = 16 (D_hi + 2^-11 D_lo), the factor 16 exact.  No per-block
// scaling is needed, so both accumulators stay in TMEM across the whole K
// loop.  (Without the 1/16, hi = fp16((q - zp) s) would overflow for scales
// above 4367, where the exact sum may still be finite.)
//
// Tile.  A CTA computes 128 weight rows x 32, 64, 128 or 256 activation rows
// (UMMA M = 128, N = the same) in K steps of 64, through two rings of stage
// buffers in the 128-byte swizzled K-major layout the tensor core reads:
//   weights      512 dequant threads (256 at 32-row tiles, two CTAs an SM)
//                write each step's hi and lo tiles (thread = one row x 16 or
//                32 k: its codes, scale and zero-point, loaded two steps
//                ahead), regrouping the dequant's exact
//                (k, k + 4) pairs into natural k order; each warp then
//                arrives on the stage's "full" mbarrier;
//   activations  a copy warp issues each step's tile as a tiled tensor
//                copy (zero fill past K and M) onto its own "xfull" barrier
//                and, once it has landed, adds the last arrival on "full".
// An MMA warp waits on "full", issues the step's eight MMAs (hi and lo, four
// K = 16 slices each) and commits them to the step's "empty" barrier, which
// gates both refills.  The epilogue reads TMEM (warp w:
// lanes 32 (w mod 4) .. + 31, 32 or 64 columns by w / 4), forms
// D_hi + 2^-11 D_lo (D_hi alone where it is not finite), rounds once to fp16
// and, on the bf16 arm, narrows.  K may be split over a cluster of up to 8
// CTAs (the launcher weighs waves of CTAs against the reduction); their fp32
// tiles are summed in rank order through distributed shared memory.
#include "mnb.h"
#include "mnb_launch.cuh"
#include "mnb_dequant.cuh"
#include "mnb_narrow.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <string>

namespace mnb {

int fail(int status, const std::string& detail);
int cuda_fail(cudaError_t e, const char* what);
extern std::atomic<unsigned long long> g_counters[MNB_NUM_COUNTERS];

namespace {

constexpr int kTcRows = 128;                 // weight rows per CTA (UMMA M)
constexpr int kTcK = 64;                     // k per step: one 128-byte swizzle row of fp16
constexpr int kTcTile = 128 * 128;           // bytes of one 128 x 64 fp16 tile
// Per activation-tile width kTok (UMMA N: 32, 64, 128 or 256): a weight
// stage holds the hi and lo tiles of a step, an activation stage its kTok x 64
// tile; step st uses stage st % R of both (R = 3 or 4).  The dequant threads
// fill the weight stages from codes they load kAhead steps ahead, a copy warp
// the activation stages.  TMEM holds D_hi (columns 0 .. kTok - 1) and D_lo
// (kTok .. 2 kTok - 1).
constexpr int kWBuf = 2 * kTcTile;                                      // one weight stage
constexpr int tc_xbuf(int kTok) { return kTok * kTcK * 2; }             // one activation stage
// 512 dequant threads run one CTA per SM; 256 (32-row tiles) run two CTAs
// per SM with two-stage rings
constexpr int tc_wring(int kTok, int kThreads) { return kThreads == 256 ? 2 : kTok == 256 ? 3 : 4; }
constexpr int tc_xring(int kTok, int kThreads) { return tc_wring(kTok, kThreads); }   // one index for both
constexpr int kAhead = 2;                    // steps of codes in flight per dequant thread
constexpr int tc_ring_bytes(int kTok, int kThreads) {
  return tc_wring(kTok, kThreads) * kWBuf + tc_xring(kTok, kThreads) * tc_xbuf(kTok);
}
constexpr int tc_smem(int kTok, int kThreads) { return tc_ring_bytes(kTok, kThreads) + 1024 + 256; }
constexpr int tc_cols(int kTok) { return 2 * kTok; }
constexpr unsigned kTcErrMma = 5;            // device error: a pipeline wait gave up
constexpr unsigned long long kTcWaitNs = 2000000000ull;

struct TcParams {
  const uint16_t* x;
  const uint8_t* q;
  const uint16_t* scales;
  const uint8_t* zp;
  void* y;
  int M, N, K;
  int blocks, zstride, block, bshift;        // bshift = log2(block)
  int out_bf16;
  unsigned int* err;                         // the device error word (mnb_device_error)
  int ksplit;                                // CTAs of a cluster that split K (grid z)
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk j (k = 8 j .. 8 j + 7) of row r in a 128-row,
// 64-k fp16 tile in the 128-byte swizzled K-major layout: 8-row groups of
// 1024 bytes, rows of 128 bytes, chunk index XOR (r mod 8).
__device__ __forceinline__ uint32_t sw128(int r, int j) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), fp16 A
// and B (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t tc_idesc(int kTok) {
  return (1u << 4) | (static_cast<uint32_t>(kTok >> 3) << 17) | ((kTcRows >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled tile:
// start address >> 4 (bits 0-13), leading offset 1 (unused for this layout,
// bits 16-29), stride between 8-row groups 1024 >> 4 (bits 32-45), descriptor
// version 1 (bits 46-47), swizzle mode 2 = 128 bytes (bits 61-63).  Its high
// word is a constant; its low word advances by 2 for a tile 32 bytes further
// along K (addresses stay below 256 KB: no carry out of the 14-bit field).
constexpr uint32_t kDescHi = 64u | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t sw128_desc_lo(uint32_t saddr) {
  return ((saddr & 0x3FFFFu) >> 4) | (1u << 16);
}

// One MMA from the descriptors' low words (the single issuing thread builds
// no 64-bit values).
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t adesc_lo, uint32_t bdesc_lo,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 da, db;\n setp.ne.b32 p, %4, 0;\n"
      " mov.b64 da, {%1, %5};\n mov.b64 db, {%2, %5};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(adesc_lo), "r"(bdesc_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ bool tc_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long tc_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for a phase of one of the pipeline's mbarriers (stage full,
// copy landed, MMAs committed); false (and the device error word set) when it
// did not complete within the limit.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, unsigned int* err) {
  if (tc_try_wait(bar, parity)) return true;
  const unsigned long long t0 = tc_now();
  while (!tc_try_wait(bar, parity)) {
    if (tc_now() - t0 > kTcWaitNs) {
      atomicCAS(err, 0u, kTcErrMma);
      return false;
    }
  }
  return true;
}

// One tiled 2-D tensor copy (global -> this CTA's shared memory) completing
// on mbarrier bar, and the expect-tx arrival that accounts for its bytes.
__device__ __forceinline__ void tc_tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 32 consecutive TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// hi = fp16(d s) and lo' = (d s - hi) 2^11, both exact fp16, for one pair
// (d = (q - zp) / 16, so |d s| < 65504).
// For |s| <= 2 (so |hi| <= 2 and both s 2^11 and hi 2^11 stay finite) one packed fp16 FMA
// forms lo' exactly: its exact value has at most 4 significant bits and is
// no larger than |hi 2^11|, so the single rounding leaves it unchanged.
// Larger scales take the fp32 form.
__device__ __forceinline__ void split_pair(uint32_t d, float s, uint32_t s2, uint32_t s2k,
                                           bool small, uint32_t& hi, uint32_t& lo) {
  hi = hmul2(d, s2);
  if (small) {
    const uint32_t hk = hmul2(hi, 0x68006800u);                  // hi 2^11, exact
    lo = hfma2(d, s2k, hk ^ 0x80008000u);                        // d s 2^11 - hi 2^11
    return;
  }
  const __half2 dh = *reinterpret_cast<const __half2*>(&d);
  const __half2 hh = *reinterpret_cast<const __half2*>(&hi);
  const float l0 = fmaf(__low2float(dh), s, -__low2float(hh)) * 2048.f;    // exact in fp32
  const float l1 = fmaf(__high2float(dh), s, -__high2float(hh)) * 2048.f;
  const __half2 lh = __floats2half2_rn(l0, l1);                           // exact: <= 4 bits
  lo = *reinterpret_cast<const uint32_t*>(&lh);
}

// The same split when |s| <= 2 holds for the whole warp: -hi 2^11 by one
// exact multiply, then the fused form above.
__device__ __forceinline__ void split_pair_small(uint32_t d, uint32_t s2, uint32_t s2k,
                                                 uint32_t& hi, uint32_t& lo) {
  hi = hmul2(d, s2);
  lo = hfma2(d, s2k, hmul2(hi, 0xE800E800u));                  // d s 2^11 + (-hi 2^11)
}

__device__ __forceinline__ void pf_out(void* y, size_t idx, float v, int out_bf16) {
  const __half h = __float2half_rn(v);
  if (out_bf16)
    static_cast<uint16_t*>(y)[idx] = narrow_f16_bits_to_bf16(__half_as_ushort(h));
  else
    static_cast<__half*>(y)[idx] = h;
}

// kThreads dequant (and epilogue) threads plus an MMA warp and a copy warp; a
// dequant thread handles one weight row x kKPer k per step.
template <int kThreads, int kTok>
__global__ void __launch_bounds__(kThreads + 64, kThreads == 256 ? 2 : 1)
    gemm_prefill_tc(const TcParams p, const __grid_constant__ CUtensorMap tm_x) {
  constexpr int kTcTok = kTok;
  constexpr int kWR = tc_wring(kTok, kThreads), kXR = tc_xring(kTok, kThreads);
  constexpr int kTcCols = tc_cols(kTok);
  constexpr int kKPer = kTcRows * kTcK / kThreads;           // k per thread and step
  constexpr int kWords = kKPer / 8;
  constexpr int kParts = kTcK / kKPer;                       // threads per weight row
  constexpr uint32_t kXBytes = tc_xbuf(kTok);               // one activation tile
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  // weight stages, activation stages, then full[R] empty[R] xfull[R] done,
  // the TMEM address and the abort flag
  unsigned char* xstages = smem + kWR * kWBuf;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + tc_ring_bytes(kTok, kThreads));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + tc_ring_bytes(kTok, kThreads) + 224);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + tc_ring_bytes(kTok, kThreads) + 240);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n0 = blockIdx.x * kTcRows;
  const int m0 = blockIdx.y * kTcTok;
  static_assert(kWR == kXR, "the weight and activation stages of a step share an index");
  const uint32_t full0 = smem_addr(bars), empty0 = full0 + 8 * kWR, xfull0 = empty0 + 8 * kWR,
                 done = xfull0 + 8 * kXR;
  const bool is_mma = warp == kThreads / 32;                // this extra warp issues the MMAs
  const bool is_copy = warp == kThreads / 32 + 1;           // this one the activation copies

  if (tid == 0) {
    *abort_flag = 0;
    for (int r = 0; r < kWR; ++r) {
      // full: every dequant warp, plus the copy thread once the activations landed
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(full0 + 8 * r), "r"(kThreads / 32 + 1) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(empty0 + 8 * r) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(xfull0 + 8 * r) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(done) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (is_copy && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTcCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // this thread's weight row and kKPer-k part of every step
  const int wr = tid / kParts, qk = tid % kParts;    // weight row, kKPer-k part of the step
  const int wrow = min(n0 + wr, p.N - 1);            // rows past N repeat row N - 1
  const uint8_t* qrow = p.q + static_cast<size_t>(wrow) * (p.K / 2);
  const uint16_t* srow = p.scales + static_cast<size_t>(wrow) * p.blocks;
  const uint8_t* zrow = p.zp ? p.zp + static_cast<size_t>(wrow) * p.zstride : nullptr;
  // this CTA's K steps: a contiguous share of all of them (grid z, cluster rank)
  const int nsteps_all = (p.K + kTcK - 1) / kTcK;
  const int st_begin = static_cast<int>(blockIdx.z) * nsteps_all / p.ksplit;
  const int nsteps = (static_cast<int>(blockIdx.z) + 1) * nsteps_all / p.ksplit - st_begin;
  bool ok = true;

  // Each thread's global inputs of a step (its weight row's kKPer codes,
  // scale and zero-point), loaded kAhead steps ahead; past K they are zero
  // (K is a multiple of 32), as the tensor copy makes the activations there.
  struct StepIn {
    uint32_t w[kWords];
    float s;
    uint32_t z;
  };
  auto load_step = [&](int st, StepIn& in) {
    const int kk = st * kTcK + kKPer * qk;
#pragma unroll
    for (int i = 0; i < kWords; ++i) in.w[i] = 0u;
    in.s = 0.f;
    in.z = 8;
    if (kk < p.K) {
      if constexpr (kWords == 4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + kk / 2));
        in.w[0] = v.x; in.w[1] = v.y; in.w[2] = v.z; in.w[3] = v.w;
      } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(qrow + kk / 2));
        in.w[0] = v.x; in.w[1] = v.y;
      }
      const int b = kk >> p.bshift;
      in.s = __half2float(__ushort_as_half(__ldg(srow + b)));
      if (zrow) {
        const uint32_t zb = __ldg(zrow + (b >> 1));
        in.z = (b & 1) ? (zb >> 4) : (zb & 0xFu);
      }
    }
  };

  // Step st uses weight stage and activation stage st % R.  Once the MMAs of
  // their previous use have committed (empty), dequant warps write the hi and
  // lo tiles and arrive on full, and the copy thread issues the activation
  // copy (xfull) and, when it has landed, adds the last arrival on full; the
  // MMA thread waits on full, issues the step's MMAs and commits them to
  // empty, and after the last step to done.  Every wait is bounded; a wait
  // that gives up raises the abort flag and the others then give up too.
  if (warp < kThreads / 32) {
    StepIn fifo[kAhead];                             // steps st .. st + kAhead - 1
#pragma unroll
    for (int i = 0; i < kAhead; ++i)
      if (i < nsteps) load_step(st_begin + i, fifo[i]);
    int rs = 0;                                      // weight stage st % WR
    uint32_t ph = 0;                                 // parity of (st / WR)
    for (int st = 0; st < nsteps; ++st) {
      unsigned char* buf = smem + rs * kWBuf;
      const StepIn cur = fifo[0];
#pragma unroll
      for (int i = 0; i + 1 < kAhead; ++i) fifo[i] = fifo[i + 1];
      if (st + kAhead < nsteps) load_step(st_begin + st + kAhead, fifo[kAhead - 1]);
      if (st >= kWR && !tc_wait(empty0 + 8 * rs, ph ^ 1u, p.err)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      const __half sh = __float2half_rn(cur.s);      // s is an fp16 value: exact
      const uint32_t s2 = static_cast<uint32_t>(__half_as_ushort(sh)) * 0x00010001u;
      const bool small = fabsf(cur.s) <= 2.f;
      const __half shk = __float2half_rn(small ? cur.s * 2048.f : 0.f);   // exact when small
      const uint32_t s2k = static_cast<uint32_t>(__half_as_ushort(shk)) * 0x00010001u;
      // (q - zp) / 16, exact: low nibbles OR-ed under 64 (ulp 1/16) read as
      // 64 + q / 16, high nibbles under 4 (ulp 1/256) as 4 + q / 16; subtracting
      // 64 + zp / 16 or 4 + zp / 16 leaves the exact quotient
      const uint32_t zl = cur.z * 0x00010001u + 0x54005400u;                //   64 + zp / 16
      const uint32_t zh = cur.z * 0x00100010u + 0x44004400u;                //    4 + zp / 16
      // exact (q - zp) / 16 of pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7) of word
      // g, regrouped into natural k order (k0,k1) (k2,k3) (k4,k5) (k6,k7)
      auto pairs = [&](int g, uint32_t (&n)[4]) {
        const uint32_t word = cur.w[g], w8 = word >> 8;
        const uint32_t d0 = hsub2(and_or(word, 0x000F000Fu, 0x54005400u), zl);
        const uint32_t d1 = hsub2(and_or(word, 0x00F000F0u, 0x44004400u), zh);
        const uint32_t d2 = hsub2(and_or(w8, 0x000F000Fu, 0x54005400u), zl);
        const uint32_t d3 = hsub2(and_or(w8, 0x00F000F0u, 0x44004400u), zh);
        n[0] = prmt(d0, d1, 0x5410u);
        n[1] = prmt(d2, d3, 0x5410u);
        n[2] = prmt(d0, d1, 0x7632u);
        n[3] = prmt(d2, d3, 0x7632u);
      };
      auto store = [&](int g, const uint4& hi, const uint4& lo) {
        const uint32_t off = sw128(wr, kWords * qk + g);
        *reinterpret_cast<uint4*>(buf + off) = hi;
        *reinterpret_cast<uint4*>(buf + kTcTile + off) = lo;
      };
      if (__all_sync(0xFFFFFFFFu, small)) {          // the usual case: fp16 split only
#pragma unroll
        for (int g = 0; g < kWords; ++g) {
          uint32_t n[4];
          pairs(g, n);
          uint4 hi, lo;
          split_pair_small(n[0], s2, s2k, hi.x, lo.x);
          split_pair_small(n[1], s2, s2k, hi.y, lo.y);
          split_pair_small(n[2], s2, s2k, hi.z, lo.z);
          split_pair_small(n[3], s2, s2k, hi.w, lo.w);
          store(g, hi, lo);
        }
      } else {
#pragma unroll
        for (int g = 0; g < kWords; ++g) {
          uint32_t n[4];
          pairs(g, n);
          uint4 hi, lo;
          split_pair(n[0], cur.s, s2, s2k, small, hi.x, lo.x);
          split_pair(n[1], cur.s, s2, s2k, small, hi.y, lo.y);
          split_pair(n[2], cur.s, s2, s2k, small, hi.z, lo.z);
          split_pair(n[3], cur.s, s2, s2k, small, hi.w, lo.w);
          store(g, hi, lo);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(full0 + 8 * rs) : "memory");
      if (++rs == kWR) {
        rs = 0;
        ph ^= 1u;
      }
    }
    // the MMAs of the last stage have completed when done arrives
    if (!*abort_flag && !tc_wait(done, 0, p.err)) *abort_flag = 1;
  } else if (is_copy && lane == 0) {
    // activation tile of step st (k0 = 64 (st_begin + st), rows m0 ..) into
    // stage st % R: 128-byte rows, 128-byte swizzle (the MMA's layout); rows
    // past M and k past K arrive as zeros.  A stage is refilled once the
    // MMAs of its previous use have committed (empty); the copy completes on
    // its own barrier (xfull), and once it has landed this thread adds the
    // last arrival to the stage's full barrier, one step behind the issue.
    auto landed = [&](int st) {                      // false: gave up (device error set)
      return tc_wait(xfull0 + 8 * (st % kXR), (st / kXR) & 1, p.err);
    };
    auto release = [&](int st) {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(full0 + 8 * (st % kWR)) : "memory");
    };
    int issued = 0, released = 0;
    for (int st = 0; st < nsteps; ++st) {
      const int xs = st % kXR;
      if (st >= kXR && !tc_wait(empty0 + 8 * xs, ((st / kXR) - 1) & 1, p.err)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      tc_expect_tx(xfull0 + 8 * xs, kXBytes);
      tc_tma_2d(smem_addr(xstages + xs * kXBytes), &tm_x, (st_begin + st) * kTcK, m0,
                xfull0 + 8 * xs);
      issued = st + 1;
      if (st >= 1) {
        if (!landed(st - 1)) {
          *abort_flag = 1;
          break;
        }
        release(st - 1);
        released = st;
      }
    }
    if (!*abort_flag && issued == nsteps && released < nsteps) {
      if (landed(nsteps - 1))
        release(nsteps - 1);
      else
        *abort_flag = 1;
      released = nsteps;
    }
    // on an abort, copies still in flight land before the CTA's shared memory
    // is released
    if (*abort_flag)
      for (int st = released; st < issued; ++st)
        if (!landed(st)) break;
  } else if (is_mma && lane == 0) {
    for (int st = 0; st < nsteps; ++st) {
      const int rs = st % kWR, xs = st % kXR;
      if (!tc_wait(full0 + 8 * rs, (st / kWR) & 1, p.err) || *abort_flag) {
        *abort_flag = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d_hi = sw128_desc_lo(smem_addr(smem + rs * kWBuf));
      const uint32_t d_lo = d_hi + (kTcTile >> 4);
      const uint32_t d_x = sw128_desc_lo(smem_addr(xstages + xs * kXBytes));
#pragma unroll
      for (int ks = 0; ks < kTcK / 16; ++ks) {       // K = 16 slices: 32 bytes (2 units) apart
        const uint32_t acc = (st > 0 || ks > 0) ? 1u : 0u;
        tc_mma(tmem, d_hi + 2 * ks, d_x + 2 * ks, tc_idesc(kTok), acc);
        tc_mma(tmem + kTcTok, d_lo + 2 * ks, d_x + 2 * ks, tc_idesc(kTok), acc);
      }
      tc_commit(empty0 + 8 * rs);                    // frees both stages of the step
    }
    if (!*abort_flag) tc_commit(done);
  }
  __syncthreads();
  ok = *abort_flag == 0;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  // warp w < kEpiWarps: TMEM lanes 32 (w mod 4) .., a 1/(kEpiWarps/4) share
  // of the columns (at least 32 a warp)
  constexpr int kEpiWarps = kTcTok >= 128 ? kThreads / 32 : 4 * (kTcTok / 32);
  constexpr int kColsPerWarp = kTcTok / (kEpiWarps / 4);
  const int lane_base = 32 * (warp & 3);
  const int col0 = kColsPerWarp * (warp >> 2);
  const int n = n0 + lane_base + lane;
  // with a K split, the fp32 tile [activation row][weight row] goes to this
  // CTA's shared memory (the stage buffers are free) instead of to y: a
  // warp's lanes store consecutive words
  float* part = reinterpret_cast<float*>(smem);
  if (ok && warp < kEpiWarps) {
#pragma unroll 1
    for (int cc = 0; cc < kColsPerWarp / 32; ++cc) {
      const int col = col0 + 32 * cc;
      float vh[32], vl[32];
      tc_ld32(tmem + (static_cast<uint32_t>(lane_base) << 16) + col, vh);
      tc_ld32(tmem + (static_cast<uint32_t>(lane_base) << 16) + kTcTok + col, vl);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        // D_hi is non-finite whenever a term is (hi is nonzero wherever w
        // is); it then holds the exact form's value (inf, or NaN for inf x 0)
        // and D_lo, whose lo' may be 0 there, must not be added.  The factor
        // 16 undoes the weights' exact 1/16.
        const float v =
            16.f * (fabsf(vh[j]) <= 3.402823466e38f ? fmaf(vl[j], 1.f / 2048.f, vh[j]) : vh[j]);
        if (p.ksplit > 1) {
          part[(col + j) * kTcRows + lane_base + lane] = v;
        } else {
          const int m = m0 + col + j;
          if (n < p.N && m < p.M) pf_out(p.y, static_cast<size_t>(m) * p.N + n, v, p.out_bf16);
        }
      }
    }
  }
  if (p.ksplit > 1) {
    // rank r sums the r-th 1/S of the tile over the ranks in rank order
    // (distributed shared memory); the second barrier keeps every tile
    // readable until all ranks are done.  Every CTA takes both barriers.
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int share = kTcRows * kTcTok / p.ksplit;
    const uint32_t part_addr = smem_addr(part);
    if (ok) {
      for (int e = tid; e < share; e += kThreads + 64) {
        const int gidx = static_cast<int>(rank) * share + e;
        const int tok = gidx / kTcRows, row = gidx - tok * kTcRows;   // y row, column
        const uint32_t local = part_addr + 4u * static_cast<uint32_t>(gidx);
        float sum = 0.f;
        for (int r = 0; r < p.ksplit; ++r) {
          uint32_t remote;
          float v;
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(r));
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
          sum += v;
        }
        const int nn = n0 + row, m = m0 + tok;
        if (nn < p.N && m < p.M) pf_out(p.y, static_cast<size_t>(m) * p.N + nn, sum, p.out_bf16);
      }
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled from the driver, fetched once through the runtime
// (no link-time dependence on libcuda); null when the driver lacks it.
using TcEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

TcEncodeFn tc_encode_fn() {
  static std::once_flag once;
  static TcEncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TcEncodeFn>(f);
  });
  return fn;
}

}  // namespace

// Launches the tensor-memory prefill GEMM; the caller has validated the
// arguments and checked that x is 16-byte aligned.
int launch_prefill_tc(const void* x, const uint8_t* qweight, const void* scales, const uint8_t* zp,
                      void* y, int M, int N, int K, int block, int out_bf16, unsigned int* err,
                      int sms, cudaStream_t stream, LaunchDesc* query) {
  TcParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.q = qweight;
  p.scales = static_cast<const uint16_t*>(scales);
  p.zp = zp;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.block = block;
  p.bshift = block == 128 ? 7 : block == 64 ? 6 : 5;     // block 32, 64 or 128 here
  p.blocks = K / block;
  p.zstride = (p.blocks + 1) / 2;
  p.out_bf16 = out_bf16;
  p.err = err;
  // Activation tiles of 256 rows (all of TMEM) for M > 128: a CTA's dequant
  // work per step does not depend on the tile width, so the wider tile does
  // twice the products per dequantized weight (small grids split K below).
  // Smaller M takes the narrowest tile of 32, 64 or 128 rows that holds it:
  // the MMA thread's issue waits for the tensor pipe, whose work per step
  // grows with the tile width.
  const long long gx = (static_cast<long long>(N) + kTcRows - 1) / kTcRows;
  const int tok = M > 128 ? 256 : M > 64 ? 128 : M > 32 ? 64 : 32;
  const long long gy = (static_cast<long long>(M) + tok - 1) / tok;
  if (gx > 0x7FFFFFFFLL || gy > 65535) return fail(MNB_ERR_SHAPE, "prefill shape too large");
  // 32-row tiles: 256 dequant threads and two CTAs per SM (two independent
  // pipelines; measured faster there, slower at 64 and 128 rows); wider
  // tiles: 512 dequant threads and one CTA per SM
  const int dq = tok == 32 ? 256 : 512;
  const long long slots = static_cast<long long>(sms) * (dq == 256 ? 2 : 1);
  // A launch takes ceil(CTAs / resident CTAs) waves of one CTA's steps; K may be split over a
  // cluster of up to 8 CTAs (each keeping at least two steps).  256-row
  // tiles (128 KB fp32 partials) split only a grid of at most half the SM
  // count, doubling while it still fits the SMs.  Narrower tiles take the
  // split with the least waves x (steps per CTA + about three steps of
  // start and epilogue + two for the reduction of their, at most 64 KB,
  // partials).
  const int nsteps = (K + kTcK - 1) / kTcK;
  p.ksplit = 1;
  if (tok == 256) {
    while (p.ksplit < 8 && gx * gy * p.ksplit * 2 <= sms && nsteps >= 4 * p.ksplit) p.ksplit *= 2;
  } else {
    long long best = ((gx * gy + slots - 1) / slots) * (nsteps + 3);
    for (int ks = 2; ks <= 8 && nsteps >= 4 * ks; ks *= 2) {
      const long long cost =
          ((gx * gy * ks + slots - 1) / slots) * ((nsteps + ks - 1) / ks + 3 + 2);
      if (cost < best) {
        best = cost;
        p.ksplit = ks;
      }
    }
  }
  const void* fn =
      tok == 256 ? reinterpret_cast<const void*>(&gemm_prefill_tc<512, 256>)
      : tok == 128 ? reinterpret_cast<const void*>(&gemm_prefill_tc<512, 128>)
      : tok == 64 ? reinterpret_cast<const void*>(&gemm_prefill_tc<512, 64>)
                  : reinterpret_cast<const void*>(&gemm_prefill_tc<256, 32>);
  const int smem = tc_smem(tok, dq);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill tc)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                     static_cast<unsigned>(p.ksplit));
  cfg.blockDim = dim3(dq + 64);
  cfg.dynamicSmemBytes = smem;
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
  if (query) {
    query->fn = fn;
    query->name = "prefill GEMM, tcgen05 form";
    query->counter = 17;
    query->grid = cfg.gridDim.x * cfg.gridDim.y * cfg.gridDim.z;
    query->threads = cfg.blockDim.x;
    query->cluster = static_cast<unsigned>(p.ksplit);
    query->smem = cfg.dynamicSmemBytes;
    return MNB_OK;
  }
  // the activations as (k, row) fp16 pairs of bits: boxes of 64 k (one
  // 128-byte swizzle row) x tok rows, zero-filled past K and M
  const TcEncodeFn encode = tc_encode_fn();
  if (!encode) return fail(MNB_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap tm_x;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcK), static_cast<cuuint32_t>(tok)};
  const cuuint32_t ones[2] = {1, 1};
  const CUresult r = encode(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(x), dims,
                            strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MNB_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult " + std::to_string(r) + ")");
  void* args[2] = {&p, &tm_x};
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC(prefill tc)");
  return MNB_OK;
}

}  // namespace mnb
