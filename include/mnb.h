/*
 * mnb.h -- C ABI of the GB300 (sm_103a) int4 block-quantized MatMulNBits
 * decode GEMV library (libmnb.so).
 *
 * The operation (one launch computes every output element):
 *
 *     y[m,n] = round( sum_k x[m,k] * (q[n,k] - zp[n, k/B]) * scale[n, k/B] )
 *
 * with 4-bit weight codes q and 4-bit asymmetric zero-points zp at block size
 * B = 32 (also 16, 64 and 128, and the symmetric form without zero-points,
 * where every zp is 8), fp16 activations x and fp16 scales, fp32
 * accumulation, and a result
 * rounded to fp16; on request the fp16 result is narrowed to bf16 in the same
 * epilogue (fp32 -> fp16 -> bf16, two round-to-nearest-even steps).
 *
 *   - "perf(cuda): let the split-K decode GEMV store bf16 directly"
 *     (onnx-genai PR 1550), paragraphs 1-2: the block-32 split-K decode GEMV,
 *     its fp16 epilogue on one lane per output column, and the launch-uniform
 *     bf16 narrowing store that is bit-identical to casting the fp16 result.
 *     Paragraph 4 (the small-batch row loop): a launch must write every
 *     element of its output; here one call always writes all M*N elements.
 *   - "PORT-1 (offline bias+interleave) -- measured NO-GO on the multicol
 *     asymmetric-zp GEMV" (onnx-genai PR 1002), "Why the premise fails
 *     here" point 1: 4-bit weights with a per-block asymmetric zero-point,
 *     and without one the symmetric dequant with a +8 bias.  Block sizes
 *     other than 32 keep the same layout with the block size as a parameter.
 *
 * Conventions shared by every entry point:
 *   - Memory: all array arguments are device pointers owned by the caller
 *     (the library allocates nothing).  Calls are asynchronous on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream); a kernel-side fault
 *     surfaces at the caller's next synchronisation.
 *   - Errors: every entry point returns an mnb_status.  Nothing is printed and
 *     no exception crosses the ABI.  mnb_last_error_detail() returns a
 *     thread-local text describing the calling thread's last failure.
 *   - Thread safety: the entry points are re-entrant; the only shared state is
 *     a set of atomic launch counters and a per-device error word.
 */
#ifndef MNB_H_
#define MNB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MNB_ABI_VERSION 2

/* Output element type of mnb_gemv. */
typedef enum mnb_out_dtype {
    MNB_OUT_F16 = 0,   /* y holds the fp16 result */
    MNB_OUT_BF16 = 1   /* y holds bf16( fp16 result ), i.e. double-rounded; an fp16
                          NaN becomes the quiet bf16 NaN 0x7FC0 with its sign */
} mnb_out_dtype;

typedef enum mnb_status {
    MNB_OK = 0,
    MNB_ERR_NULL = 1,    /* a required pointer is NULL */
    MNB_ERR_SHAPE = 2,   /* M, N or K outside the supported range */
    MNB_ERR_BLOCK = 3,   /* block size other than 16, 32, 64 or 128 */
    MNB_ERR_DTYPE = 4,   /* out_dtype not an mnb_out_dtype */
    MNB_ERR_SPLITK = 5,  /* split_k outside [0, mnb_max_split_k] or too small for K */
    MNB_ERR_ALIGN = 6,   /* a pointer is misaligned for its element type (see mnb_gemv) */
    MNB_ERR_CUDA = 7,    /* a CUDA runtime call failed; see mnb_last_cuda_error */
    MNB_ERR_ALIAS = 8,   /* y overlaps an input array */
    MNB_ERR_DEVICE = 9,  /* the current device is not an sm_103 GPU */
    MNB_ERR_FLAGS = 10   /* unknown bits in the flags of mnb_gemv_flags */
} mnb_status;

/* Limits of mnb_gemv. */
#define MNB_MAX_M 8            /* decode batch rows per call (the GEMV kernels) */
#define MNB_MAX_PREFILL_M 4194240 /* rows of the prefill path: 65535 tiles of 64 */
#define MNB_BLOCK 32           /* quantization block along K */
#define MNB_MAX_SPLIT_K 8      /* K-partitions reduced inside one thread-block cluster */

/*
 * mnb_gemv -- the decode GEMV, all M rows in one launch.
 *
 *   x        [M][K] fp16, row-major, 2-byte aligned (16-byte alignment is
 *            faster).
 *   qweight  [N][K/2] uint8, row-major, 16-byte aligned.  Byte k/2 of row n
 *            holds code q[n,k] in its low nibble for even k and in its high
 *            nibble for odd k.
 *   scales   [N][K/block] fp16, row-major, 2-byte aligned.
 *   zp       [N][ceil(K/block/2)] uint8, row-major, any alignment.  Byte b/2
 *            of row n holds zero-point zp[n,b] in its low nibble for even
 *            block index b and in its high nibble for odd b; when K/block is
 *            odd the last high nibble of each row is ignored.  NULL selects
 *            the symmetric format: every zero-point is 8.
 *   y        [M][N] fp16 (out_dtype MNB_OUT_F16) or bf16 (MNB_OUT_BF16),
 *            row-major, 2-byte aligned, must not overlap any input.  Every
 *            one of its M*N elements is written by this call.
 *   M        1..MNB_MAX_M: the decode GEMV kernels; MNB_MAX_M + 1 ..
 *            MNB_MAX_PREFILL_M: the prefill path, a tensor-core GEMM with the
 *            same exact products, fp32 sums and epilogue (block 32, 64 or 128;
 *            split_k 0 or 1).   N >= 1.   K >= 32, a multiple of 32 and of
 *            block.
 *   block    16, 32 (MNB_BLOCK), 64 or 128.  Block 32 with zero-points runs
 *            the kernels tuned for it, and so does block 32 without them
 *            where the TMA step kernel applies (constant zero-points of 8 in
 *            its stages).  The step kernel also takes blocks 16, 64 and 128
 *            where it applies (no tensor-core flag, split_k 0 or 1, K a
 *            multiple of 1024, and the staged activations fit).  Elsewhere
 *            the other formats run one
 *            CUDA-core kernel of the same exact arithmetic, where split_k
 *            (0 = chosen by the library) is the number of warps that split
 *            each row's K range inside one CTA, at most 8.
 *   out_dtype  an mnb_out_dtype.  It changes only the final store: for the
 *            same inputs and split_k the bf16 result equals the
 *            round-to-nearest-even bf16 narrowing of the fp16 result, bit
 *            for bit.
 *   split_k  number of contiguous K ranges (whole 32-blocks) each output is
 *            split into; the ranges are reduced in a fixed order inside one
 *            thread-block cluster.  0 = chosen by the library
 *            (mnb_split_k_auto); otherwise 1..min(MNB_MAX_SPLIT_K, K/32) and
 *            at least mnb_min_split_k(M, K).  Results meet the same error
 *            bound for every split_k; the fp16 bits may differ between
 *            split_k values.
 *   stream   cudaStream_t to launch on (NULL = legacy default stream).
 *
 * Returns MNB_OK once the kernel is enqueued, or the first failing check.
 * Nothing is launched on a non-OK return.
 */
int mnb_gemv(const void *x, const uint8_t *qweight, const void *scales, const uint8_t *zp,
             void *y, int M, int N, int K, int block, int out_dtype, int split_k,
             void *stream);

/*
 * Flags of mnb_gemv_flags.
 *
 * Every GEMV launch lets the next kernel on its stream launch early
 * (programmatic dependent launch) and, before it reads or writes any caller
 * array, waits until the kernel launched before it on the stream has completed
 * and its writes are visible.  So back-to-back calls overlap launch latency
 * and drain time while keeping stream order for every array.
 *
 * MNB_FLAG_WEIGHTS_READY: the caller promises that qweight, scales and zp are
 * not written by the kernel launched just before this call on the stream (they
 * are static model weights).  The call then starts streaming them before that
 * kernel completes; x is still read, and y written, only after it completes.
 */
#define MNB_FLAG_WEIGHTS_READY 1u

/*
 * MNB_FLAG_TENSOR_CORES: permit tensor-core math in the step kernel where it
 * applies (no K split, K a multiple of 1024, scales and zp 16-byte aligned,
 * M times K at most 33792). It forms the same exact fp16 products (q - zp) * x and
 * accumulates them in fp32 with mma.sync m16n8k16 instead of fp32 FMAs;
 * results meet the same error bound and bf16 invariant, but their bits may
 * differ from the default kernels'. Without the flag no decode launch (M <=
 * MNB_MAX_M) uses a tensor-core instruction. The prefill path (M >
 * MNB_MAX_M) always runs on tensor cores and ignores this flag.
 */
#define MNB_FLAG_TENSOR_CORES 2u

/*
 * The prefill path (M > MNB_MAX_M) has two forms of one GEMM, both with exact
 * products, fp32 sums and the decode epilogue, meeting the same bound and
 * bf16 invariant (their fp16 bits may differ: different summation order):
 *   tcgen05   the default where x is 16-byte aligned.  Every dequantized
 *             weight, as v = ((q - zp) / 16) s, is split exactly into two
 *             fp16 parts (hi = fp16(v), which cannot overflow, and
 *             lo = (v - hi) 2^11; exact for every finite fp16 scale); two
 *             fp16 tcgen05 GEMMs accumulate x hi and x lo in fp32 in tensor
 *             memory and the epilogue forms 16 (hi + 2^-11 lo) (16 hi alone
 *             where it is not finite, so infinities and NaNs follow the exact
 *             form).
 *   mma.sync  per-block fp32 sums of the exact fp16 products (q - zp) x,
 *             scaled into fp32 accumulators.  Used where x is not 16-byte
 *             aligned, and on request:
 * MNB_FLAG_PREFILL_MMA_SYNC: run the mma.sync form of the prefill GEMM.  No
 * effect for M <= MNB_MAX_M.
 */
#define MNB_FLAG_PREFILL_MMA_SYNC 4u

/* mnb_gemv with flags (0 or an OR of the MNB_FLAG_* bits); mnb_gemv(...) is
 * mnb_gemv_flags(..., 0, stream).  Same arguments, checks and statuses, plus
 * MNB_ERR_FLAGS for unknown flag bits. */
int mnb_gemv_flags(const void *x, const uint8_t *qweight, const void *scales, const uint8_t *zp,
                   void *y, int M, int N, int K, int block, int out_dtype, int split_k,
                   unsigned int flags, void *stream);

/*
 * mnb_cast_f16_to_bf16 -- dst[i] = bf16(src[i]) for n elements: fp16 -> fp32
 * exactly, then round-to-nearest-even to bf16 (a NaN becomes the quiet NaN
 * 0x7FC0 with its sign), the same narrowing mnb_gemv's bf16 output applies.  It is the separate
 * narrowing launch of the staged route ("perf(cuda): let the split-K decode
 * GEMV store bf16 directly", onnx-genai PR 1550, paragraphs 1-3), provided to
 * measure that route against the direct bf16 store.
 *   src, dst  device arrays of n 16-bit values, 2-byte aligned (16-byte
 *             alignment of both is faster); dst may equal src (in place) but
 *             must not otherwise overlap it.
 * n = 0 launches nothing.  Asynchronous on `stream`; MNB_OK once enqueued.
 */
int mnb_cast_f16_to_bf16(const void *src, void *dst, size_t n, void *stream);

/* split_k that mnb_gemv uses for split_k = 0 on the current device, for
 * 16-byte aligned scales and zp and without MNB_FLAG_TENSOR_CORES (1 whenever
 * the step kernel takes the launch: K a multiple of 1024 and staged
 * activations (K / 32) * (64 M + 16) bytes at most 136 KiB).  Writes it to
 * *split_k.  Same shape checks and statuses as mnb_gemv. */
int mnb_split_k_auto(int M, int N, int K, int *split_k);

/* Smallest split_k mnb_gemv accepts for this M and K (one CTA covers at most
 * 12288 values of K when M <= 2, 16384 when M = 3 and 8192 when M >= 4).
 * Writes it to *min_split. */
int mnb_min_split_k(int M, int K, int *min_split);

/* Largest split_k mnb_gemv accepts for this K: min(MNB_MAX_SPLIT_K, K/32). */
int mnb_max_split_k(int K, int *max_split);

/* Static text for a status code (never NULL). */
const char *mnb_status_string(int status);

/* Thread-local text about the calling thread's last non-OK return (empty when
 * none).  Valid until the thread's next call into the library. */
const char *mnb_last_error_detail(void);

/* The same thread-local text, under the name that says what it holds after
 * MNB_ERR_CUDA: the failing CUDA call with its error name and message. */
const char *mnb_last_cuda_error(void);

/* Device-side error word of the current device: 0, or the first code a
 * kernel recorded when one of its bounded waits gave up (1 = stage data never
 * arrived, 2 = a stage was never released, 3 = copies still in flight at exit,
 * 4 = a reduction slot was never filled or freed, 5 = a stage, activation copy
 * or MMA completion of the tensor-memory prefill GEMM never arrived).  Enqueues a read on
 * `stream`, synchronises that stream and writes the word to *code; clears it
 * when `clear` is non-zero.  Returns MNB_ERR_CUDA if the read fails. */
int mnb_device_error(void *stream, unsigned int *code, int clear);

/*
 * mnb_launch_info -- what one mnb_gemv_flags call with these arguments would
 * launch on the current device, for measurement harnesses (registers,
 * occupancy) and tests.  Filled by mnb_gemv_launch_info; nothing is launched.
 */
typedef struct mnb_launch_info {
    char kernel[64];          /* name of the kernel family, e.g. "step kernel (CUDA-core, 4 rows/lane)" */
    int counter;              /* mnb_debug_counters index that the launch bumps for its kernel
                                 family (13 step, 15 general, 16 prefill), or -1 for the
                                 row-tile kernel, which has none of its own */
    int grid;                 /* CTAs in the grid */
    int threads;              /* threads per CTA */
    int cluster;              /* CTAs per thread-block cluster (1 = no cluster) */
    int dynamic_smem;         /* dynamic shared memory per CTA, bytes */
    int static_smem;          /* static shared memory per CTA, bytes */
    int registers_per_thread; /* registers the compiled kernel uses per thread */
    int ctas_per_sm;          /* resident CTAs per SM (occupancy calculator) */
    int max_threads_per_sm;   /* the device's limit */
    double theoretical_occupancy; /* ctas_per_sm * threads / max_threads_per_sm */
} mnb_launch_info;

/* The arguments, checks and statuses of mnb_gemv_flags (the pointers are only
 * inspected for their alignment and overlap, never dereferenced); on MNB_OK
 * *info describes the launch that call would make.  Needs an sm_103 device
 * current (MNB_ERR_DEVICE otherwise). */
int mnb_gemv_launch_info(const void *x, const uint8_t *qweight, const void *scales,
                         const uint8_t *zp, const void *y, int M, int N, int K, int block,
                         int out_dtype, int split_k, unsigned int flags, mnb_launch_info *info);

/* Launch counters, for tests that must prove the GPU kernel ran:
 *   [0] launches, [1] fp16-output launches, [2] bf16-output launches,
 *   [3] launches with split_k > 1 (cluster reduction), [4 + M - 1] launches
 *   with M rows (M = 1..8), [12] decode launches with tensor-core math (only
 *   with MNB_FLAG_TENSOR_CORES), [13] launches of the step kernel (either math:
 *   tiles streamed in K steps by TMA tensor copies, no K split), [14]
 *   launches of mnb_cast_f16_to_bf16, [15] launches of the general-format
 *   kernel (block size other than 32, or no zero-points), [16] launches of the
 *   prefill GEMM (M > MNB_MAX_M), [17] prefill launches of its tcgen05 form.
 * Copies min(n, MNB_NUM_COUNTERS) counters to out; returns how many. */
#define MNB_NUM_COUNTERS 18
int mnb_debug_counters(uint64_t *out, int n);
void mnb_debug_counters_reset(void);

/* MNB_ABI_VERSION of the loaded library. */
int mnb_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MNB_H_ */
