/*
 * mnb_oracle.c -- CPU oracle for the int4 block-quantized MatMulNBits decode GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the
 * package's smoke check and the benchmark's CPU-baseline arm load it; the
 * product library never links, includes or calls it, and it shares no code,
 * header, table or constant with the CUDA sources.
 *
 * What it computes (one output element, written out in f64):
 *
 *     y[m,n] = sum_k  x[m,k] * (q[n,k] - zp[n, k/block]) * scale[n, k/block]
 *
 *   - "perf(cuda): let the split-K decode GEMV store bf16 directly"
 *     (onnx-genai PR 1550), first two paragraphs: a block-32 split-K GEMV
 *     over INT4 weights whose epilogue rounds the fp32 accumulator to fp16,
 *     and whose bf16 arm narrows that fp16 value to bf16 (fp32 -> fp16 ->
 *     bf16, double rounding, bit-identical to casting the fp16 result).
 *   - "PORT-1 (offline bias+interleave) -- measured NO-GO on the multicol
 *     asymmetric-zp GEMV" (onnx-genai PR 1002), "Why the premise fails
 *     here", point 1: 4-bit weights with an asymmetric per-block zero-point
 *     subtracted before scaling; without a zero-point the dequant is the
 *     symmetric one with an implicit +8 bias (zp = 8).
 *
 * Layout (the plain reading of the packed format; the pages name no other):
 *   x       [M][K]            IEEE binary16 bit patterns
 *   qweight [N][K/2]          uint8, low nibble = even k, high nibble = odd k
 *   scales  [N][K/block]      IEEE binary16 bit patterns
 *   zp      [N][ceil(K/block/2)] uint8, low nibble = even block index,
 *                             high nibble = odd block index (the last high
 *                             nibble of a row is padding when K/block is odd);
 *                             NULL means symmetric (zp = 8 everywhere)
 *
 * Arithmetic: every product x * (q - zp) * scale is formed and summed in
 * IEEE double.  For fp16 inputs each product carries at most 26 significant
 * bits, so for the shapes and value ranges used here the f64 sum is exact;
 * the single rounding to fp16 is then the correctly rounded result.  The
 * fp16 result is narrowed to bf16 by a second, separate rounding.
 * Rounding is IEEE round-to-nearest, ties-to-even, written out below from
 * the binary16 / bfloat16 format definitions (1-5-10 and 1-8-7 bit fields).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* ---- format conversions ------------------------------------------------ */

/* binary16 bit pattern -> its exact value as a double. */
double mnbo_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal: f * 2^-24 */
    else if (e == 31)
        v = (f != 0) ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 bit pattern -> its exact value as a double. */
double mnbo_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* f * 2^-126 / 128 */
    else if (e == 255)
        v = (f != 0) ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a non-negative double holding a value below 2^52 to an integer,
 * ties to even. */
static double round_half_even(double m)
{
    double fl = floor(m);
    double d = m - fl;                             /* exact */
    if (d > 0.5)
        return fl + 1.0;
    if (d < 0.5)
        return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> binary16, round to nearest, ties to even.  Magnitudes at or above
 * 65520 (the midpoint between the largest finite value 65504 and 2^16)
 * overflow to infinity; below 2^-14 the quantum is the subnormal 2^-24. */
uint16_t mnbo_f64_to_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v))
        return sign | 0x7E00;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {
        double m = round_half_even(ldexp(a, 24));  /* count of 2^-24 quanta */
        return sign | (uint16_t)m;                 /* 1024 quanta = 2^-14, the smallest normal */
    }
    int e2;
    frexp(a, &e2);                                 /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;                                /* a in [2^E, 2^(E+1)) */
    double m = round_half_even(ldexp(a, 10 - E));  /* 11-bit significand, in [1024, 2048] */
    if (m == 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7C00;
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)(m - 1024.0);
}

/* binary16 -> bfloat16, round to nearest, ties to even, applied to the exact
 * fp16 value.  Every finite fp16 magnitude lies inside bfloat16's normal
 * range, so only the 8-bit significand rounds. */
uint16_t mnbo_f16_to_bf16(uint16_t h)
{
    uint16_t sign = h & 0x8000;
    double v = mnbo_f16_to_f64(h);
    if (isnan(v))
        return sign | 0x7FC0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;
    double m = round_half_even(ldexp(a, 7 - E));   /* 8-bit significand, in [128, 256] */
    if (m == 256.0) {
        m = 128.0;
        E += 1;
    }
    return sign | (uint16_t)((E + 127) << 7) | (uint16_t)(m - 128.0);
}

void mnbo_f16_to_f64_array(const uint16_t *in, double *out, size_t n)
{
    for (size_t i = 0; i < n; i++)
        out[i] = mnbo_f16_to_f64(in[i]);
}

void mnbo_bf16_to_f64_array(const uint16_t *in, double *out, size_t n)
{
    for (size_t i = 0; i < n; i++)
        out[i] = mnbo_bf16_to_f64(in[i]);
}

void mnbo_f64_to_f16_array(const double *in, uint16_t *out, size_t n)
{
    for (size_t i = 0; i < n; i++)
        out[i] = mnbo_f64_to_f16(in[i]);
}

void mnbo_f16_to_bf16_array(const uint16_t *in, uint16_t *out, size_t n)
{
    for (size_t i = 0; i < n; i++)
        out[i] = mnbo_f16_to_bf16(in[i]);
}

/* ---- packed-format accessors ------------------------------------------- */

/* 4-bit weight code of row n at position k: byte k/2 of the row, low nibble
 * for even k, high nibble for odd k. */
int mnbo_q_at(const uint8_t *qweight, int K, int64_t n, int k)
{
    uint8_t byte = qweight[(size_t)n * (size_t)(K / 2) + (size_t)(k / 2)];
    return (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
}

/* 4-bit zero-point of row n, block b: byte b/2 of the row (rows are
 * ceil(blocks/2) bytes long), low nibble for even b, high nibble for odd b.
 * Without a zero-point array the dequant is symmetric: zp = 8. */
int mnbo_zp_at(const uint8_t *zp, int K, int block, int64_t n, int b)
{
    if (zp == NULL)
        return 8;
    int blocks = K / block;
    int stride = (blocks + 1) / 2;
    uint8_t byte = zp[(size_t)n * (size_t)stride + (size_t)(b / 2)];
    return (b % 2 == 0) ? (byte & 0xF) : (byte >> 4);
}

/* ---- the GEMV ------------------------------------------------------------ */

/*
 * Computes output columns cols[0..ncols) of all M rows.  Outputs are dense
 * [M][ncols] arrays (any of them may be NULL):
 *   y_exact  the f64 sum (exact for the value ranges used here)
 *   abs_sum  sum_k |x[m,k] * w[n,k]|, the scale of the tolerance's second term
 *   y_f16    y_exact rounded once to binary16 (RNE)
 *   y_bf16   y_f16 rounded again to bfloat16 (RNE): the double-rounded arm
 * Returns 0, or -1 when the shape is not one the format defines.
 */
int mnbo_gemv_cols(const uint16_t *x, const uint8_t *qweight, const uint16_t *scales,
                   const uint8_t *zp, int M, int N, int K, int block,
                   const int64_t *cols, int64_t ncols,
                   double *y_exact, double *abs_sum, uint16_t *y_f16, uint16_t *y_bf16)
{
    if (M < 1 || N < 1 || K < 2 || block < 2 || K % block != 0 || K % 2 != 0)
        return -1;
    int blocks = K / block;
    for (int m = 0; m < M; m++) {
        for (int64_t j = 0; j < ncols; j++) {
            int64_t n = cols[j];
            if (n < 0 || n >= N)
                return -1;
            double acc = 0.0;
            double aacc = 0.0;
            for (int k = 0; k < K; k++) {
                int b = k / block;
                double xv = mnbo_f16_to_f64(x[(size_t)m * (size_t)K + (size_t)k]);
                int q = mnbo_q_at(qweight, K, n, k);
                int z = mnbo_zp_at(zp, K, block, n, b);
                double s = mnbo_f16_to_f64(scales[(size_t)n * (size_t)blocks + (size_t)b]);
                double w = (double)(q - z) * s;
                acc += xv * w;
                aacc += fabs(xv * w);
            }
            size_t o = (size_t)m * (size_t)ncols + (size_t)j;
            uint16_t h = mnbo_f64_to_f16(acc);
            if (y_exact)
                y_exact[o] = acc;
            if (abs_sum)
                abs_sum[o] = aacc;
            if (y_f16)
                y_f16[o] = h;
            if (y_bf16)
                y_bf16[o] = mnbo_f16_to_bf16(h);
        }
    }
    return 0;
}
