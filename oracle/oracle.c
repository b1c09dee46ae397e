/*
 * CPU oracle for the skinny BF16 linear layer  out[M,N] = x[M,K] @ W[N,K]^T (+ bias[N]).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into a separate shared
 * object that only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark load.  The CUDA library never links, includes or calls it,
 * and it shares no header, helper or table with the CUDA sources.
 *
 * What it computes (the plain definition, written out):
 *
 *   acc[m,n] = sum_{k=0}^{K-1} f64(x[m,k]) * f64(W[n,k])        ascending k
 *   acc[m,n] += f64(bias[n])                                      if bias given
 *   out[m,n] = RNE_bf16(acc[m,n])                                 one rounding
 *
 * Source of the definition: sglang PR #30117 page, section "关键源码片段",
 * header comment of the TGV BF16 GEMM kernel (out[M,N] = x[M,K] @ weight[N,K].T
 * (+ bias[N]); bf16 in and out; fp32 accumulation inside).  The oracle widens
 * to f64 instead of f32 so that only the final rounding matters: a product of
 * two bf16 values has at most 16 significant bits and is exact in f64, so the
 * only other error is the f64 summation (~1e-16 relative).
 *
 * Readings where the page is silent (also listed in the design notes):
 *  - bias enters before the single rounding (the FP8 wrapper on the
 *    sglang PR #28333 page adds bias after the GEMM in the output dtype;
 *    the difference is one extra rounding, inside the test tolerance);
 *  - rounding is IEEE round-to-nearest, ties to even;
 *  - the router variant of the vLLM PR #42562 page writes fp32 logits
 *    (LLBf16SplitK, out_dtype=Float32): oracle_linear_f32 rounds the same
 *    f64 sum once to binary32 instead of bf16.
 *
 * The narrowing conversion (rne_narrow) is written from the IEEE 754 binary
 * interchange format definition (sign, biased exponent, trailing significand)
 * on the bit pattern of the f64 value; it calls no library cast.
 */
#include <stdint.h>
#include <string.h>

/* bf16 is the upper 16 bits of an IEEE binary32; widening is exact. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round an f64 value to the nearest value of a narrower IEEE binary format with
 * `ebits` exponent bits and `mbits` trailing-significand bits, ties to even.
 * Returns the bit pattern of the narrow format (sign in bit ebits+mbits).
 * NaN maps to the canonical quiet NaN; overflow rounds to infinity.
 */
static uint32_t rne_narrow(double v, int ebits, int mbits)
{
    uint64_t b;
    memcpy(&b, &v, sizeof b);
    const uint32_t sign = (uint32_t)(b >> 63) << (ebits + mbits);
    const int e = (int)((b >> 52) & 0x7FF);
    const uint64_t f = b & ((1ULL << 52) - 1);
    const uint32_t exp_ones = ((1u << ebits) - 1u) << mbits;

    if (e == 0x7FF)                         /* NaN or infinity */
        return f ? (exp_ones | (1u << (mbits - 1))) : (sign | exp_ones);
    if (e == 0)                             /* f64 zero or f64 subnormal (< 2^-1022) */
        return sign;                        /* far below half the narrow format's smallest subnormal */

    const int bias = (1 << (ebits - 1)) - 1;
    const int E = e - 1023;                 /* v = S * 2^(E-52), S the 53-bit significand */
    const int emin = 1 - bias;              /* exponent of the smallest normal */
    if (E > bias)                           /* at or above 2^(bias+1): infinity */
        return sign | exp_ones;

    const uint64_t S = (1ULL << 52) | f;
    const int q = (E >= emin ? E : emin) - mbits;   /* exponent of one unit in the last place */
    const int shift = q - (E - 52);                  /* low bits of S that fall below that unit */
    if (shift > 54)                         /* |v| < 2^(q-2): rounds to zero */
        return sign;

    uint64_t kept = S >> shift;
    const uint64_t rem = S & ((1ULL << shift) - 1);
    const uint64_t half = 1ULL << (shift - 1);
    if (rem > half || (rem == half && (kept & 1)))
        kept++;

    uint32_t bits;
    if (E >= emin)                          /* kept in [2^mbits, 2^(mbits+1)]; a carry bumps the exponent */
        bits = ((uint32_t)(E + bias - 1) << mbits) + (uint32_t)kept;
    else                                    /* subnormal: kept <= 2^mbits (== 2^mbits is the smallest normal) */
        bits = (uint32_t)kept;
    return sign | bits;
}

uint16_t oracle_rne_bf16(double v) { return (uint16_t)rne_narrow(v, 8, 7); }
uint32_t oracle_rne_f32(double v) { return rne_narrow(v, 8, 23); }
double oracle_bf16_to_f64(uint16_t h) { return bf16_to_f64(h); }

/* One output element, unrounded: ascending-k f64 sum, then bias. */
static double dot_row(const uint16_t *xrow, const uint16_t *wrow, const uint16_t *bias,
                      int64_t n, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
        acc += bf16_to_f64(xrow[k]) * bf16_to_f64(wrow[k]);
    if (bias)
        acc += bf16_to_f64(bias[n]);
    return acc;
}

/* acc[M*N] (row-major), unrounded f64.  bias may be NULL. */
void oracle_linear_f64(const uint16_t *x, const uint16_t *W, const uint16_t *bias,
                       int64_t M, int64_t N, int64_t K, double *acc)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            acc[m * N + n] = dot_row(x + m * K, W + n * K, bias, n, K);
}

/* out[M*N] bf16 bits (row-major): the defined result. */
void oracle_linear_bf16(const uint16_t *x, const uint16_t *W, const uint16_t *bias,
                        int64_t M, int64_t N, int64_t K, uint16_t *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] = oracle_rne_bf16(dot_row(x + m * K, W + n * K, bias, n, K));
}

/* out[M*N] binary32 bits: the fp32-logits variant (one rounding to binary32). */
void oracle_linear_f32(const uint16_t *x, const uint16_t *W, const uint16_t *bias,
                       int64_t M, int64_t N, int64_t K, uint32_t *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] = oracle_rne_f32(dot_row(x + m * K, W + n * K, bias, n, K));
}

/*
 * Selected output rows only: out[r*N + n] for m = rows[r].  Used to check
 * sampled rows of shapes too large to evaluate in full on the CPU.
 */
void oracle_linear_rows_bf16(const uint16_t *x, const uint16_t *W, const uint16_t *bias,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t *rows, int64_t nrows, uint16_t *out)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = rows[r];
        for (int64_t n = 0; n < N; ++n)
            out[r * N + n] = oracle_rne_bf16(dot_row(x + m * K, W + n * K, bias, n, K));
    }
}

/* Unrounded selected rows (for the per-row cosine check at full size). */
void oracle_linear_rows_f64(const uint16_t *x, const uint16_t *W, const uint16_t *bias,
                            int64_t M, int64_t N, int64_t K,
                            const int64_t *rows, int64_t nrows, double *acc)
{
    (void)M;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = rows[r];
        for (int64_t n = 0; n < N; ++n)
            acc[r * N + n] = dot_row(x + m * K, W + n * K, bias, n, K);
    }
}

/*
 * ---------------------------------------------------------------------------
 * Per-tensor FP8 linear (the scope's FP8 row).
 *
 * Source: the sglang PR #28333 page, section "关键源码片段":
 *  - apply_fp8_linear_bmm_flashinfer (fp8_utils.py) quantises the input with
 *    a given per-tensor scale (static_quant_fp8), multiplies the e4m3 operands
 *    with per-tensor scales x_scale and weight_scale (bmm_fp8, output in the
 *    input dtype), then adds bias;
 *  - the static quantisation kernel (fp8_kernel.py, _static_quant_fp8) forms
 *    y_s_inv = 1 / y_s and stores clamp(y * y_s_inv, fp8_min, fp8_max)
 *    converted to the e4m3 type, with y and y_s read as fp32.
 * Readings (also in the design notes): the product and the reciprocal round
 * to binary32 as in the kernel; the conversion to e4m3 is round-to-nearest
 * even (the clamp keeps it in range); the scaled sum and the bias meet before
 * one rounding to bf16, as for the bf16 linear (the page adds bias after a
 * bf16 result: one more rounding, inside the tolerance).
 *
 * e4m3 (the "fn" variant: no infinities), code c:
 *   s = c >> 7, E = (c >> 3) & 15, m = c & 7
 *   E == 0                 : (-1)^s * (m / 8) * 2^-6        (subnormal)
 *   E == 15 and m == 7     : NaN
 *   otherwise              : (-1)^s * (1 + m / 8) * 2^(E - 7)
 * Largest finite value 448 = 1.75 * 2^8.
 * ---------------------------------------------------------------------------
 */
static double e4m3_to_f64(uint8_t c)
{
    const int s = c >> 7, E = (c >> 3) & 15, m = c & 7;
    double v;
    if (E == 15 && m == 7) {
        uint64_t qnan = 0x7FF8000000000000ULL;
        memcpy(&v, &qnan, sizeof v);
        return v;
    }
    if (E == 0)
        v = (double)m / 8.0 * 0.015625;                  /* 2^-6 */
    else {
        v = 1.0 + (double)m / 8.0;
        for (int i = 7; i < E; ++i) v *= 2.0;             /* scale by 2^(E-7) exactly */
        for (int i = E; i < 7; ++i) v *= 0.5;
    }
    return s ? -v : v;
}

/*
 * Round a finite value with |v| <= 448 to the nearest e4m3 code, ties to an
 * even significand; 3 trailing significand bits, exponent bias 7, smallest
 * normal 2^-6, subnormal unit 2^-9.  Written on the f64 bit pattern like
 * rne_narrow, with e4m3's own top binade (exponent field 15 is finite).
 */
static uint8_t rne_e4m3(double v)
{
    uint64_t b;
    memcpy(&b, &v, sizeof b);
    const uint8_t sign = (uint8_t)((b >> 63) << 7);
    const int e = (int)((b >> 52) & 0x7FF);
    if (e == 0) return sign;                              /* zero (or far below 2^-10) */
    const uint64_t S = (1ULL << 52) | (b & ((1ULL << 52) - 1));
    const int E = e - 1023;
    const int emin = -6, mbits = 3;
    const int q = (E >= emin ? E : emin) - mbits;         /* exponent of one unit in the last place */
    const int shift = q - (E - 52);
    if (shift > 54) return sign;                          /* below a quarter of the smallest subnormal */
    uint64_t kept = S >> shift;
    const uint64_t rem = S & ((1ULL << shift) - 1);
    const uint64_t half = 1ULL << (shift - 1);
    if (rem > half || (rem == half && (kept & 1))) kept++;
    if (E >= emin)                                        /* kept in [8, 16]; a carry bumps the exponent */
        return (uint8_t)(sign | (((E + 7 - 1) << mbits) + (int)kept));
    return (uint8_t)(sign | (int)kept);                   /* subnormal (kept == 8 is the smallest normal) */
}

double oracle_e4m3_to_f64(uint8_t c) { return e4m3_to_f64(c); }
uint8_t oracle_rne_e4m3(double v) { return rne_e4m3(v); }

/* Static per-tensor quantisation of n bf16 values with the given scale. */
void oracle_quant_fp8(const uint16_t *x, int64_t n, float scale, uint8_t *q)
{
    const float inv = 1.0f / scale;                       /* binary32 reciprocal */
    for (int64_t i = 0; i < n; ++i) {
        float y = (float)bf16_to_f64(x[i]) * inv;          /* binary32 product */
        if (y > 448.0f) y = 448.0f;
        if (y < -448.0f) y = -448.0f;
        q[i] = rne_e4m3((double)y);
    }
}

/*
 * One FP8 output element, unrounded: the exact f64 sum of the e4m3 products
 * (each product has at most 8 significant bits between 2^-18 and 2^18, so
 * sums of up to 2^13 of them are exact in f64), times the two scales, plus
 * bias.
 */
static double dot_row_fp8(const uint8_t *xrow, const uint8_t *wrow, double sxw, const uint16_t *bias,
                          int64_t n, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
        acc += e4m3_to_f64(xrow[k]) * e4m3_to_f64(wrow[k]);
    acc *= sxw;
    if (bias)
        acc += bf16_to_f64(bias[n]);
    return acc;
}

void oracle_linear_fp8_f64(const uint8_t *xq, const uint8_t *wq, float sx, float sw, const uint16_t *bias,
                           int64_t M, int64_t N, int64_t K, double *acc)
{
    const double sxw = (double)sx * (double)sw;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            acc[m * N + n] = dot_row_fp8(xq + m * K, wq + n * K, sxw, bias, n, K);
}

void oracle_linear_fp8(const uint8_t *xq, const uint8_t *wq, float sx, float sw, const uint16_t *bias,
                       int64_t M, int64_t N, int64_t K, uint16_t *out)
{
    const double sxw = (double)sx * (double)sw;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] = oracle_rne_bf16(dot_row_fp8(xq + m * K, wq + n * K, sxw, bias, n, K));
}

/*
 * ---------------------------------------------------------------------------
 * MXFP8 linear (the scope's MXFP8 row).
 *
 * Source: the sglang PR #34042 page ("执行摘要", "实现拆解" items 2-3): a dense
 * MXFP8 GEMM on SM10x whose weights carry block scales (weight_scale_inv, fed
 * to the kernel in a swizzled layout), with activations quantised the same
 * way.  The page does not spell the format out.  Reading (also in the design
 * notes): the OCP microscaling format MXFP8 -- each run of 32 consecutive
 * elements along K shares one E8M0 scale byte e (value 2^(e - 127), e = 255
 * is NaN and never produced), the elements are e4m3 codes as above; a block's
 * value is scale x element.  Scales are stored plainly, row-major [rows][K/32]
 * (the swizzle is a layout for the hardware, not arithmetic).
 *
 * Quantisation of one block of bf16 values v (the OCP conversion):
 *   s = floor(log2(max |v|)) - 8   (8: the exponent of e4m3's largest binade),
 *   clamped below at -127 (an all-zero block gets s = -127), e = s + 127,
 *   code_i = e4m3 of v_i * 2^-s, rounded to nearest even, values past 448
 *   saturating to +-448.
 * The linear: out[m,n] = RNE_bf16( sum_k e4m3(xq[m,k]) e4m3(wq[n,k])
 *   * 2^(sx[m][k/32]-127) * 2^(sw[n][k/32]-127) + bias[n] ), every term exact
 *   in f64 and summed in ascending k.
 * ---------------------------------------------------------------------------
 */
static double pow2_exact(int e)
{
    double v = 1.0;
    for (int i = 0; i < e; ++i) v *= 2.0;
    for (int i = e; i < 0; ++i) v *= 0.5;
    return v;
}

double oracle_e8m0_to_f64(uint8_t e)
{
    if (e == 255) {
        uint64_t qnan = 0x7FF8000000000000ULL;
        double v;
        memcpy(&v, &qnan, sizeof v);
        return v;
    }
    return pow2_exact((int)e - 127);
}

/* x[rows][K] bf16, K % 32 == 0 -> q[rows][K] e4m3 codes, scales[rows][K/32] E8M0. */
void oracle_quant_mxfp8(const uint16_t *x, int64_t rows, int64_t K, uint8_t *q, uint8_t *scales)
{
    const int64_t nb = K / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t *v = x + r * K + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                const double f = bf16_to_f64(v[i]);
                const double a = f < 0.0 ? -f : f;
                if (a > amax) amax = a;
            }
            int s = -127;
            if (amax > 0.0) {
                uint64_t bits;
                memcpy(&bits, &amax, sizeof bits);
                const int lg = (int)((bits >> 52) & 0x7FF) - 1023; /* floor(log2(amax)): amax is an f64 normal */
                s = lg - 8;
                if (s < -127) s = -127;
                if (s > 127) s = 127;
            }
            scales[r * nb + b] = (uint8_t)(s + 127);
            const double inv = pow2_exact(-s);
            for (int i = 0; i < 32; ++i) {
                double y = bf16_to_f64(v[i]) * inv;             /* exact: a power of two */
                if (y > 448.0) y = 448.0;
                if (y < -448.0) y = -448.0;
                q[r * K + b * 32 + i] = rne_e4m3(y);
            }
        }
}

static double dot_row_mxfp8(const uint8_t *xr, const uint8_t *xs, const uint8_t *wr, const uint8_t *ws,
                            const uint16_t *bias, int64_t n, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
        acc += e4m3_to_f64(xr[k]) * e4m3_to_f64(wr[k]) * pow2_exact((int)xs[k / 32] - 127) *
               pow2_exact((int)ws[k / 32] - 127);
    if (bias)
        acc += bf16_to_f64(bias[n]);
    return acc;
}

void oracle_linear_mxfp8_f64(const uint8_t *xq, const uint8_t *sx, const uint8_t *wq, const uint8_t *sw,
                             const uint16_t *bias, int64_t M, int64_t N, int64_t K, double *acc)
{
    const int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            acc[m * N + n] = dot_row_mxfp8(xq + m * K, sx + m * nb, wq + n * K, sw + n * nb, bias, n, K);
}

void oracle_linear_mxfp8(const uint8_t *xq, const uint8_t *sx, const uint8_t *wq, const uint8_t *sw,
                         const uint16_t *bias, int64_t M, int64_t N, int64_t K, uint16_t *out)
{
    const int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] =
                oracle_rne_bf16(dot_row_mxfp8(xq + m * K, sx + m * nb, wq + n * K, sw + n * nb, bias, n, K));
}

/* Selected output rows of the MXFP8 linear (bf16 bits), for full-size checks on samples. */
void oracle_linear_rows_mxfp8(const uint8_t *xq, const uint8_t *sx, const uint8_t *wq, const uint8_t *sw,
                              const uint16_t *bias, int64_t M, int64_t N, int64_t K, const int64_t *rows,
                              int64_t nrows, uint16_t *out)
{
    (void)M;
    const int64_t nb = K / 32;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = rows[r];
        for (int64_t n = 0; n < N; ++n)
            out[r * N + n] =
                oracle_rne_bf16(dot_row_mxfp8(xq + m * K, sx + m * nb, wq + n * K, sw + n * nb, bias, n, K));
    }
}
