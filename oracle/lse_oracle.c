/*
 * lse_oracle.c -- fp64 CPU oracle for the row-wise log-sum-exp.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It shares
 * no source, header, table or helper with the CUDA path, and the CUDA path
 * never calls it.
 *
 * What it computes (source: "Speeding up Log-Sum-Exp: Kernel Fusion at the
 * Memory Wall, Integer Arithmetic at the Compute Wall", TL;DR and Sec. 2):
 * for every row b of a [B, N] tensor,
 *
 *     out[b] = log( sum_{n<N} exp(x[b, n]) ).
 *
 * The fused method of Sec. 3.1 reaches this same value up to float rounding
 * (Sec. 4.1: it "matches torch at float precision", accuracy measured against
 * an FP64 baseline in Sec. 4).  So the oracle is the plain definition, written
 * as the max-subtract recipe of Sec. 2.1 (Fig. 1) evaluated in double:
 *
 *     m = max_n x[b, n];   s = sum_n exp(x[b, n] - m)  (index order);
 *     out[b] = m + log(s).
 *
 * Special values follow torch.logsumexp over the last dimension (the paper's
 * Table 3 covers edge cases but its cells are not reproduced on the page):
 *   any NaN in the row            -> NaN
 *   else any +inf in the row      -> +inf
 *   else every entry -inf, or N=0 -> -inf   (log of an empty / zero sum)
 * Mixed finite and -inf entries: each -inf contributes exp(-inf) = 0.
 *
 * Inputs are decoded exactly to double: f32 by widening, bf16 as the top 16
 * bits of an IEEE-754 binary32, f16 from the IEEE-754 binary16 fields.
 * Single-threaded on purpose; no blocking, fusion or reordering.
 *
 * Two consumers of the row value are defined here as well, each by its plain
 * formula in double with IEEE special-value arithmetic:
 *   token log-probability (the RLHF log-prob step of Sec. 5.1 / Fig. 6):
 *       logprob[b] = x[b, target[b]] - lse[b]   (NaN if target[b] not in [0, N))
 *   gradient of the row value (backward support, Table 3):
 *       dx[b, n] = grad[b] * exp(x[b, n] - lse[b])
 * and the same value over a non-last dimension (probabilistic-circuit sum
 * layers, Sec. 5.2) with its gradient:
 *       out[a, c] = log sum_r exp(x[a * stride_a + r * stride_r + c])
 *       dx[a, r, c] = grad[a, c] * exp(x[a * stride_a + r * stride_r + c] - lse[a, c])
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* IEEE-754 binary32 element -> double (exact widening). */
static double decode_f32(const unsigned char *p)
{
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

/* bfloat16 element: the upper half of a binary32 with the lower half zero. */
static double decode_bf16(const unsigned char *p)
{
    uint16_t h;
    uint32_t bits;
    float f;
    memcpy(&h, p, sizeof h);
    bits = (uint32_t)h << 16;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* IEEE-754 binary16 element: sign, 5-bit biased exponent (bias 15), 10-bit
 * fraction.  Normal: (1024 + frac) * 2^(e - 25); subnormal: frac * 2^-24. */
static double decode_f16(const unsigned char *p)
{
    uint16_t h;
    unsigned sign, e, frac;
    double mag;
    memcpy(&h, p, sizeof h);
    sign = (unsigned)(h >> 15) & 1u;
    e = (unsigned)(h >> 10) & 0x1fu;
    frac = (unsigned)h & 0x3ffu;
    if (e == 0u)
        mag = ldexp((double)frac, -24);
    else if (e == 31u)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024u + frac), (int)e - 25);
    return sign ? -mag : mag;
}

static double decode(int dtype, const unsigned char *row, int64_t n)
{
    switch (dtype) {
    case ORACLE_F32:  return decode_f32(row + 4 * n);
    case ORACLE_BF16: return decode_bf16(row + 2 * n);
    default:          return decode_f16(row + 2 * n);
    }
}

static int64_t elem_size(int dtype)
{
    return dtype == ORACLE_F32 ? 4 : 2;
}

/* LSE of count elements at element indices 0, step, 2*step, ... from base:
 * max-subtract in double (Sec. 2.1), special values as above. */
static double lse_strided(int dtype, const unsigned char *base, int64_t count, int64_t step)
{
    int any_nan = 0, any_pos_inf = 0;
    double m = -INFINITY, s = 0.0;
    int64_t n;

    for (n = 0; n < count; ++n) {
        double v = decode(dtype, base, n * step);
        if (isnan(v))
            any_nan = 1;
        else if (v == INFINITY)
            any_pos_inf = 1;
        else if (v > m)
            m = v;
    }
    if (any_nan)
        return NAN;
    if (any_pos_inf)
        return INFINITY;
    if (m == -INFINITY)
        return -INFINITY;

    for (n = 0; n < count; ++n)
        s += exp(decode(dtype, base, n * step) - m);
    return m + log(s);
}

/* One contiguous row. */
static double lse_row(int dtype, const unsigned char *row, int64_t N)
{
    return lse_strided(dtype, row, N, 1);
}

/*
 * oracle_lse: out[b] = log sum_n exp(x[b, n]) for b < B, in double.
 *   x          host pointer to B rows; row b starts at element b*row_stride
 *   dtype      0 = f32, 1 = bf16, 2 = f16 (raw element bits)
 *   row_stride elements between row starts, >= N
 *   out        host pointer to B doubles
 * Returns 0, or -1 on an invalid argument (nothing written).
 */
int oracle_lse(const void *x, int dtype, int64_t B, int64_t N,
               int64_t row_stride, double *out)
{
    const unsigned char *base = (const unsigned char *)x;
    int64_t b, es;

    if (dtype < ORACLE_F32 || dtype > ORACLE_F16)
        return -1;
    if (B < 0 || N < 0 || row_stride < N)
        return -1;
    if (B > 0 && (out == NULL || (N > 0 && x == NULL)))
        return -1;
    es = elem_size(dtype);
    for (b = 0; b < B; ++b)
        out[b] = lse_row(dtype, base + b * row_stride * es, N);
    return 0;
}

/* Exact decode of n raw elements to double, for checking the decoders
 * against independent conversions. */
int oracle_decode(const void *x, int dtype, int64_t n, double *out)
{
    int64_t i;
    if (dtype < ORACLE_F32 || dtype > ORACLE_F16 || n < 0)
        return -1;
    for (i = 0; i < n; ++i)
        out[i] = decode(dtype, (const unsigned char *)x, i);
    return 0;
}

/*
 * oracle_token_logprob: logprob[b] = x[b, t] - log sum_n exp(x[b, n]) with
 * t = target[b]; NaN when t is outside [0, N).  lse (may be NULL) receives
 * the row values.  Returns 0, or -1 on an invalid argument.
 */
int oracle_token_logprob(const void *x, int dtype, int64_t B, int64_t N,
                         int64_t row_stride, const int64_t *target,
                         double *logprob, double *lse)
{
    const unsigned char *base = (const unsigned char *)x;
    int64_t b, es;

    if (dtype < ORACLE_F32 || dtype > ORACLE_F16)
        return -1;
    if (B < 0 || N < 0 || row_stride < N)
        return -1;
    if (B > 0 && (logprob == NULL || target == NULL || (N > 0 && x == NULL)))
        return -1;
    es = elem_size(dtype);
    for (b = 0; b < B; ++b) {
        const unsigned char *row = base + b * row_stride * es;
        const double v = lse_row(dtype, row, N);
        const int64_t t = target[b];
        if (lse)
            lse[b] = v;
        logprob[b] = (t >= 0 && t < N) ? decode(dtype, row, t) - v : NAN;
    }
    return 0;
}

/*
 * oracle_lse_backward: dx[b * N + n] = grad[b] * exp(x[b, n] - lse[b]) for a
 * dense [B, N] double output.  lse and grad are given per row (lse normally
 * from oracle_lse).  Returns 0, or -1 on an invalid argument.
 */
int oracle_lse_backward(const void *x, int dtype, int64_t B, int64_t N,
                        int64_t row_stride, const double *lse, const double *grad,
                        double *dx)
{
    const unsigned char *base = (const unsigned char *)x;
    int64_t b, n, es;

    if (dtype < ORACLE_F32 || dtype > ORACLE_F16)
        return -1;
    if (B < 0 || N < 0 || row_stride < N)
        return -1;
    if (B > 0 && N > 0 && (x == NULL || lse == NULL || grad == NULL || dx == NULL))
        return -1;
    es = elem_size(dtype);
    for (b = 0; b < B; ++b) {
        const unsigned char *row = base + b * row_stride * es;
        for (n = 0; n < N; ++n)
            dx[b * N + n] = grad[b] * exp(decode(dtype, row, n) - lse[b]);
    }
    return 0;
}

/*
 * oracle_lse_strided: out[a * C + c] = log sum_{r<R} exp(x[a*stride_a + r*stride_r + c])
 * for a < A, c < C (element strides).  R = 0 gives -inf.  Returns 0, or -1 on
 * an invalid argument.
 */
int oracle_lse_strided(const void *x, int dtype, int64_t A, int64_t R, int64_t C,
                       int64_t stride_a, int64_t stride_r, double *out)
{
    const unsigned char *base = (const unsigned char *)x;
    int64_t a, c, es;

    if (dtype < ORACLE_F32 || dtype > ORACLE_F16)
        return -1;
    if (A < 0 || R < 0 || C < 0 || stride_a < 0 || stride_r < 0)
        return -1;
    if (A > 0 && C > 0 && (out == NULL || (R > 0 && x == NULL)))
        return -1;
    es = elem_size(dtype);
    for (a = 0; a < A; ++a)
        for (c = 0; c < C; ++c)
            out[a * C + c] = lse_strided(dtype, base + (a * stride_a + c) * es, R, stride_r);
    return 0;
}

/*
 * oracle_lse_backward_strided: gradient of oracle_lse_strided's value,
 *     dx[(a * R + r) * C + c] = grad[a * C + c]
 *                               * exp(x[a*stride_a + r*stride_r + c] - lse[a * C + c])
 * for a dense [A, R, C] double output; lse and grad are [A, C] (lse normally
 * from oracle_lse_strided).  Returns 0, or -1 on an invalid argument.
 */
int oracle_lse_backward_strided(const void *x, int dtype, int64_t A, int64_t R, int64_t C,
                                int64_t stride_a, int64_t stride_r, const double *lse,
                                const double *grad, double *dx)
{
    const unsigned char *base = (const unsigned char *)x;
    int64_t a, r, c, es;

    if (dtype < ORACLE_F32 || dtype > ORACLE_F16)
        return -1;
    if (A < 0 || R < 0 || C < 0 || stride_a < 0 || stride_r < 0)
        return -1;
    if (A > 0 && R > 0 && C > 0 && (x == NULL || lse == NULL || grad == NULL || dx == NULL))
        return -1;
    es = elem_size(dtype);
    for (a = 0; a < A; ++a)
        for (r = 0; r < R; ++r) {
            const unsigned char *row = base + (a * stride_a + r * stride_r) * es;
            for (c = 0; c < C; ++c)
                dx[(a * R + r) * C + c] =
                    grad[a * C + c] * exp(decode(dtype, row, c) - lse[a * C + c]);
        }
    return 0;
}
