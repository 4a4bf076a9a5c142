/*
 * oracle.c -- plain, slow, fp64 CPU restatement of the row-wise RMSNorm forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA path is
 * checked against.  Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline / reference arm may load it.  The product path
 * (the CUDA library under rmsnorm_fwd_gb300/) never calls, links or includes
 * anything from here, and this file includes nothing from there.
 *
 * What it computes (one row i of a row-major [rows, hidden] tensor):
 *
 *   "Build a GPU compiler from scratch: from PyTorch to CUDA via multi-level
 *    IR (Emmy)", introduction (the RMSNorm running example) and section
 *    "Tensor IR" (the arithmetic steps: square, sum, divide by the count,
 *    add epsilon, rsqrt, two multiplies):
 *
 *        S   = sum_j x[i,j]^2
 *        r   = 1 / sqrt(S / hidden + eps)
 *        y   = x[i,j] * r * w[j]
 *
 *   "CuTeDSL at Perplexity", section "QK Norm": the same statistic taken as
 *   rsqrt(sum / head_dim + EPS), each element scaled by that factor and by
 *   its weight plus WEIGHT_BIAS, the result cast back to the input's element
 *   type.
 *
 *   Same page, section "Blackwell support" (MXFP8 / MXFP4 / NVFP4, absolute
 *   maxima over blocks of 16 or 32 elements): the normalised row may instead
 *   leave as MXFP8 (E4M3 elements, one power-of-two E8M0 scale per 32
 *   consecutive elements), MXFP4 (E2M1 elements, the same scales) or NVFP4
 *   (E2M1 elements, one E4M3 scale per 16 elements times a per-tensor fp32
 *   scale).  The pages name the formats but do not define them; the
 *   definitions used are the OCP Microscaling (MX) v1.0 specification's for
 *   the MX formats and NVIDIA's published description of NVFP4 (see the
 *   sections below).
 *
 * Every value is widened exactly to IEEE binary64 and every operation runs in
 * binary64, left to right, with no blocking, fusion or reordering.  The final
 * rounding to a 16-bit format is done directly from binary64 with
 * round-to-nearest-even (no intermediate binary32 step, so no double
 * rounding).
 *
 * Formats: 0 = IEEE binary32, 1 = bfloat16, 2 = IEEE binary16.  16-bit
 * values travel as raw uint16 bit patterns.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

/* ---- exact widening of one stored element to binary64 ------------------ */

static double widen_f32(uint32_t bits)
{
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f; /* every binary32 value is exactly a binary64 value */
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double widen_bf16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xFF;
    int frac = bits & 0x7F;
    double mag;
    if (expo == 0xFF)
        mag = frac ? NAN : INFINITY;
    else if (expo == 0)
        mag = ldexp((double)frac, -126 - 7); /* subnormal: frac * 2^-133 */
    else
        mag = ldexp((double)(128 + frac), expo - 127 - 7);
    return sign ? -mag : mag;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double widen_f16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1F;
    int frac = bits & 0x3FF;
    double mag;
    if (expo == 0x1F)
        mag = frac ? NAN : INFINITY;
    else if (expo == 0)
        mag = ldexp((double)frac, -14 - 10); /* subnormal: frac * 2^-24 */
    else
        mag = ldexp((double)(1024 + frac), expo - 15 - 10);
    return sign ? -mag : mag;
}

double oracle_widen(const void *base, int64_t index, int fmt)
{
    if (fmt == ORACLE_F32) {
        uint32_t b;
        memcpy(&b, (const char *)base + 4 * index, 4);
        return widen_f32(b);
    }
    uint16_t h;
    memcpy(&h, (const char *)base + 2 * index, 2);
    return fmt == ORACLE_BF16 ? widen_bf16(h) : widen_f16(h);
}

/* ---- round binary64 to a narrow binary format, nearest-even ------------ */

/*
 * A binary format with p significand bits (counting the hidden bit), minimum
 * normal exponent emin and maximum exponent emax.  The representable numbers
 * in the binade [2^e, 2^(e+1)) are integer multiples of 2^(e-p+1); below 2^emin
 * they are multiples of 2^(emin-p+1).  Rounding a = |v| therefore means: take
 * the spacing q of the binade a falls in, round a/q to the nearest integer
 * with ties to even (rint() under the default rounding mode does exactly
 * that, and a/q is exact because q is a power of two), and multiply back.
 * Results above the largest finite value become infinity.
 */
static double round_to_format(double v, int p, int emin, int emax)
{
    if (isnan(v) || isinf(v) || v == 0.0)
        return v;
    double a = fabs(v);
    int k;
    frexp(a, &k);          /* a = m * 2^k with m in [0.5, 1): a in [2^(k-1), 2^k) */
    int e = k - 1;
    if (e < emin)
        e = emin;
    int qexp = e - (p - 1);
    double n = rint(ldexp(a, -qexp));
    double r = ldexp(n, qexp);
    double maxfinite = ldexp((double)((1 << p) - 1), emax - p + 1);
    if (r > maxfinite)
        r = INFINITY;
    return v < 0 ? -r : r;
}

/* Encode a value that is already exactly representable in the format. */
static uint16_t encode_narrow(double v, int p, int emin, int ebits)
{
    uint16_t sign = signbit(v) ? (uint16_t)(1u << 15) : 0;
    int fbits = p - 1;
    uint16_t expmask = (uint16_t)((1u << ebits) - 1);
    if (isnan(v))
        return (uint16_t)(sign | (expmask << fbits) | (1u << (fbits - 1)));
    if (isinf(v))
        return (uint16_t)(sign | (expmask << fbits));
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int bias = 1 - emin;
    if (a < ldexp(1.0, emin)) { /* subnormal: a = frac * 2^(emin - fbits) */
        uint16_t frac = (uint16_t)ldexp(a, -(emin - fbits));
        return (uint16_t)(sign | frac);
    }
    int k;
    frexp(a, &k);
    int e = k - 1;
    uint16_t frac = (uint16_t)(ldexp(a, -(e - fbits)) - ldexp(1.0, fbits));
    return (uint16_t)(sign | ((uint16_t)(e + bias) << fbits) | frac);
}

double oracle_round_value(double v, int fmt)
{
    switch (fmt) {
    case ORACLE_F32:
        return round_to_format(v, 24, -126, 127);
    case ORACLE_BF16:
        return round_to_format(v, 8, -126, 127);
    default:
        return round_to_format(v, 11, -14, 15);
    }
}

void oracle_store(double v, void *base, int64_t index, int fmt)
{
    double r = oracle_round_value(v, fmt);
    if (fmt == ORACLE_F32) {
        float f = (float)r; /* exact: r is already a binary32 value */
        memcpy((char *)base + 4 * index, &f, 4);
        return;
    }
    uint16_t h = fmt == ORACLE_BF16 ? encode_narrow(r, 8, -126, 8)
                                    : encode_narrow(r, 11, -14, 5);
    memcpy((char *)base + 2 * index, &h, 2);
}

/* ---- the method --------------------------------------------------------- */

/*
 * One row: square every element, sum them, divide the sum by the row length,
 * add epsilon, take the reciprocal square root, then multiply each element
 * by that factor and by its weight.  The statistic S is a row-local value
 * and is never stored.
 */
static double row_factor(const void *x, int64_t row, int64_t hidden, double eps, int fmt)
{
    double S = 0.0;
    for (int64_t j = 0; j < hidden; ++j) {
        double xv = oracle_widen(x, row * hidden + j, fmt);
        S += xv * xv;
    }
    double mean = S / (double)hidden;
    return 1.0 / sqrt(mean + eps);
}

int oracle_rmsnorm_f64(const void *x, const void *w, double *y, int64_t rows,
                       int64_t hidden, float eps, int fmt)
{
    if (rows < 0 || hidden <= 0 || fmt < 0 || fmt > 2)
        return -1;
    double e = (double)eps; /* both sides see the same binary32 epsilon */
    for (int64_t i = 0; i < rows; ++i) {
        double r = row_factor(x, i, hidden, e, fmt);
        for (int64_t j = 0; j < hidden; ++j) {
            double xv = oracle_widen(x, i * hidden + j, fmt);
            double wv = oracle_widen(w, j, fmt);
            y[i * hidden + j] = xv * r * wv;
        }
    }
    return 0;
}

int oracle_rmsnorm(const void *x, const void *w, void *y, int64_t rows,
                   int64_t hidden, float eps, int fmt)
{
    if (rows < 0 || hidden <= 0 || fmt < 0 || fmt > 2)
        return -1;
    double e = (double)eps;
    for (int64_t i = 0; i < rows; ++i) {
        double r = row_factor(x, i, hidden, e, fmt);
        for (int64_t j = 0; j < hidden; ++j) {
            double xv = oracle_widen(x, i * hidden + j, fmt);
            double wv = oracle_widen(w, j, fmt);
            oracle_store(xv * r * wv, y, i * hidden + j, fmt);
        }
    }
    return 0;
}

int oracle_round_array(const double *v, void *out, int64_t n, int fmt)
{
    if (n < 0 || fmt < 0 || fmt > 2)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        oracle_store(v[i], out, i, fmt);
    return 0;
}

int oracle_widen_array(const void *in, double *out, int64_t n, int fmt)
{
    if (n < 0 || fmt < 0 || fmt > 2)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_widen(in, i, fmt);
    return 0;
}

/* ---- per-head QK norm ----------------------------------------------------- */

/*
 * "CuTeDSL at Perplexity", section "QK Norm": every attention head of q
 * (q_heads per token) and of k (k_heads per token) is normalised on its own,
 * over head_dim elements, with the q or the k weight plus WEIGHT_BIAS, and
 * the result replaces the head in place:
 *
 *     S = sum_d x[d]^2,  r = 1 / sqrt(S / head_dim + eps),
 *     x[d] <- x[d] * r * (w[d] + weight_bias)
 *
 * Token t's heads start at element t * token_stride of q (resp. k); heads are
 * contiguous within a token.  In binary64, rounded back nearest-even.
 */
static void norm_heads(void *base, const void *w, int64_t tokens, int64_t heads,
                       int64_t head_dim, int64_t stride, double bias, double eps, int fmt)
{
    for (int64_t t = 0; t < tokens; ++t) {
        for (int64_t h = 0; h < heads; ++h) {
            const int64_t off = t * stride + h * head_dim;
            double S = 0.0;
            for (int64_t d = 0; d < head_dim; ++d) {
                double xv = oracle_widen(base, off + d, fmt);
                S += xv * xv;
            }
            double r = 1.0 / sqrt(S / (double)head_dim + eps);
            for (int64_t d = 0; d < head_dim; ++d) {
                double xv = oracle_widen(base, off + d, fmt);
                double wv = oracle_widen(w, d, fmt) + bias;
                oracle_store(xv * r * wv, base, off + d, fmt);
            }
        }
    }
}

int oracle_qk_norm(void *q, void *k, const void *q_weight, const void *k_weight, int64_t tokens,
                   int64_t q_heads, int64_t k_heads, int64_t head_dim, int64_t q_token_stride,
                   int64_t k_token_stride, float weight_bias, float eps, int fmt)
{
    if (tokens < 0 || q_heads < 0 || k_heads < 0 || head_dim <= 0 || fmt < 0 || fmt > 2)
        return -1;
    if (q_token_stride < q_heads * head_dim || k_token_stride < k_heads * head_dim)
        return -1;
    norm_heads(q, q_weight, tokens, q_heads, head_dim, q_token_stride, (double)weight_bias,
               (double)eps, fmt);
    norm_heads(k, k_weight, tokens, k_heads, head_dim, k_token_stride, (double)weight_bias,
               (double)eps, fmt);
    return 0;
}

/* ---- weight bias ---------------------------------------------------------- */

/*
 * The row normalisation with the weight offset of "CuTeDSL at Perplexity",
 * section "QK Norm" (w + WEIGHT_BIAS) applied to whole rows:
 *     y[i,j] = x[i,j] * r_i * (w[j] + weight_bias)
 * in binary64, unrounded.
 */
int oracle_rmsnorm_bias_f64(const void *x, const void *w, double *y, int64_t rows,
                            int64_t hidden, float weight_bias, float eps, int fmt)
{
    if (rows < 0 || hidden <= 0 || fmt < 0 || fmt > 2)
        return -1;
    double e = (double)eps;
    double b = (double)weight_bias;
    for (int64_t i = 0; i < rows; ++i) {
        double r = row_factor(x, i, hidden, e, fmt);
        for (int64_t j = 0; j < hidden; ++j) {
            double xv = oracle_widen(x, i * hidden + j, fmt);
            double wv = oracle_widen(w, j, fmt) + b;
            y[i * hidden + j] = xv * r * wv;
        }
    }
    return 0;
}

/* The same, rounded nearest-even to the element format. */
int oracle_rmsnorm_bias(const void *x, const void *w, void *y, int64_t rows, int64_t hidden,
                        float weight_bias, float eps, int fmt)
{
    if (rows < 0 || hidden <= 0 || fmt < 0 || fmt > 2)
        return -1;
    double e = (double)eps;
    double b = (double)weight_bias;
    for (int64_t i = 0; i < rows; ++i) {
        double r = row_factor(x, i, hidden, e, fmt);
        for (int64_t j = 0; j < hidden; ++j) {
            double xv = oracle_widen(x, i * hidden + j, fmt);
            double wv = oracle_widen(w, j, fmt) + b;
            oracle_store(xv * r * wv, y, i * hidden + j, fmt);
        }
    }
    return 0;
}

/* ---- MXFP8: E4M3 elements, one E8M0 scale per 32 elements ----------------- */

/*
 * E4M3 (the OCP 8-bit floating-point format "E4M3"): 1 sign bit, 4 exponent
 * bits with bias 7, 3 fraction bits; no infinities; exponent field 15 with
 * fraction 7 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448;
 * exponent field 0 holds the subnormals f * 2^-9.
 */
double oracle_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int frac = code & 0x7;
    double mag;
    if (expo == 0xF && frac == 0x7)
        mag = NAN;
    else if (expo == 0)
        mag = ldexp((double)frac, -9);
    else
        mag = ldexp((double)(8 + frac), expo - 7 - 3);
    return sign ? -mag : mag;
}

/*
 * Round to E4M3, nearest with ties to even, saturating: a magnitude that
 * rounds above 448 becomes 448 (the format has no infinity; the MX
 * specification leaves overflow to the implementation, and clamping is the
 * plainest choice).  NaN becomes the NaN code with the input's sign.
 */
uint8_t oracle_e4m3_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    double a = fabs(v);
    /* p = 4 significand bits, minimum normal exponent -6; the generic
     * rounding's overflow to infinity is replaced by the clamp. */
    double r = isinf(a) ? 448.0 : round_to_format(a, 4, -6, 8);
    if (isinf(r) || r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -6))
        return (uint8_t)(sign | (uint8_t)ldexp(r, 9)); /* subnormal: r = f * 2^-9 */
    int k;
    frexp(r, &k);
    int e = k - 1; /* r in [2^e, 2^(e+1)) */
    uint8_t frac = (uint8_t)(ldexp(r, 3 - e) - 8.0);
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | frac);
}

/*
 * One MX block (OCP Microscaling v1.0, conversion of a vector of scalars to
 * an MX block): the shared exponent is floor(log2(max |v|)) minus the
 * largest exponent of the element format (8 for E4M3), clamped to the E8M0
 * range [-127, 127]; the scale is X = 2^shared; every element is v / X
 * rounded to E4M3 as above.  E8M0 stores shared + 127; 0xFF (NaN) when the
 * block holds a NaN or an infinity.  An all-zero block takes the smallest
 * scale, 2^-127 (code 0).
 */
static void mx_block(const double *v, int n, uint8_t *codes, uint8_t *scale)
{
    double amax = 0.0;
    int special = 0;
    for (int i = 0; i < n; ++i) {
        if (isnan(v[i]) || isinf(v[i]))
            special = 1;
        else if (fabs(v[i]) > amax)
            amax = fabs(v[i]);
    }
    int shared;
    if (amax == 0.0) {
        shared = -127;
    } else {
        int k;
        frexp(amax, &k); /* amax in [2^(k-1), 2^k): floor(log2 amax) = k - 1 */
        shared = (k - 1) - 8;
        if (shared < -127)
            shared = -127;
        if (shared > 127)
            shared = 127;
    }
    *scale = special ? 0xFF : (uint8_t)(shared + 127);
    for (int i = 0; i < n; ++i)
        codes[i] = oracle_e4m3_encode(ldexp(v[i], -shared)); /* v / X, exact */
}

int oracle_mxfp8_quantize(const double *v, int64_t rows, int64_t cols, uint8_t *codes,
                          uint8_t *scales)
{
    if (rows < 0 || cols <= 0 || cols % 32 != 0)
        return -1;
    const int64_t nb = cols / 32;
    for (int64_t i = 0; i < rows; ++i)
        for (int64_t b = 0; b < nb; ++b)
            mx_block(v + i * cols + b * 32, 32, codes + i * cols + b * 32, scales + i * nb + b);
    return 0;
}

/* ---- MXFP4 and NVFP4: E2M1 elements -------------------------------------- */

/*
 * E2M1 (the OCP 4-bit floating-point element format): 1 sign bit, 2 exponent
 * bits with bias 1, 1 fraction bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no
 * infinity or NaN.  Codes are 4-bit values 0..15 (sign in bit 3).
 */
double oracle_e2m1_value(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int expo = (code >> 1) & 0x3;
    int frac = code & 0x1;
    double mag = expo == 0 ? 0.5 * frac : ldexp(1.0 + 0.5 * frac, expo - 1);
    return sign ? -mag : mag;
}

/* Round to E2M1, nearest with ties to even, saturating at +-6 (the largest
 * magnitude).  The format has no NaN: a NaN input gives the code of +-6
 * (only inside a block whose scale is NaN, where element codes carry no
 * value). */
uint8_t oracle_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    if (isnan(v))
        return (uint8_t)(sign | 0x7);
    double a = fabs(v);
    /* p = 2 significand bits, minimum normal exponent 0, largest exponent 2 */
    double r = isinf(a) ? 6.0 : round_to_format(a, 2, 0, 2);
    if (isinf(r) || r > 6.0)
        r = 6.0;
    if (r == 0.0)
        return sign;
    if (r < 1.0)
        return (uint8_t)(sign | 0x1); /* the subnormal 0.5 */
    int k;
    frexp(r, &k);
    int e = k - 1; /* r in [2^e, 2^(e+1)), e in 0..2 */
    uint8_t frac = (uint8_t)(ldexp(r, 1 - e) - 2.0);
    return (uint8_t)(sign | (uint8_t)((e + 1) << 1) | frac);
}

/* Element j of a row goes to byte j / 2, low nibble for even j. */
static void put_nibble(uint8_t *row, int64_t j, uint8_t code)
{
    if (j % 2 == 0)
        row[j / 2] = (uint8_t)((row[j / 2] & 0xF0) | (code & 0xF));
    else
        row[j / 2] = (uint8_t)((row[j / 2] & 0x0F) | (uint8_t)((code & 0xF) << 4));
}

/*
 * MXFP4 (OCP MX v1.0 with E2M1 elements): per 32 consecutive elements the
 * shared exponent floor(log2(max |v|)) - 2 (2 = the largest E2M1 exponent),
 * clamped to [-127, 127], stored as E8M0 (0xFF for a block holding a NaN or
 * an infinity; an all-zero block takes -127); each element v / 2^shared
 * rounded to E2M1.  Codes are packed two per byte, the even element in the
 * low nibble: codes [rows, cols / 2], scales [rows, cols / 32].
 */
int oracle_mxfp4_quantize(const double *v, int64_t rows, int64_t cols, uint8_t *codes,
                          uint8_t *scales)
{
    if (rows < 0 || cols <= 0 || cols % 32 != 0)
        return -1;
    const int64_t nb = cols / 32;
    for (int64_t i = 0; i < rows; ++i) {
        uint8_t *crow = codes + i * (cols / 2);
        for (int64_t b = 0; b < nb; ++b) {
            const double *blk = v + i * cols + b * 32;
            double amax = 0.0;
            int special = 0;
            for (int j = 0; j < 32; ++j) {
                if (isnan(blk[j]) || isinf(blk[j]))
                    special = 1;
                else if (fabs(blk[j]) > amax)
                    amax = fabs(blk[j]);
            }
            int shared = -127;
            if (amax > 0.0) {
                int k;
                frexp(amax, &k);
                shared = (k - 1) - 2;
                if (shared < -127)
                    shared = -127;
                if (shared > 127)
                    shared = 127;
            }
            scales[i * nb + b] = special ? 0xFF : (uint8_t)(shared + 127);
            for (int j = 0; j < 32; ++j)
                put_nibble(crow, b * 32 + j, oracle_e2m1_encode(ldexp(blk[j], -shared)));
        }
    }
    return 0;
}

/*
 * NVFP4 (NVIDIA's description of the format: E2M1 elements, an E4M3 scale
 * per 16 consecutive elements, and a per-tensor fp32 scale g).  A value is
 * represented as code * scale * g.  Per block:
 *     s      = E4M3( max |v| / (6 * g) )        nearest-even, saturating at 448
 *     code_j = E2M1( v_j / (value(s) * g) )     (every code zero when value(s) = 0)
 * The division by 6 maps the block maximum onto the largest E2M1 magnitude.
 * A NaN in the block gives the NaN scale code 0x7F.  g must be positive and
 * finite.  Codes [rows, cols / 2] packed as for MXFP4, scales [rows, cols / 16].
 */
int oracle_nvfp4_quantize(const double *v, int64_t rows, int64_t cols, double g, uint8_t *codes,
                          uint8_t *scales)
{
    if (rows < 0 || cols <= 0 || cols % 16 != 0 || !(g > 0.0) || isinf(g))
        return -1;
    const int64_t nb = cols / 16;
    for (int64_t i = 0; i < rows; ++i) {
        uint8_t *crow = codes + i * (cols / 2);
        for (int64_t b = 0; b < nb; ++b) {
            const double *blk = v + i * cols + b * 16;
            double amax = 0.0;
            int nan = 0;
            for (int j = 0; j < 16; ++j) {
                if (isnan(blk[j]))
                    nan = 1;
                else if (fabs(blk[j]) > amax)
                    amax = fabs(blk[j]);
            }
            uint8_t s = nan ? 0x7F : oracle_e4m3_encode(amax / (6.0 * g));
            scales[i * nb + b] = s;
            double d = nan ? NAN : oracle_e4m3_value(s);
            for (int j = 0; j < 16; ++j) {
                double t = d == 0.0 ? blk[j] * 0.0 : blk[j] / (d * g);
                put_nibble(crow, b * 16 + j, oracle_e2m1_encode(t));
            }
        }
    }
    return 0;
}
