/*
 * oracle.h -- interface of the fp64 CPU oracle for the row-wise RMSNorm
 * forward.  TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and
 * the benchmark's CPU baseline; never by the CUDA library.
 *
 * Element formats: ORACLE_F32 (IEEE binary32), ORACLE_BF16 (bfloat16 bit
 * patterns as uint16), ORACLE_F16 (IEEE binary16 bit patterns as uint16).
 * All arrays are host memory, row-major, rows x hidden, contiguous.
 * Functions return 0 on success and -1 on a bad argument.
 */
#ifndef RMSNORM_ORACLE_H
#define RMSNORM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* y[i, j] = x[i, j] * (1 / sqrt(sum_k x[i, k]^2 / hidden + eps)) * w[j], in
 * binary64, written as binary64 (no final rounding). */
int oracle_rmsnorm_f64(const void *x, const void *w, double *y, int64_t rows,
                       int64_t hidden, float eps, int fmt);

/* The same result rounded to the element format with round-to-nearest-even
 * directly from binary64. */
int oracle_rmsnorm(const void *x, const void *w, void *y, int64_t rows,
                   int64_t hidden, float eps, int fmt);

/* Exact widening of n stored elements to binary64. */
int oracle_widen_array(const void *in, double *out, int64_t n, int fmt);

/* Round n binary64 values to the format (nearest-even, overflow to inf). */
int oracle_round_array(const double *v, void *out, int64_t n, int fmt);

/* Per-head QK norm, in place: each head of q and of k (head_dim contiguous
 * elements; token t's heads start at t * token_stride) becomes
 * x * (1 / sqrt(sum x^2 / head_dim + eps)) * (w + weight_bias), rounded
 * nearest-even to the element format. */
int oracle_qk_norm(void *q, void *k, const void *q_weight, const void *k_weight, int64_t tokens,
                   int64_t q_heads, int64_t k_heads, int64_t head_dim, int64_t q_token_stride,
                   int64_t k_token_stride, float weight_bias, float eps, int fmt);

/* Row normalisation with a weight offset: y = x * r * (w + weight_bias),
 * binary64 (the _f64 form) or rounded nearest-even to the element format. */
int oracle_rmsnorm_bias_f64(const void *x, const void *w, double *y, int64_t rows,
                            int64_t hidden, float weight_bias, float eps, int fmt);
int oracle_rmsnorm_bias(const void *x, const void *w, void *y, int64_t rows, int64_t hidden,
                        float weight_bias, float eps, int fmt);

/* MXFP8: rows x cols binary64 values (cols a multiple of 32) to E4M3 codes
 * [rows, cols] and E8M0 scales [rows, cols / 32], one scale per 32
 * consecutive elements of a row. */
int oracle_mxfp8_quantize(const double *v, int64_t rows, int64_t cols, uint8_t *codes,
                          uint8_t *scales);
double oracle_e4m3_value(uint8_t code);
uint8_t oracle_e4m3_encode(double v);

/* MXFP4: E2M1 codes packed two per byte (even element in the low nibble)
 * [rows, cols / 2], E8M0 scales [rows, cols / 32]; cols a multiple of 32. */
int oracle_mxfp4_quantize(const double *v, int64_t rows, int64_t cols, uint8_t *codes,
                          uint8_t *scales);
/* NVFP4: E2M1 codes as for MXFP4, E4M3 scales [rows, cols / 16] against the
 * per-tensor scale g > 0; cols a multiple of 16. */
int oracle_nvfp4_quantize(const double *v, int64_t rows, int64_t cols, double g, uint8_t *codes,
                          uint8_t *scales);
double oracle_e2m1_value(uint8_t code);
uint8_t oracle_e2m1_encode(double v);

/* Single-element helpers behind the array functions. */
double oracle_widen(const void *base, int64_t index, int fmt);
double oracle_round_value(double v, int fmt);
void oracle_store(double v, void *base, int64_t index, int fmt);

#ifdef __cplusplus
}
#endif

#endif
