/*
 * CPU oracle for the fused 4-bit block-quantized GEMV — TEST INFRASTRUCTURE.
 * Used only by the tests, the smoke check and the bench's CPU baseline; the
 * CUDA library never includes or links it.  See oracle.c for the readings.
 */
#ifndef SKINNY_Q4_ORACLE_H
#define SKINNY_Q4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Format ids (the K-quant numbers follow GGML's type enumeration). */
enum { OR_Q4_K = 12, OR_Q5_K = 13, OR_Q6_K = 14, OR_NVFP4 = 256, OR_FP8 = 257 };

double or_f16_to_f64(uint16_t h);
double or_e4m3_to_f64(uint8_t c);
double or_e2m1_to_f64(uint8_t c);
double or_bf16_to_f64(uint16_t b);

int64_t or_block_bytes(int type);
int64_t or_row_bytes(int type, int64_t K);
void or_unpack_scale_min(const uint8_t *scales, int s, int *sc, int *m);

int or_dequant(int type, const uint8_t *w, const uint8_t *scales, float g,
               int64_t M, int64_t K, float *out);
int or_dequant_rows(int type, const uint8_t *w, const uint8_t *scales, float g,
                    int64_t M, int64_t K, const int64_t *rows, int64_t nrows,
                    float *out);
int or_qgemv_rows(int type, const uint8_t *w, const uint8_t *scales, float g,
                  int64_t M, int64_t K, const int64_t *rows, int64_t nrows,
                  const uint16_t *x, int64_t N, const uint16_t *residual,
                  double *y, double *mag, float *scratch);

double or_silu(double v);
void or_swiglu(const double *g, const double *u, int64_t n, double *h);

#ifdef __cplusplus
}
#endif

#endif
