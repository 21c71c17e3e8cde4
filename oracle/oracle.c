/*
 * CPU oracle for the fused 4-bit block-quantized GEMV / skinny GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file.  Only the
 * tests, the package smoke check and the bench's CPU-baseline leg use it.
 * It shares no code, header, table or constant generator with the GPU path.
 *
 * What it computes (plain definitions, single-threaded, no blocking):
 *
 *   1. Decode every super-block of a weight matrix W[M][K] to real values
 *      w[m][k], following the stored block layouts, evaluate each weight in
 *      float64 (exact for every format below) and round once to float32
 *      (round-to-nearest-even), mapping -0 to +0.
 *   2. y[n][m] = sum_k w[m][k] * x[n][k], summed in increasing k in float64
 *      (each product of a float32 and an fp16 value is exact in float64).
 *   3. mag[n][m] = sum_k |w[m][k] * x[n][k]|, the scale of the tolerance.
 *   4. Residual variant: y += residual[n][m] and mag += |residual[n][m]|.
 *
 * Sources (web pages on the subject; cited by page title and section):
 *   - reflex-llm "docs/kernels.md", K-quant GEMV section: y[M] = W[M x K] x[K]
 *     for GGML K-quant weights, types selected by GGML tensor type, weights
 *     dequantized and multiplied without writing fp16 weights back.
 *   - reflex-llm "docs/kernels.md", uint32-loads section: block_q4_K is 144
 *     bytes and qs is read in four 32-byte sub-blocks; block_q6_K is 210 bytes.
 *   - reflex-llm "docs/kernels.md", batched K-quant GEMM section:
 *     y[N x M] = x[N x K] . W^T, output stored token-outer y[token*M + row].
 *   - reflex-llm "docs/performance.md", Path E "What worked": a Q4_K weight is
 *     d * sc[sb] * nibble - dmin * m[sb] over 8 sub-blocks of 32 quants, with
 *     the 6-bit scale/min pairs packed (get_scale_min_k4).
 *   - TandemLLM "Kernels", NVFP4 matrix products: e2m1 weights, one e4m3 scale
 *     per group of 16, products e2m1*e4m3 exact in fp16 (six significant bits).
 *
 * Where the pages name a field but not its bit position, this file follows
 * the GGML K-quant layout (super-block of 256, fields in the order below);
 * each such reading is stated next to the function that uses it.
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar code tables, written from the formats' definitions.               */
/* ------------------------------------------------------------------------ */

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double or_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);             /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* OCP MX e4m3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN. */
double or_e4m3_to_f64(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int f = c & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);              /* f/8 * 2^-6 */
    else
        v = ldexp((double)(8 + f), e - 10);    /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* OCP MX e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit. */
double or_e2m1_to_f64(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int f = c & 0x1;
    double v;
    if (e == 0)
        v = 0.5 * f;                           /* subnormal: f/2 */
    else
        v = ldexp((double)(2 + f), e - 2);     /* (1 + f/2) * 2^(e-1) */
    return sign ? -v : v;
}

/* One rounding to float32 (the C conversion rounds to nearest-even in the
 * default floating-point environment), with -0 mapped to +0. */
static float to_f32_canonical(double v)
{
    float f = (float)v;
    if (f == 0.0f)
        f = 0.0f;
    return f;
}

static uint16_t rd16(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));     /* little-endian fp16 field */
}

/* ------------------------------------------------------------------------ */
/* Row sizes.                                                               */
/* ------------------------------------------------------------------------ */

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits -- the upper half
 * of an IEEE-754 binary32. */
double or_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* subnormal: f * 2^-7 * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);  /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

int64_t or_block_bytes(int type)
{
    switch (type) {
    case OR_Q4_K: return 144;   /* d, dmin, scales[12], qs[128] */
    case OR_Q5_K: return 176;   /* d, dmin, scales[12], qh[32], qs[128] */
    case OR_Q6_K: return 210;   /* ql[128], qh[64], scales[16], d */
    default: return -1;
    }
}

int64_t or_row_bytes(int type, int64_t K)
{
    if (type == OR_NVFP4)
        return K / 2;           /* packed e2m1 codes; scales are separate */
    if (type == OR_FP8)
        return K;               /* one e4m3 code per weight; scales are separate */
    int64_t bb = or_block_bytes(type);
    if (bb < 0 || K % 256 != 0)
        return -1;
    return (K / 256) * bb;
}

/* ------------------------------------------------------------------------ */
/* Q4_K / Q5_K scale and min unpacking.                                     */
/*                                                                          */
/* Reading (GGML layout; the pages only name get_scale_min_k4): the 12      */
/* bytes hold eight 6-bit scales sc[0..7] and eight 6-bit mins m[0..7].     */
/*   s < 4 : sc = scales[s] & 63,            m = scales[s+4] & 63           */
/*   s >= 4: sc = (scales[s+4] & 15) | ((scales[s-4] >> 6) << 4)            */
/*           m  = (scales[s+4] >> 4) | ((scales[s]   >> 6) << 4)            */
/* ------------------------------------------------------------------------ */
void or_unpack_scale_min(const uint8_t *scales, int s, int *sc, int *m)
{
    if (s < 4) {
        *sc = scales[s] & 63;
        *m = scales[s + 4] & 63;
    } else {
        *sc = (scales[s + 4] & 15) | ((scales[s - 4] >> 6) << 4);
        *m = (scales[s + 4] >> 4) | ((scales[s] >> 6) << 4);
    }
}

/* Q4_K block, 144 bytes: d fp16 @0, dmin fp16 @2, scales[12] @4, qs[128] @16.
 * Element order (four 32-byte qs sub-blocks, two nibbles per byte):
 *   byte qs[32c + l] low nibble  -> element 64c + l       (sub-block 2c)
 *   byte qs[32c + l] high nibble -> element 64c + 32 + l  (sub-block 2c+1)
 * Weight: w = d * sc[s] * q - dmin * m[s].  Every term is a multiple of 2^-24
 * below 2^27, so the float64 evaluation is exact. */
static void dequant_block_q4k(const uint8_t *blk, float *out)
{
    double d = or_f16_to_f64(rd16(blk));
    double dmin = or_f16_to_f64(rd16(blk + 2));
    const uint8_t *scales = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        int sc_lo, m_lo, sc_hi, m_hi;
        or_unpack_scale_min(scales, 2 * c, &sc_lo, &m_lo);
        or_unpack_scale_min(scales, 2 * c + 1, &sc_hi, &m_hi);
        for (int l = 0; l < 32; ++l) {
            int byte = qs[32 * c + l];
            int q_lo = byte & 15;
            int q_hi = byte >> 4;
            out[64 * c + l] = to_f32_canonical(d * sc_lo * q_lo - dmin * m_lo);
            out[64 * c + 32 + l] = to_f32_canonical(d * sc_hi * q_hi - dmin * m_hi);
        }
    }
}

/* Q5_K block, 176 bytes: d @0, dmin @2, scales[12] @4, qh[32] @16, qs[128] @48.
 * Reading (GGML layout): the fifth bit of the element in qs byte 32c + l
 * comes from qh[l]: bit 2c for the low nibble (sub-block 2c), bit 2c+1 for
 * the high nibble (sub-block 2c+1).  q5 = nibble + 16 * bit, and
 * w = d * sc[s] * q5 - dmin * m[s]. */
static void dequant_block_q5k(const uint8_t *blk, float *out)
{
    double d = or_f16_to_f64(rd16(blk));
    double dmin = or_f16_to_f64(rd16(blk + 2));
    const uint8_t *scales = blk + 4;
    const uint8_t *qh = blk + 16;
    const uint8_t *qs = blk + 48;
    for (int c = 0; c < 4; ++c) {
        int sc_lo, m_lo, sc_hi, m_hi;
        or_unpack_scale_min(scales, 2 * c, &sc_lo, &m_lo);
        or_unpack_scale_min(scales, 2 * c + 1, &sc_hi, &m_hi);
        for (int l = 0; l < 32; ++l) {
            int byte = qs[32 * c + l];
            int q_lo = (byte & 15) + 16 * ((qh[l] >> (2 * c)) & 1);
            int q_hi = (byte >> 4) + 16 * ((qh[l] >> (2 * c + 1)) & 1);
            out[64 * c + l] = to_f32_canonical(d * sc_lo * q_lo - dmin * m_lo);
            out[64 * c + 32 + l] = to_f32_canonical(d * sc_hi * q_hi - dmin * m_hi);
        }
    }
}

/* Q6_K block, 210 bytes: ql[128] @0, qh[64] @128, int8 scales[16] @192,
 * d fp16 @208.  Reading (GGML layout): two halves h of 128 elements; within
 * half h, for s = 0..3 and l = 0..31, element 128h + 32s + l takes
 *   low 4 bits : ql[64h + 32*(s&1) + l], low nibble for s < 2, high for s >= 2
 *   high 2 bits: bits 2s, 2s+1 of qh[32h + l]
 * q = value - 32 and w = d * scales[8h + l/16 + 2s] * q.  d*sc*q has at most
 * 23 significant bits, so it is exact in float32 and in float64. */
static void dequant_block_q6k(const uint8_t *blk, float *out)
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *scales = (const int8_t *)(blk + 192);
    double d = or_f16_to_f64(rd16(blk + 208));
    for (int h = 0; h < 2; ++h) {
        for (int s = 0; s < 4; ++s) {
            for (int l = 0; l < 32; ++l) {
                int lowbyte = ql[64 * h + 32 * (s & 1) + l];
                int low4 = (s < 2) ? (lowbyte & 15) : (lowbyte >> 4);
                int high2 = (qh[32 * h + l] >> (2 * s)) & 3;
                int q = (low4 | (high2 << 4)) - 32;
                int sc = scales[8 * h + l / 16 + 2 * s];
                out[128 * h + 32 * s + l] = to_f32_canonical(d * sc * q);
            }
        }
    }
}

/* NVFP4 W4A16.  Reading: codes uint8[M][K/2] row-major, element 2i in the low
 * nibble of byte i and element 2i+1 in the high nibble; e4m3 scales
 * uint8[M][K/16] row-major (one per group of 16 consecutive elements); one
 * float32 per-tensor scale g.  w = RN_f32(e2m1 * e4m3 * g); e2m1*e4m3 is exact
 * and the product with g has at most 30 significant bits, exact in float64. */
static void dequant_row_nvfp4(const uint8_t *codes, const uint8_t *scales,
                              float g, int64_t K, float *out)
{
    for (int64_t k = 0; k < K; ++k) {
        uint8_t byte = codes[k / 2];
        uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
        double v = or_e2m1_to_f64(code) * or_e4m3_to_f64(scales[k / 16]) * (double)g;
        out[k] = to_f32_canonical(v);
    }
}

/* FP8 block-scaled (TandemLLM "Kernels", FP8 matrix products: e4m3 codes
 * with one BF16 scale per 128 x 128 block).  Reading: codes uint8[M][K]
 * row-major; scales bf16[ceil(M/128)][K/128] row-major; the weight of
 * (m, k) is e4m3(code) * bf16(scale[m / 128][k / 128]).  The product needs
 * 4 + 8 significant bits, so it is exact in float64 and in float32. */
static void dequant_row_fp8(const uint8_t *codes, const uint16_t *scale_row, int64_t K,
                            float *out)
{
    for (int64_t k = 0; k < K; ++k) {
        double v = or_e4m3_to_f64(codes[k]) * or_bf16_to_f64(scale_row[k / 128]);
        out[k] = to_f32_canonical(v);
    }
}

/* ------------------------------------------------------------------------ */
/* Public dequantization entry points.                                      */
/* ------------------------------------------------------------------------ */

int or_dequant_rows(int type, const uint8_t *w, const uint8_t *scales, float g,
                    int64_t M, int64_t K, const int64_t *rows, int64_t nrows,
                    float *out)
{
    int64_t rb = or_row_bytes(type, K);
    if (rb < 0 || M < 0 || K <= 0)
        return -1;
    if (type == OR_NVFP4 && (K % 16 != 0 || scales == NULL))
        return -1;
    if (type == OR_FP8 && (K % 128 != 0 || scales == NULL))
        return -1;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= M)
            return -2;
        const uint8_t *row = w + r * rb;
        float *dst = out + i * K;
        if (type == OR_NVFP4) {
            dequant_row_nvfp4(row, scales + r * (K / 16), g, K, dst);
            continue;
        }
        if (type == OR_FP8) {
            dequant_row_fp8(row, (const uint16_t *)scales + (r / 128) * (K / 128), K, dst);
            continue;
        }
        for (int64_t b = 0; b < K / 256; ++b) {
            const uint8_t *blk = row + b * or_block_bytes(type);
            float *o = dst + b * 256;
            if (type == OR_Q4_K)
                dequant_block_q4k(blk, o);
            else if (type == OR_Q5_K)
                dequant_block_q5k(blk, o);
            else
                dequant_block_q6k(blk, o);
        }
    }
    return 0;
}

int or_dequant(int type, const uint8_t *w, const uint8_t *scales, float g,
               int64_t M, int64_t K, float *out)
{
    return or_dequant_rows(type, w, scales, g, M, K, NULL, M, out);
}

/* ------------------------------------------------------------------------ */
/* The product.                                                             */
/* ------------------------------------------------------------------------ */

/* The whole path for one weight matrix on selected rows: dequantize the rows
 * and multiply.  rows == NULL means rows 0..nrows-1.  y and mag are
 * [N][nrows]; residual (nullable) is [N][M] and indexed by the real row. */
int or_qgemv_rows(int type, const uint8_t *w, const uint8_t *scales, float g,
                  int64_t M, int64_t K, const int64_t *rows, int64_t nrows,
                  const uint16_t *x, int64_t N, const uint16_t *residual,
                  double *y, double *mag, float *scratch /* [K] */)
{
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        int rc = or_dequant_rows(type, w, scales, g, M, K, &r, 1, scratch);
        if (rc)
            return rc;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *xn = x + n * K;
            double acc = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)scratch[k] * or_f16_to_f64(xn[k]);
                acc += p;
                a += fabs(p);
            }
            if (residual) {
                double rv = or_f16_to_f64(residual[n * M + r]);
                acc += rv;
                a += fabs(rv);
            }
            y[n * nrows + i] = acc;
            if (mag)
                mag[n * nrows + i] = a;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* SwiGLU of the gate/up pair (reflex-llm "docs/kernels.md", SwiGLU         */
/* section: output = silu(gate) x up, silu(v) = v / (1 + exp(-v))).         */
/* ------------------------------------------------------------------------ */

double or_silu(double v)
{
    return v / (1.0 + exp(-v));
}

/* h[i] = silu(g[i]) * u[i] in float64, i < n (g and u are the oracle's
 * float64 products of the gate and up matrices for the same x). */
void or_swiglu(const double *g, const double *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; ++i)
        h[i] = or_silu(g[i]) * u[i];
}
