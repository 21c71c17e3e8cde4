// Dequantize entry through the product kernels' own decoders.
//
// The product never writes weights back: each warp decodes 16 rows of one
// super-block straight into mma A fragments (kq_decode, q6_decode,
// fp4_decode and the per-row constants k_row_consts / fp4_scales in
// qg_kernels.cuh).  This kernel runs those same functions on the same
// thread mapping and turns every decoded A element into the weight the
// product would return for a one-hot x = e_k, with the product's own
// rounding steps:
//   FP8          w = scale * A             (A = e4m3, exact in fp16)
//   Q4_K / Q5_K  w = fma(-dmin * 2^24, m * 2^-24, (d * 2^22) * A)
//                (A = sc * q * 2^-22; one rounding, as the product's fold)
//   Q6_K         w = d * (sc * A)          (A = q - 32; both products exact)
//   NVFP4        w = A * global_scale      (A = e2m1 * e4m3, exact in fp16)
// so the weights equal the exact values rounded once to fp32 exactly when the
// product's decoders are right (reflex-llm "docs/kernels.md", K-quant GEMV:
// dequantize in registers; the weight formula of "docs/performance.md",
// Path E).  A test path, not a hot path: block bytes are copied to shared
// memory with plain loads.
#include <cuda_runtime.h>

#include "qg_launch.cuh"

namespace qg {

namespace {

constexpr int kDqWarps = 4;
constexpr int kDqPitch = 272;  // bytes per row in shared memory (>= 256, 16-byte multiple)

__device__ __forceinline__ float h_lo(uint32_t v)
{
    return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
__device__ __forceinline__ float h_hi(uint32_t v)
{
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// One warp: rows row0 .. row0 + 15, super-block sb.  rows[] in shared memory
// at `base`: 16 x kDqPitch (K-quants: the block at offset 0; NVFP4: 128 code
// bytes, then the 16 scale bytes at +128).
template <int T>
__device__ void dq_tile(const Mat &m, int K, int row0, int sb, uint32_t base, float *out)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float *const orow[2] = {out + (int64_t)(row0 + g) * K + 256 * sb,
                            out + (int64_t)(row0 + g + 8) * K + 256 * sb};
    const bool live[2] = {row0 + g < m.M, row0 + g + 8 < m.M};
    // (element offset within the super-block, value) -> w_out
    auto put = [&](int rr, int el, float v) {
        if (live[rr]) orow[rr][el] = v;
    };
    if (T == T_Q4K || T == T_Q5K) {
        constexpr int QS = (T == T_Q4K) ? 16 : 48;
        const KSel ks = k_sel(t);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t ra = base + (g + 8 * rr) * kDqPitch;
            const KRow rc = k_row_consts<T>(lds128(ra), ks);
            const uint4 q0 = lds128(ra + QS + 32 * t), q1 = lds128(ra + QS + 32 * t + 16);
            uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
            if (T == T_Q5K) {
                h0 = lds128(ra + 16);
                h1 = lds128(ra + 32);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t w = word_of(j < 4 ? q0 : q1, j & 3);
                const uint32_t hj = word_of(j < 4 ? h0 : h1, j & 3);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint32_t x02, x13;
                    kq_decode<T>(w, hj, t, e, rc.slo, rc.shi, x02, x13);
                    const float mn = e ? h_hi(rc.amin) : h_lo(rc.amin);  // m * 2^-24, exact
                    const int el = 64 * t + 32 * e + 4 * j;  // element of byte 0 of the word
                    const float a[4] = {h_lo(x02), h_lo(x13), h_hi(x02), h_hi(x13)};
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        put(rr, el + b, __fmaf_rn(rc.dm, mn, __fmul_rn(rc.dd, a[b])));
                }
            }
        }
    } else if (T == T_Q6K) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t ba = base + (g + 8 * rr) * kDqPitch;
            uint32_t sw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) sw[i] = lds32(ba + 192 + 4 * i);
            const float dq = h_lo(lds32(ba + 208));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t lo = 64 * h + 16 * i + 4 * t;
                    const uint32_t ql0 = lds32(ba + lo), ql1 = lds32(ba + lo + 32);
                    const uint32_t qh = lds32(ba + 128 + 32 * h + 16 * i + 4 * t);
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        uint32_t x02, x13;
                        q6_decode((s & 1) ? ql1 : ql0, qh, s, x02, x13);
                        const int grp = 8 * h + i + 2 * s;
                        const float scf = (float)(int8_t)((sw[grp >> 2] >> (8 * (grp & 3))) & 0xffu);
                        const int el = 128 * h + 32 * s + 16 * i + 4 * t;
                        const float a[4] = {h_lo(x02), h_lo(x13), h_hi(x02), h_hi(x13)};
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            put(rr, el + b, __fmul_rn(dq, __fmul_rn(scf, a[b])));
                    }
                }
            }
        }
    } else if (T == T_FP8) {
        // compute_fp8's mapping, without the swizzle (rows copied plainly):
        // thread t, scale block c, word j -> elements 128c + 32t + 4j .. + 3
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int row = row0 + g + 8 * rr;
            const uint32_t ca = base + (g + 8 * rr) * kDqPitch;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float sc = 0.0f;
                if (row < m.M) {
                    const uint8_t *sp = m.sc + (int64_t)(row >> 7) * m.sc_row_bytes + 2 * (2 * sb + c);
                    sc = bf16_to_f32((uint32_t)sp[0] | ((uint32_t)sp[1] << 8));
                }
                const uint4 w0 = lds128(ca + 128 * c + 32 * t), w1 = lds128(ca + 128 * c + 32 * t + 16);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t x01, x23;
                    fp8_decode(word_of(j < 4 ? w0 : w1, j & 3), x01, x23);
                    const int el = 128 * c + 32 * t + 4 * j;
                    const float a[4] = {h_lo(x01), h_hi(x01), h_lo(x23), h_hi(x23)};
#pragma unroll
                    for (int b = 0; b < 4; ++b) put(rr, el + b, __fmul_rn(sc, a[b]));
                }
            }
        }
    } else {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t ca = base + (g + 8 * rr) * kDqPitch;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint4 cw = lds128(ca + 64 * hf + 16 * t);
                uint32_t sA, sB;
                fp4_scales(lds32(ca + 128 + 8 * hf + 4 * (t >> 1)), t, sA, sB);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    uint32_t x02, x13;
                    fp4_decode(word_of(cw, s >> 1) >> (16 * (s & 1)), s < 4 ? sA : sB, x02, x13);
                    const int el = 2 * (64 * hf + 16 * t + 2 * s);  // element of code byte B: 2B
                    const float a[4] = {h_lo(x02), h_hi(x02), h_lo(x13), h_hi(x13)};
#pragma unroll
                    for (int b = 0; b < 4; ++b) put(rr, el + b, __fmul_rn(a[b], m.gscale));
                }
            }
        }
    }
}

__global__ void __launch_bounds__(32 * kDqWarps) qg_dequant_kernel(const Mat m, int K,
                                                                      float *out)
{
    __shared__ __align__(16) uint8_t rows[kDqWarps][16 * kDqPitch];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = K / 256;
    const int tiles = (m.M + 15) / 16;
    const int64_t item = (int64_t)blockIdx.x * kDqWarps + warp;
    if (item >= (int64_t)tiles * nb) return;
    const int tile = (int)(item / nb), sb = (int)(item - (int64_t)tile * nb);
    const int row0 = 16 * tile;
    uint8_t *dst = rows[warp];
    // Copy the 16 rows' blocks (rows past M: zeros), 2 bytes at a time (Q6_K
    // blocks are 2-byte aligned; the others are read the same way).
    const int bytes = (m.type == T_FP4) ? 144 : (m.type == T_Q6K) ? 210
                    : (m.type == T_Q5K) ? 176 : (m.type == T_FP8) ? 256 : 144;
    for (int v = lane; v < 16 * (bytes / 2); v += 32) {
        const int r = v / (bytes / 2), c = 2 * (v - r * (bytes / 2));
        const int row = row0 + r;
        uint16_t val = 0;
        if (row < m.M) {
            const uint8_t *src;
            if (m.type == T_FP4)
                src = (c < 128) ? m.w + (int64_t)row * m.row_bytes + 128 * sb + c
                                : m.sc + (int64_t)row * m.sc_row_bytes + 16 * sb + (c - 128);
            else
                src = m.w + (int64_t)row * m.row_bytes + (int64_t)sb * bytes + c;
            val = *reinterpret_cast<const uint16_t *>(src);
        }
        *reinterpret_cast<uint16_t *>(dst + r * kDqPitch + c) = val;
    }
    __syncwarp();
    const uint32_t base = smem_u32(dst);
    switch (m.type) {
    case T_Q4K: dq_tile<T_Q4K>(m, K, row0, sb, base, out); break;
    case T_Q5K: dq_tile<T_Q5K>(m, K, row0, sb, base, out); break;
    case T_Q6K: dq_tile<T_Q6K>(m, K, row0, sb, base, out); break;
    case T_FP8: dq_tile<T_FP8>(m, K, row0, sb, base, out); break;
    default: dq_tile<T_FP4>(m, K, row0, sb, base, out); break;
    }
}

}  // namespace

cudaError_t launch_dequant_fast(const Mat &m, int K, float *out, cudaStream_t stream)
{
    const int64_t items = (int64_t)((m.M + 15) / 16) * (K / 256);
    const int64_t blocks = (items + kDqWarps - 1) / kDqWarps;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    qg_dequant_kernel<<<(unsigned)blocks, 32 * kDqWarps, 0, stream>>>(m, K, out);
    return cudaGetLastError();
}

}  // namespace qg
