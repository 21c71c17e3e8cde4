// Skinny fused dequantize-and-multiply kernels: y[N x M] = x[N x K] . W^T for
// Q4_K, Q5_K, Q6_K and NVFP4 weights, fp16 x, fp32 accumulation, N <= 32 per
// launch chunk.
//
// Scheme (one arithmetic path for every N, so a row's bits never depend on N;
// TandemLLM "Kernels", Row invariance):
//   * Weights are the A operand of mma.m16n8k16 (16 rows x 16 k per
//     instruction); x is the B operand (8 tokens per n8 column group).  N only
//     sets how many column groups an A fragment is multiplied with.
//   * A is decoded in registers straight from the packed bytes, exactly:
//       Q4_K  A = sc*q * 2^-14           (nibble as an fp16 subnormal times sc*2^k)
//       Q5_K  A = sc*q5 * 2^-14          (fifth bit merged into the subnormal)
//       Q6_K  A = q - 32                 (magic-number decode)
//       NVFP4 A = e2m1 * e4m3            (hardware cvt, exact in fp16: six bits)
//     (reflex-llm "docs/kernels.md": dequantize in registers, never write fp16
//     weights; TandemLLM "Kernels", NVFP4 matrix products: e2m1*e4m3 is exact.)
//   * Q4_K/Q5_K: per super-block one MMA chain D1 = sum A*x plus one MMA of the
//     6-bit mins against the per-sub-block sums of x (split hi+lo in fp16),
//     folded as acc = fma(d*2^14, D1, acc); acc = fma(-dmin*2^24, D2, acc).
//     Q6_K: one MMA per 16-weight scale group, acc = fma(d*sc, D, acc).
//     NVFP4: one MMA chain over all of K, times the global scale at the end.
//   * The K range is split over a cluster of `ks` CTAs fixed by K alone; the
//     ranks' partial sums are added in rank order through distributed shared
//     memory.  No atomics anywhere.
//   * Weight tiles stream through a multi-stage cp.async (16-byte, L1-bypass)
//     ring in shared memory; the 210-byte Q6_K blocks are copied as their
//     16-byte-aligned supersets and decoded at their byte offset.
//   * x arrives pre-arranged by the staging kernel (qg_stage.cu) in the
//     B-fragment order of each format, so every B load is one conflict-free
//     16-byte shared load.
#pragma once

#include "qg_ptx.cuh"

namespace qg {

enum { T_Q4K = 12, T_Q5K = 13, T_Q6K = 14, T_FP4 = 256 };
enum { TS_Q4K = 1, TS_Q5K = 2, TS_Q6K = 4, TS_FP4 = 8 };
enum { XL_Q4 = 0, XL_Q6 = 1, XL_FP4 = 2, XL_COUNT = 3 };

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kXTok = 576;     // staged bytes per (token, super-block): 512 x + 32 sums + pad
constexpr int kTokChunk = 32;  // tokens per launch chunk
constexpr int kMaxMats = 3;

struct Mat {
    const uint8_t *w;      // packed weights (codes for NVFP4)
    const uint8_t *sc;     // NVFP4 e4m3 scales [M][K/16]
    void *y;               // output [N][M]
    const __half *res;     // residual [N][M] or null
    int64_t row_bytes;     // bytes per packed row
    int64_t sc_row_bytes;  // NVFP4 scale bytes per row
    int64_t w_bytes;       // total packed bytes (Q6_K tail guard)
    int M;
    int type;
    int tile_begin;        // first row tile of this matrix in blockIdx.y
    float gscale;          // NVFP4 per-tensor scale
};

struct Params {
    Mat mat[kMaxMats];
    int nmat;
    const uint8_t *xs[XL_COUNT];  // staged x per layout
    int64_t xs_tok_stride;        // bytes per token in the staged buffers (nb * kXTok)
    int N;                        // tokens of this call
    int tok_base;                 // first token of blockIdx.z == 0
    int nb;                       // 256-wide super-blocks along K
    int ks;                       // K-split ranks (cluster size along x)
    int out_f32;
};

template <int T>
struct Fmt;
template <>
struct Fmt<T_Q4K> {
    static constexpr int BB = 144, RB = 144, VPR = 9, XL = XL_Q4, XV = 34;
};
template <>
struct Fmt<T_Q5K> {
    static constexpr int BB = 176, RB = 176, VPR = 11, XL = XL_Q4, XV = 34;
};
template <>
struct Fmt<T_Q6K> {
    static constexpr int BB = 210, RB = 224, VPR = 14, XL = XL_Q6, XV = 32;
};
template <>
struct Fmt<T_FP4> {
    static constexpr int BB = 128, RB = 144, VPR = 9, XL = XL_FP4, XV = 32;
};

template <int G>
struct Cfg {
    static constexpr int MT = (G <= 2) ? 1 : 2;      // m16 tiles per warp
    static constexpr int STAGES = (G <= 2) ? 4 : 3;  // ring depth
    static constexpr int ROWS = kWarps * MT * 16;    // rows per CTA
};

template <int T, int G>
struct Smem {
    static constexpr int WSLOT = Cfg<G>::MT * 16 * Fmt<T>::RB;
    static constexpr int WPART = kWarps * WSLOT;
    static constexpr int XPART = 8 * G * kXTok;
    static constexpr int STAGE = WPART + XPART;
    static constexpr int TOTAL = Cfg<G>::STAGES * STAGE;
};

template <int TSET, int G>
struct SmemMax {
    static constexpr int a = (TSET & TS_Q4K) ? Smem<T_Q4K, G>::TOTAL : 0;
    static constexpr int b = (TSET & TS_Q5K) ? Smem<T_Q5K, G>::TOTAL : 0;
    static constexpr int c = (TSET & TS_Q6K) ? Smem<T_Q6K, G>::TOTAL : 0;
    static constexpr int d = (TSET & TS_FP4) ? Smem<T_FP4, G>::TOTAL : 0;
    static constexpr int ab = a > b ? a : b;
    static constexpr int cd = c > d ? c : d;
    static constexpr int TOTAL = ab > cd ? ab : cd;
};

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Misaligned (2-byte aligned) 32-bit shared-memory read.
__device__ __forceinline__ uint32_t lds32_any(uint32_t addr)
{
    uint32_t a0 = addr & ~3u;
    uint32_t lo = lds32(a0), hi = lds32(a0 + 4);
    return __funnelshift_r(lo, hi, (addr & 3u) * 8u);
}

// ---------------------------------------------------------------------------
// Q4_K / Q5_K per-row constants from the 16-byte block header.
// Thread t owns sub-blocks 2t (low nibbles of qs chunk t) and 2t+1 (high).
// ---------------------------------------------------------------------------
struct KRow {
    uint32_t slo, shi;  // fp16x2 broadcast scale for the two sub-blocks
    uint32_t amin;      // fp16x2 (m_2t, m_2t+1) * 2^-24 (subnormals)
    float dd, dm;       // d * 2^14 and -dmin * 2^24
};

template <int T>
__device__ __forceinline__ KRow k_row_consts(const uint4 &h, int t)
{
    const int sh = (t & 1) * 16;
    const uint32_t Y = h.y >> sh, Z = h.z >> sh, W = h.w >> sh;
    uint32_t sc, mn;
    if (t < 2) {
        sc = Y & 0x3f3fu;
        mn = Z & 0x3f3fu;
    } else {
        sc = (W & 0x0f0fu) | ((Y >> 2) & 0x3030u);
        mn = ((W >> 4) & 0x0f0fu) | ((Z >> 2) & 0x3030u);
    }
    KRow r;
    const uint32_t v = __byte_perm(sc, 0x6464u, 0x5140u);  // (1024+sc0, 1024+sc1)
    const uint32_t s01 = hsub2(v, 0x64006400u);           // (sc0, sc1), exact
    // Q4_K: low nibbles are q*2^-24 -> scale sc*2^10; high nibbles sit at
    // bits 4..7 (q*2^-20) -> scale sc*2^6.  Q5_K decodes both at q*2^-24.
    const uint32_t hm = hmul2(s01, (T == T_Q4K) ? 0x54006400u : 0x64006400u);
    r.slo = __byte_perm(hm, 0u, 0x1010u);
    r.shi = __byte_perm(hm, 0u, 0x3232u);
    r.amin = __byte_perm(mn, 0u, 0x4140u);
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    r.dd = d * 16384.0f;
    r.dm = -dmin * 16777216.0f;
    return r;
}

// ---------------------------------------------------------------------------
// Per-stage compute, one function per format.  `acc` is [MT][G][4] in the
// mma C-fragment layout: c0/c1 row g tokens 2t/2t+1, c2/c3 row g+8.
// ---------------------------------------------------------------------------
template <int T, int G>
__device__ __forceinline__ void compute_kquant(uint32_t wsl, uint32_t xsl, int g, int t,
                                               int ntok, float (&acc)[Cfg<G>::MT][G][4])
{
    constexpr int MT = Cfg<G>::MT;
    constexpr int RB = Fmt<T>::RB;
    constexpr int QS = (T == T_Q4K) ? 16 : 48;  // qs offset in the block
    KRow rc[MT][2];
    uint4 q[MT][2][2];
    uint4 qh[MT][2][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t ra = wsl + (mt * 16 + g + 8 * rr) * RB;
            const uint4 h = lds128(ra);
            rc[mt][rr] = k_row_consts<T>(h, t);
            q[mt][rr][0] = lds128(ra + QS + 32 * t);
            q[mt][rr][1] = lds128(ra + QS + 32 * t + 16);
            if (T == T_Q5K) {
                qh[mt][rr][0] = lds128(ra + 16);
                qh[mt][rr][1] = lds128(ra + 32);
            }
        }
    }
    float d1[MT][G][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
#pragma unroll
            for (int c = 0; c < 4; ++c) d1[mt][gi][c] = 0.0f;

#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
            uint4 B[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                const int tok = 8 * gi + g;
                B[gi] = (tok < ntok) ? lds128(xsl + tok * kXTok + ((jp * 2 + e) * 4 + t) * 16)
                                     : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * jp + jj;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t p[2][2];  // [row][pair 02/13]
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const uint32_t w = word_of(q[mt][rr][j >> 2], j & 3);
                        if (T == T_Q4K) {
                            if (e == 0) {
                                p[rr][0] = w & 0x000f000fu;
                                p[rr][1] = (w >> 8) & 0x000f000fu;
                            } else {
                                p[rr][0] = w & 0x00f000f0u;
                                p[rr][1] = (w >> 8) & 0x00f000f0u;
                            }
                        } else {
                            const uint32_t hj = word_of(qh[mt][rr][j >> 2], j & 3);
                            const uint32_t hb = hj >> (2 * t + e);
                            const uint32_t ws = e ? (w >> 4) : w;
                            p[rr][0] = (ws & 0x000f000fu) | ((hb << 4) & 0x00100010u);
                            p[rr][1] = ((ws >> 8) & 0x000f000fu) | ((hb >> 4) & 0x00100010u);
                        }
                    }
                    const uint32_t s0 = e ? rc[mt][0].shi : rc[mt][0].slo;
                    const uint32_t s1 = e ? rc[mt][1].shi : rc[mt][1].slo;
                    const uint32_t a0 = hmul2(p[0][0], s0);
                    const uint32_t a1 = hmul2(p[1][0], s1);
                    const uint32_t a2 = hmul2(p[0][1], s0);
                    const uint32_t a3 = hmul2(p[1][1], s1);
#pragma unroll
                    for (int gi = 0; gi < G; ++gi)
                        mma16816(d1[mt][gi], a0, a1, a2, a3, jj ? B[gi].z : B[gi].x,
                                 jj ? B[gi].w : B[gi].y);
                }
            }
        }
    }
    // Mins: one MMA against the per-sub-block sums of x, then the fold.
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        const int tok = 8 * gi + g;
        const uint2 bm = (tok < ntok) ? lds64(xsl + tok * kXTok + 512 + 8 * t) : make_uint2(0u, 0u);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            float d2[4];
            mma16816_zc(d2, rc[mt][0].amin, rc[mt][1].amin, rc[mt][0].amin, rc[mt][1].amin, bm.x,
                        bm.y);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const KRow &r = rc[mt][c >> 1];
                acc[mt][gi][c] = __fmaf_rn(r.dd, d1[mt][gi][c], acc[mt][gi][c]);
                acc[mt][gi][c] = __fmaf_rn(r.dm, d2[c], acc[mt][gi][c]);
            }
        }
    }
}

template <int G>
__device__ __forceinline__ void compute_q6k(uint32_t wsl, uint32_t xsl, int g, int t, int ntok,
                                            const int (&boff)[Cfg<G>::MT][2],
                                            float (&acc)[Cfg<G>::MT][G][4])
{
    constexpr int MT = Cfg<G>::MT;
    constexpr int RB = Fmt<T_Q6K>::RB;
    uint32_t sw[MT][2][4];  // int8 scales, 4 per word
    float dq[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t ba = wsl + (mt * 16 + g + 8 * rr) * RB + boff[mt][rr];
#pragma unroll
            for (int i = 0; i < 4; ++i) sw[mt][rr][i] = lds32_any(ba + 192 + 4 * i);
            dq[mt][rr] =
                __half2float(__ushort_as_half((unsigned short)(lds32_any(ba + 208) & 0xffffu)));
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint32_t ql0[MT][2], ql1[MT][2], qh[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const uint32_t ba = wsl + (mt * 16 + g + 8 * rr) * RB + boff[mt][rr];
                    const uint32_t lo = 64 * h + 16 * i + 4 * t;
                    ql0[mt][rr] = lds32_any(ba + lo);
                    ql1[mt][rr] = lds32_any(ba + lo + 32);
                    qh[mt][rr] = lds32_any(ba + 128 + 32 * h + 16 * i + 4 * t);
                }
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint2 B[G];
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    const int tok = 8 * gi + g;
                    // unit (h, s, t) holds the 4-groups i = 0 and 1
                    B[gi] = (tok < ntok)
                                ? lds64(xsl + tok * kXTok + ((h * 4 + s) * 4 + t) * 16 + 8 * i)
                                : make_uint2(0u, 0u);
                }
                const int grp = 8 * h + i + 2 * s;  // scale index
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a[2][2];
                    float dsc[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const uint32_t ql = (s & 1) ? ql1[mt][rr] : ql0[mt][rr];
                        const uint32_t nw = ((s >> 1) ? (ql >> 4) : ql) & 0x0f0f0f0fu;
                        const uint32_t hw = (s <= 2) ? (qh[mt][rr] << (4 - 2 * s))
                                                     : (qh[mt][rr] >> 2);
                        const uint32_t v = nw | (hw & 0x30303030u);
                        a[rr][0] = hsub2(__byte_perm(v, 0x6464u, 0x5240u), 0x64206420u);
                        a[rr][1] = hsub2(__byte_perm(v, 0x6464u, 0x5341u), 0x64206420u);
                        const int scv = (int)(int8_t)((sw[mt][rr][grp >> 2] >> (8 * (grp & 3))) & 0xffu);
                        dsc[rr] = dq[mt][rr] * (float)scv;
                    }
#pragma unroll
                    for (int gi = 0; gi < G; ++gi) {
                        float d[4];
                        mma16816_zc(d, a[0][0], a[1][0], a[0][1], a[1][1], B[gi].x, B[gi].y);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            acc[mt][gi][c] = __fmaf_rn(dsc[c >> 1], d[c], acc[mt][gi][c]);
                    }
                }
            }
        }
    }
}

template <int G>
__device__ __forceinline__ void compute_fp4(uint32_t wsl, uint32_t xsl, int g, int t, int ntok,
                                            float (&acc)[Cfg<G>::MT][G][4])
{
    constexpr int MT = Cfg<G>::MT;
    constexpr int RB = Fmt<T_FP4>::RB;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint4 cw[MT][2];
        uint32_t sA[MT][2], sB[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const uint32_t ra = wsl + (mt * 16 + g + 8 * rr) * RB;
                cw[mt][rr] = lds128(ra + 64 * hf + 16 * t);
                // scale bytes 8hf + 2t, 8hf + 2t + 1 of the chunk's 16
                const uint32_t sw = lds32(ra + 128 + 8 * hf + 4 * (t >> 1));
                const uint32_t s2 = e4m3x2_to_h2((sw >> (16 * (t & 1))) & 0xffffu);
                sA[mt][rr] = __byte_perm(s2, 0u, 0x1010u);
                sB[mt][rr] = __byte_perm(s2, 0u, 0x3232u);
            }
        }
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
            uint4 B[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                const int tok = 8 * gi + g;
                B[gi] = (tok < ntok) ? lds128(xsl + tok * kXTok + ((hf * 4 + sp) * 4 + t) * 16)
                                     : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int s = 2 * sp + jj;  // step: bytes 2s, 2s+1 of the thread's 16
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a[2][2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const uint32_t w = word_of(cw[mt][rr], s >> 1) >> (16 * (s & 1));
                        const uint32_t sc = (s < 4) ? sA[mt][rr] : sB[mt][rr];
                        a[rr][0] = hmul2(e2m1x2_to_h2(w & 0xffu), sc);
                        a[rr][1] = hmul2(e2m1x2_to_h2((w >> 8) & 0xffu), sc);
                    }
#pragma unroll
                    for (int gi = 0; gi < G; ++gi)
                        mma16816(acc[mt][gi], a[0][0], a[1][0], a[0][1], a[1][1],
                                 jj ? B[gi].z : B[gi].x, jj ? B[gi].w : B[gi].y);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// One CTA: ROWS rows of one matrix, super-blocks [sb0, sb1) of K.
// ---------------------------------------------------------------------------
template <int T, int G>
__device__ __forceinline__ void run_tile(const Params &p, const Mat &m, int rtile, uint8_t *smem)
{
    using F = Fmt<T>;
    using S = Smem<T, G>;
    constexpr int MT = Cfg<G>::MT;
    constexpr int STAGES = Cfg<G>::STAGES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rank = blockIdx.x;
    const int ks = p.ks;
    const int sb0 = (rank * p.nb) / ks;
    const int sb1 = ((rank + 1) * p.nb) / ks;
    const int nsb = sb1 - sb0;
    const int tok0 = p.tok_base + blockIdx.z * kTokChunk;
    const int ntok = min(8 * G, p.N - tok0);
    const int row_w = rtile * Cfg<G>::ROWS + warp * MT * 16;
    const uint32_t sbase = smem_u32(smem);
    const uint8_t *xs = p.xs[F::XL] + (int64_t)tok0 * p.xs_tok_stride;

    auto issue_w = [&](int i) {
        const int sb = sb0 + i;
        const uint32_t dst = sbase + (i % STAGES) * S::STAGE + warp * S::WSLOT;
#pragma unroll 1
        for (int v = lane; v < MT * 16 * F::VPR; v += 32) {
            const int r = v / F::VPR, c = v - r * F::VPR;
            const int row = row_w + r;
            const uint8_t *src = m.w;
            int nbytes = 0;
            if (row < m.M) {
                nbytes = 16;
                if (T == T_FP4) {
                    src = (c < 8) ? m.w + (int64_t)row * m.row_bytes + sb * 128 + c * 16
                                  : m.sc + (int64_t)row * m.sc_row_bytes + sb * 16;
                } else if (T == T_Q6K) {
                    const uint8_t *blk = m.w + (int64_t)row * m.row_bytes + (int64_t)sb * 210;
                    const uint8_t *al = (const uint8_t *)((uintptr_t)blk & ~(uintptr_t)15);
                    src = al + c * 16;
                    const int64_t left = (m.w + m.w_bytes) - src;
                    nbytes = left >= 16 ? 16 : (left > 0 ? (int)left : 0);
                } else {
                    src = m.w + (int64_t)row * m.row_bytes + (int64_t)sb * F::BB + c * 16;
                }
            }
            cp_async16(dst + r * F::RB + c * 16, src, nbytes);
        }
    };
    auto issue_x = [&](int i) {
        const int sb = sb0 + i;
        const uint32_t dst = sbase + (i % STAGES) * S::STAGE + S::WPART;
#pragma unroll 1
        for (int v = threadIdx.x; v < ntok * F::XV; v += kThreads) {
            const int n = v / F::XV, c = v - n * F::XV;
            const uint8_t *src = xs + (int64_t)n * p.xs_tok_stride + (int64_t)sb * kXTok + c * 16;
            cp_async16(dst + n * kXTok + c * 16, src, 16);
        }
    };

    // Weights do not depend on earlier kernels: start them before waiting.
#pragma unroll
    for (int i = 0; i < STAGES - 1; ++i) {
        if (i < nsb) issue_w(i);
        cp_async_commit();
    }
    pdl_wait();
#pragma unroll
    for (int i = 0; i < STAGES - 1; ++i)
        if (i < nsb) issue_x(i);
    cp_async_commit();

    float acc[MT][G][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][gi][c] = 0.0f;

#pragma unroll 1
    for (int i = 0; i < nsb; ++i) {
        if (i == 0)
            cp_async_wait<0>();
        else
            cp_async_wait<STAGES - 2>();
        __syncthreads();
        if (i + STAGES - 1 < nsb) {
            issue_w(i + STAGES - 1);
            issue_x(i + STAGES - 1);
        }
        cp_async_commit();
        const uint32_t stage = sbase + (i % STAGES) * S::STAGE;
        const uint32_t wsl = stage + warp * S::WSLOT;
        const uint32_t xsl = stage + S::WPART;
        if (T == T_Q4K || T == T_Q5K) {
            compute_kquant<T, G>(wsl, xsl, g, t, ntok, acc);
        } else if (T == T_Q6K) {
            int boff[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = min(row_w + mt * 16 + g + 8 * rr, m.M - 1);
                    boff[mt][rr] = (int)((uintptr_t)(m.w + (int64_t)row * m.row_bytes +
                                                     (int64_t)(sb0 + i) * 210) &
                                         15);
                }
            compute_q6k<G>(wsl, xsl, g, t, ntok, boff, acc);
        } else {
            compute_fp4<G>(wsl, xsl, g, t, ntok, acc);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // K-split: ranks 1..ks-1 publish their partial sums; rank 0 adds them in
    // rank order and writes y.
    constexpr int NACC = MT * G * 4;
    if (ks > 1) {
        float *red = reinterpret_cast<float *>(smem);
        if (rank != 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int gi = 0; gi < G; ++gi)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        red[((mt * G + gi) * 4 + c) * kThreads + threadIdx.x] = acc[mt][gi][c];
        }
        cluster_sync();
        if (rank == 0) {
            for (int r = 1; r < ks; ++r) {
                const uint32_t ra = map_shared_rank(smem_u32(red), (uint32_t)r);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int gi = 0; gi < G; ++gi)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            acc[mt][gi][c] += ld_dsmem_f32(
                                ra + (((mt * G + gi) * 4 + c) * kThreads + threadIdx.x) * 4);
            }
        }
        cluster_sync();
    }
    (void)NACC;
    if (rank != 0) return;

#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int row = row_w + mt * 16 + g + 8 * (c >> 1);
                const int tok = tok0 + 8 * gi + 2 * t + (c & 1);
                if (row >= m.M || tok >= p.N) continue;
                float v = acc[mt][gi][c];
                if (T == T_FP4) v = v * m.gscale;
                const int64_t o = (int64_t)tok * m.M + row;
                if (m.res) v = __fadd_rn(__half2float(m.res[o]), v);
                if (p.out_f32)
                    reinterpret_cast<float *>(m.y)[o] = v;
                else
                    reinterpret_cast<__half *>(m.y)[o] = __float2half_rn(v);
            }
        }
    }
}

template <int TSET, int G>
__global__ void __launch_bounds__(kThreads) skinny_kernel(const __grid_constant__ Params p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    // Let the next kernel in the stream start launching; it waits for this
    // grid to finish before touching anything this grid writes.
    pdl_trigger();
    const int tile = blockIdx.y;
    int mi = 0;
    if (p.nmat > 1 && tile >= p.mat[1].tile_begin) mi = 1;
    if (p.nmat > 2 && tile >= p.mat[2].tile_begin) mi = 2;
    const Mat &m = p.mat[mi];
    const int rtile = tile - m.tile_begin;
    if constexpr ((TSET & TS_Q4K) != 0) {
        if (m.type == T_Q4K) {
            run_tile<T_Q4K, G>(p, m, rtile, smem);
            return;
        }
    }
    if constexpr ((TSET & TS_Q5K) != 0) {
        if (m.type == T_Q5K) {
            run_tile<T_Q5K, G>(p, m, rtile, smem);
            return;
        }
    }
    if constexpr ((TSET & TS_Q6K) != 0) {
        if (m.type == T_Q6K) {
            run_tile<T_Q6K, G>(p, m, rtile, smem);
            return;
        }
    }
    if constexpr ((TSET & TS_FP4) != 0) {
        if (m.type == T_FP4) {
            run_tile<T_FP4, G>(p, m, rtile, smem);
            return;
        }
    }
}

// Host-side launch entry generated per type set (one translation unit each).
struct LaunchCfg {
    dim3 grid;
    int smem_bytes;
    int cluster_x;
    bool pdl;
    void *stream;
};

}  // namespace qg
