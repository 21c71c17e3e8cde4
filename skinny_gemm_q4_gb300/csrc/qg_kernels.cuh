// Skinny fused dequantize-and-multiply kernels: y[N x M] = x[N x K] . W^T for
// Q4_K, Q5_K, Q6_K and NVFP4 weights, fp16 x, fp32 accumulation.
//
// Scheme (one arithmetic path for every N, so a row's bits never depend on N;
// TandemLLM "Kernels", Row invariance):
//   * Weights are the A operand of mma.m16n8k16 (16 rows x 16 k per
//     instruction); x is the B operand (8 tokens per n8 column group).  N only
//     sets how many column groups an A fragment is multiplied with.
//   * A is decoded in registers straight from the packed bytes, exactly:
//       Q4_K  A = sc*q * 2^-22          (nibble as an fp16 subnormal times sc*2^k)
//       Q5_K  A = sc*q5 * 2^-22         (fifth bit merged into the subnormal)
//       Q6_K  A = q - 32                (magic-number decode)
//       NVFP4 A = e2m1 * e4m3           (hardware cvt, exact in fp16: six bits)
//     (reflex-llm "docs/kernels.md": dequantize in registers, never write fp16
//     weights; TandemLLM "Kernels", NVFP4 matrix products: e2m1*e4m3 is exact.)
//   * Q4_K/Q5_K: per super-block two MMA chains, D1a (low nibbles, sub-block
//     2t of thread t) and D1b (high nibbles, 2t+1), plus one MMA of the 6-bit
//     mins against the per-sub-block sums of x (split S = 32 hi + lo in fp16,
//     so every finite fp16 x fits), folded as
//       acc = fma(d*2^22, D1a, acc); acc = fma(d*2^22, D1b, acc);
//       acc = fma(-dmin*2^24, D2, acc).
//     Q6_K: one MMA per 16-weight scale group, accs += sc*D, acc += d*accs.
//     NVFP4: two MMA chains over all of K (even / odd steps), added at the
//     end and multiplied by the global scale.
//   * The K range is cut into kw slices fixed by (M, K) (super-block sb goes
//     to slice sb mod kw); slice partials are added in slice order (shared
//     memory inside a CTA, or distributed shared memory across the cluster
//     ranks of one row tile).  No atomics in the arithmetic.
//   * x arrives in the B-fragment order of each format (stage_sb below), so
//     every B load is one conflict-free 16-byte shared load.
//
// Two data-movement variants share the arithmetic above bit for bit:
//   qg_n8_kernel  (N <= 8, x for the whole K within 48 KB; for N >= 2 not
//                 for Q4_K/Q5_K matrices of at most 4096 rows): a producer
//                 warp streams the weight tiles into an mbarrier ring with one
//                 3-D tensor copy (TMA) per stage (Q6_K, whose 210-byte blocks
//                 are not 16-byte aligned: one 1-D bulk copy per row of the
//                 aligned superset); 8 consumer warps decode and multiply; x
//                 is staged inside the kernel.
//   qg_sk_kernel  (the rest up to N = 32; N >= 33 for NVFP4 and FP8, and for
//                 K-quants created with QG_FLAG_MMA_SYNC_PREFILL; the other
//                 K-quant calls at N >= 33 run on the tcgen05 engine): x staged
//                 once per call by qg_stage.cu; a producer warp streams 128
//                 weight rows and the staged x of one super-block per stage by
//                 TMA; cluster ranks are slices.
#pragma once

#include <cuda.h>

#include "qg_ptx.cuh"

namespace qg {

enum { T_Q4K = 12, T_Q5K = 13, T_Q6K = 14, T_FP4 = 256, T_FP8 = 257 };
enum { TS_Q4K = 1, TS_Q5K = 2, TS_Q6K = 4, TS_FP4 = 8, TS_FP8 = 16 };
// Staged-x layouts: B-fragment orders of the mma.sync kernels, and the
// tensor-core core-matrix layout of qg_tc_kernel (qg_tc.cuh).
enum { XL_Q4 = 0, XL_Q6 = 1, XL_FP4 = 2, XL_TC4 = 3, XL_COUNT = 4 };

constexpr int kXTok = 576;     // staged bytes per (token, super-block): 512 x + 32 sums + pad
constexpr int kTokChunk = 32;  // tokens per blockIdx.z chunk (qg_sk_kernel)
constexpr int kMaxMats = 3;

// Error bits written to Params::err by a kernel (never trap).
enum { ERR_FULL_TIMEOUT = 1, ERR_EMPTY_TIMEOUT = 2 };

struct Mat {
    CUtensorMap tmw;       // 3-D map of the packed rows (Q4_K, Q5_K, NVFP4 codes), gemv box
    CUtensorMap tms;       // 3-D map of the NVFP4 scale rows, gemv box
    CUtensorMap tmw1;      // the same maps with a box of 128 rows x 1 block (qg_sk_kernel)
    CUtensorMap tms1;
    const uint8_t *w;      // packed weights (codes for NVFP4)
    const uint8_t *sc;     // NVFP4 e4m3 scales [M][K/16]; FP8 bf16 scales [ceil(M/128)][K/128]
    void *y;               // output [N][M]
    const __half *res;     // residual [N][M] or null
    int64_t row_bytes;     // bytes per packed row
    int64_t sc_row_bytes;  // NVFP4 scale bytes per row; FP8 per 128-row block
    int64_t w_bytes;       // total packed bytes (Q6_K tail guard)
    int M;
    int type;
    int tile_begin;        // first row tile of this matrix in blockIdx.y
    int kw;                // K slices (fixed by M and K): super-block sb belongs to
                           // slice sb % kw; slice partial sums are added in slice order
    float gscale;          // NVFP4 per-tensor scale
};

struct Params {
    Mat mat[kMaxMats];
    int nmat;
    CUtensorMap xm[XL_COUNT];     // 2-D maps (576-byte super-block units, token) of the staged x
                                  // per layout, box 8G tokens (qg_sk_kernel)
    const uint8_t *xs[XL_COUNT];  // staged x per layout (qg_tc_kernel)
    int64_t xs_tok_stride;        // bytes per token in the staged buffers (nb * kXTok)
    const __half *x;              // raw x [N][K] (qg_n8_kernel stages it itself)
    int N;                        // tokens of this launch
    int tok_base;                 // first token of blockIdx.z == 0
    int K;
    int nb;                       // 256-wide super-blocks along K
    int ks;                       // cluster size along x (the matrices' kw)
    int stages;                   // ring depth (qg_n8_kernel)
    int xstages;                  // x ring depth (qg_tc_kernel; p.stages: its weight ring)
    int xtok;                     // token stride of the in-kernel x region (qg_n8_kernel)
    int out_f32;
    unsigned int *err;            // error word (timeouts)
    int xin;                      // qg_sk_kernel: x staged inside the kernel from p.x
    int swiglu;                   // gate/up pair with the SwiGLU epilogue: mat[0] gate (its y
                                  // receives h = silu(g) * u), mat[1] up, same M and K;
                                  // blockIdx.y = 2 tile + matrix, and the two CTAs of a
                                  // tile (times the K-split ranks) form one cluster
};

template <int T>
struct Fmt;
template <>
struct Fmt<T_Q4K> {
    static constexpr int BB = 144, RB = 144, VPR = 9, XL = XL_Q4, XV = 34, RBG = 144;
};
template <>
struct Fmt<T_Q5K> {
    static constexpr int BB = 176, RB = 176, VPR = 11, XL = XL_Q4, XV = 34, RBG = 176;
};
template <>
struct Fmt<T_Q6K> {
    static constexpr int BB = 210, RB = 224, VPR = 14, XL = XL_Q6, XV = 32, RBG = 224;
};
template <>
struct Fmt<T_FP4> {
    // row in shared memory: 128 code bytes, 16 scale bytes, 48 bytes of pad
    // (a 192-byte pitch keeps the two rows of an 8-lane phase on disjoint banks)
    static constexpr int BB = 128, RB = 192, VPR = 9, XL = XL_FP4, XV = 32, RBG = 144;
};
template <>
struct Fmt<T_FP8> {
    // 256 e4m3 codes per super-block and row; staged x in the NVFP4 order
    static constexpr int BB = 256, RB = 256, VPR = 16, XL = XL_FP4, XV = 32, RBG = 256;
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
// x staging for one (token, super-block): lane l holds x[256 sb + 8l .. +8].
// Writes the layouts that are non-null (generic addresses: global or shared).
//   Q4 : 4-group q = 16t + 8e + j -> 16-byte unit ((j/2)*2 + e)*4 + t, half
//        j&1, stored (x0, x2, x1, x3); bytes 512..543: for t = 0..3 the fp16
//        (hi[2t], hi[2t+1], lo[2t], lo[2t+1]) of the sub-block sums
//        S_s = sum of the 32 x of sub-block s (fp32: sequential within the
//        lane, then a fixed butterfly), hi = fp16(S * 2^-5),
//        lo = fp16(S - 32 hi).  The 2^-5 keeps hi finite for every finite
//        fp16 x (|S| <= 32 * 65504, so |hi| <= 65504) and |lo| <= 512; the
//        min MMA multiplies hi by m * 2^-19 and lo by m * 2^-24.  (hi is an
//        fp16 normal, and power-of-two scaling of x scales the pair exactly,
//        while |S| >= 2^-9.)
//   Q6 : 4-group q = 32h + 8s + 4i + t -> unit (h*4 + s)*4 + t, half i,
//        stored (x0, x2, x1, x3).
//   FP4: the raw 8 values of lane l -> unit ((l/16)*4 + (l&3))*4 + ((l/4)&3).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void stage_sb(uint4 v, int lane, uint8_t *q4, uint8_t *q6, uint8_t *fp4)
{
    if (q4) {
        uint4 o;
        o.x = __byte_perm(v.x, v.y, 0x5410);
        o.y = __byte_perm(v.x, v.y, 0x7632);
        o.z = __byte_perm(v.z, v.w, 0x5410);
        o.w = __byte_perm(v.z, v.w, 0x7632);
        const int u = ((lane & 3) * 2 + ((lane >> 2) & 1)) * 4 + (lane >> 3);
        *reinterpret_cast<uint4 *>(q4 + 16 * u) = o;
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s = __fadd_rn(s, __half2float(__ushort_as_half((unsigned short)(w4[i] & 0xffffu))));
            s = __fadd_rn(s, __half2float(__ushort_as_half((unsigned short)(w4[i] >> 16))));
        }
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2));
        const __half hi = __float2half_rn(__fmul_rn(s, 0.03125f));
        const __half lo = __float2half_rn(__fsub_rn(s, __fmul_rn(__half2float(hi), 32.0f)));
        const uint32_t hib = __half_as_ushort(hi), lob = __half_as_ushort(lo);
        const uint32_t hin = __shfl_down_sync(0xffffffffu, hib, 4);
        const uint32_t lon = __shfl_down_sync(0xffffffffu, lob, 4);
        if ((lane & 7) == 0) {
            uint2 o2;
            o2.x = hib | (hin << 16);
            o2.y = lob | (lon << 16);
            *reinterpret_cast<uint2 *>(q4 + 512 + 8 * (lane >> 3)) = o2;
        }
    }
    if (q6) {
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            const int q = 2 * lane + hq;
            const int h = q >> 5, s = (q >> 3) & 3, i = (q >> 2) & 1, t = q & 3;
            const uint32_t a = hq ? v.z : v.x, b = hq ? v.w : v.y;
            uint2 o2;
            o2.x = __byte_perm(a, b, 0x5410);
            o2.y = __byte_perm(a, b, 0x7632);
            *reinterpret_cast<uint2 *>(q6 + 16 * ((h * 4 + s) * 4 + t) + 8 * i) = o2;
        }
    }
    if (fp4) {
        const int u = ((lane >> 4) * 4 + (lane & 3)) * 4 + ((lane >> 2) & 3);
        *reinterpret_cast<uint4 *>(fp4 + 16 * u) = v;
    }
}

// ---------------------------------------------------------------------------
// Q4_K / Q5_K per-row constants from the 16-byte block header.
// Thread t owns sub-blocks 2t (low nibbles of qs chunk t) and 2t+1 (high).
// A operand = sc * q * 2^-22, exact in fp16 for every sc*q < 2048:
//   Q4_K low nibble  (w & 0x000f000f)  = q * 2^-24, times 4 * sc
//   Q4_K high nibble (w & 0x00f000f0)  = q * 2^-20, times sc / 4
//   Q5_K both (five bits at bits 0..4) = q5 * 2^-24, times 4 * sc
// Both scales come from a magic-number fp16 (0x6C00 | sc = 4096 + 4 sc;
// 0x5C00 | sc = 256 + sc / 4) minus the magic.
// ---------------------------------------------------------------------------
struct KRow {
    uint32_t slo, shi;  // fp16x2 broadcast scale for the two sub-blocks
    uint32_t amin;      // fp16x2 (m_2t, m_2t+1) * 2^-24 (subnormals): times the lo sums,
                        // and times 32 (exact) against the hi sums (S = 32 hi + lo)
    float dd, dm;       // d * 2^22 and -dmin * 2^24
};

// Per-thread selectors for the 6-bit scale/min unpacking (constant per lane).
struct KSel {
    uint32_t selx, selz;  // byte gathers of (scales[0..3], scales[8..11]) / (scales[4..7], ..)
    uint32_t ma, mb;      // 0x3f3f, 0 for t < 2; 0x0f0f, 0x3030 for t >= 2
    uint32_t sh;          // 0 for t < 2; 4 for t >= 2 (mins: high nibble)
};

__device__ __forceinline__ KSel k_sel(int t)
{
    KSel s;
    if (t < 2) {
        // bytes 2t, 2t+1 of word y (scales) / z (mins)
        s.selx = (t == 0) ? 0x3210u : 0x3232u;
        s.selz = s.selx;
        s.ma = 0x3f3fu;
        s.mb = 0u;
        s.sh = 0u;
    } else {
        // [w_2u, w_2u+1, y_2u, y_2u+1] (u = t - 2), word y/z first, w second
        s.selx = (t == 2) ? 0x1054u : 0x3276u;
        s.selz = s.selx;
        s.ma = 0x0f0fu;
        s.mb = 0x3030u;
        s.sh = 4u;
    }
    return s;
}

template <int T>
__device__ __forceinline__ KRow k_row_consts(const uint4 &h, const KSel &ks)
{
    // scales: t < 2: y bytes & 63; t >= 2: (w & 15) | ((y >> 6) << 4)
    const uint32_t X = __byte_perm(h.y, h.w, ks.selx);
    const uint32_t sc = (X & ks.ma) | ((X >> 18) & ks.mb);
    // mins:   t < 2: z bytes & 63; t >= 2: (w >> 4) | ((z >> 6) << 4)
    const uint32_t Z = __byte_perm(h.z, h.w, ks.selz);
    const uint32_t mn = ((Z >> ks.sh) & ks.ma) | ((Z >> 18) & ks.mb);
    KRow r;
    if (T == T_Q4K) {
        r.slo = hsub2(__byte_perm(sc, 0x5C6Cu, 0x4040u), 0x6C006C00u);  // 4 sc0
        r.shi = hsub2(__byte_perm(sc, 0x5C6Cu, 0x5151u), 0x5C005C00u);  // sc1 / 4
    } else {
        r.slo = hsub2(__byte_perm(sc, 0x6C6Cu, 0x4040u), 0x6C006C00u);  // 4 sc0
        r.shi = hsub2(__byte_perm(sc, 0x6C6Cu, 0x5151u), 0x6C006C00u);  // 4 sc1
    }
    r.amin = __byte_perm(mn, 0u, 0x4140u);
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    r.dd = d * 4194304.0f;
    r.dm = -dmin * 16777216.0f;
    return r;
}

// ---------------------------------------------------------------------------
// Exact decoders of one 32-bit word of packed weights into the two fp16x2
// A-operand registers it feeds: x02 holds the elements of bytes 0 and 2 of
// the word (low half, high half), x13 those of bytes 1 and 3.  The product
// kernels and the dequantize entry (qg_dequant.cu) call the same functions.
// ---------------------------------------------------------------------------
// Q4_K / Q5_K: qs word w of thread t, nibble half e (0: low nibbles, sub-block
// 2t; 1: high nibbles, sub-block 2t + 1); Q5_K also takes the qh word hj at
// the same byte offset.  slo / shi: the k_row_consts scales.  Result
// sc * q * 2^-22, exact.
template <int T>
__device__ __forceinline__ void kq_decode(uint32_t w, uint32_t hj, int t, int e, uint32_t slo,
                                          uint32_t shi, uint32_t &x02, uint32_t &x13)
{
    uint32_t p0, p1;
    if (T == T_Q4K) {
        (void)hj;
        (void)t;
        if (e == 0) {
            p0 = w & 0x000f000fu;
            p1 = (w >> 8) & 0x000f000fu;
        } else {
            p0 = w & 0x00f000f0u;
            p1 = (w >> 8) & 0x00f000f0u;
        }
    } else {
        const uint32_t hb = hj >> (2 * t + e);
        const uint32_t ws = e ? (w >> 4) : w;
        p0 = (ws & 0x000f000fu) | ((hb << 4) & 0x00100010u);
        p1 = ((ws >> 8) & 0x000f000fu) | ((hb >> 4) & 0x00100010u);
    }
    const uint32_t sc = e ? shi : slo;
    x02 = hmul2(p0, sc);
    x13 = hmul2(p1, sc);
}

// Q6_K: the ql word (its low nibbles for s < 2, high for s >= 2) and the qh
// word (bits 2s, 2s + 1 of each byte) of scale step s.  Result q - 32, exact.
__device__ __forceinline__ void q6_decode(uint32_t ql, uint32_t qh, int s, uint32_t &x02,
                                          uint32_t &x13)
{
    const uint32_t nw = ((s >> 1) ? (ql >> 4) : ql) & 0x0f0f0f0fu;
    const uint32_t hw = (s <= 2) ? (qh << (4 - 2 * s)) : (qh >> 2);
    const uint32_t v = nw | (hw & 0x30303030u);
    x02 = hsub2(__byte_perm(v, 0x6464u, 0x5240u), 0x64206420u);
    x13 = hsub2(__byte_perm(v, 0x6464u, 0x5341u), 0x64206420u);
}

// NVFP4 group scales of thread t from the scale word sw holding bytes
// 4 (t / 2) .. + 3 of a 64-element half: bytes 2t, 2t + 1 (mod 4), the scales
// of its code bytes 0..7 (sA) and 8..15 (sB), as fp16x2 broadcasts.
__device__ __forceinline__ void fp4_scales(uint32_t sw, int t, uint32_t &sA, uint32_t &sB)
{
    const uint32_t s2 = e4m3x2_to_h2((sw >> (16 * (t & 1))) & 0xffffu);
    sA = __byte_perm(s2, 0u, 0x1010u);
    sB = __byte_perm(s2, 0u, 0x3232u);
}

// NVFP4: two code bytes (low 16 bits of w: elements 2B .. 2B + 3 of code
// byte B, B + 1) times the fp16x2 broadcast group scale.  Result e2m1 * e4m3,
// exact in fp16.
__device__ __forceinline__ void fp4_decode(uint32_t w, uint32_t sc, uint32_t &x02, uint32_t &x13)
{
    x02 = hmul2(e2m1x2_to_h2(w & 0xffu), sc);
    x13 = hmul2(e2m1x2_to_h2((w >> 8) & 0xffu), sc);
}

// FP8: one 32-bit word of e4m3 codes (elements e0..e3 in bytes 0..3) ->
// (e0, e1) and (e2, e3) as fp16x2, exact (every e4m3 value is an fp16 value).
__device__ __forceinline__ void fp8_decode(uint32_t w, uint32_t &x01, uint32_t &x23)
{
    e4m3x4_to_h2x2(w, x01, x23);
}

// bf16 bits -> fp32 (exact).
__device__ __forceinline__ float bf16_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// ---------------------------------------------------------------------------
// Per-super-block compute, one function per format.  wsl: this warp's first
// weight row in shared memory (row pitch RBP); xsl: this super-block's staged
// x for token 0 (token stride xtok).  acc is [MT][G][4] in the mma C-fragment
// layout: c0/c1 row g tokens 2t/2t+1, c2/c3 row g+8.
// ---------------------------------------------------------------------------
template <int T, int MT, int G, bool ODD = true, int RBP = Fmt<T>::RB>
__device__ __forceinline__ void compute_kquant(uint32_t wsl, uint32_t xsl, int xtok, int g, int t,
                                               int ntok, const KSel &ksel, float (&acc)[MT][G][4])
{
    constexpr int QS = (T == T_Q4K) ? 16 : 48;  // qs offset in the block
    KRow rc[MT][2];
    uint4 q[MT][2][2];
    uint4 qh[MT][2][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t ra = wsl + (mt * 16 + g + 8 * rr) * RBP;
            const uint4 h = lds128(ra);
            rc[mt][rr] = k_row_consts<T>(h, ksel);
            q[mt][rr][0] = lds128(ra + QS + 32 * t);
            q[mt][rr][1] = lds128(ra + QS + 32 * t + 16);
            if (T == T_Q5K) {
                qh[mt][rr][0] = lds128(ra + 16);
                qh[mt][rr][1] = lds128(ra + 32);
            }
        }
    }
    // Token columns past ntok read the last real token (their results are
    // never stored), so the B loads need no predicate.
    uint32_t xb[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) xb[gi] = xsl + min(8 * gi + g, ntok - 1) * xtok;
    // Two MMA chains (low and high nibbles) halve the dependent-MMA latency
    // per super-block; the same for every G, so a row's bits do not depend on N.
    constexpr int NC = 2;
    float d1[NC][MT][G][4];
#pragma unroll
    for (int jp = 0; jp < 4; ++jp) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            uint4 B[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi) B[gi] = lds128(xb[gi] + ((jp * 2 + e) * 4 + t) * 16);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * jp + jj;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    kq_decode<T>(word_of(q[mt][0][j >> 2], j & 3),
                                 T == T_Q5K ? word_of(qh[mt][0][j >> 2], j & 3) : 0u, t, e,
                                 rc[mt][0].slo, rc[mt][0].shi, a0, a2);
                    kq_decode<T>(word_of(q[mt][1][j >> 2], j & 3),
                                 T == T_Q5K ? word_of(qh[mt][1][j >> 2], j & 3) : 0u, t, e,
                                 rc[mt][1].slo, rc[mt][1].shi, a1, a3);
#pragma unroll
                    for (int gi = 0; gi < G; ++gi) {
                        const uint32_t b0 = jj ? B[gi].z : B[gi].x, b1 = jj ? B[gi].w : B[gi].y;
                        const int ch = (NC == 2) ? e : 0;
                        if (j == 0 && (NC == 2 || e == 0))
                            mma16816_zc(d1[ch][mt][gi], a0, a1, a2, a3, b0, b1);
                        else
                            mma16816(d1[ch][mt][gi], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
        }
    }
    // Mins: one MMA against the per-sub-block sums of x, then the fold.
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        const uint2 bm = lds64(xb[gi] + 512 + 8 * t);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            float d2[4];
            mma16816_zc(d2, hmul2(rc[mt][0].amin, 0x50005000u), hmul2(rc[mt][1].amin, 0x50005000u),
                        rc[mt][0].amin, rc[mt][1].amin, bm.x,
                        bm.y);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (!ODD && (c & 1)) continue;
                const KRow &r = rc[mt][c >> 1];
#pragma unroll
                for (int ch = 0; ch < NC; ++ch)
                    acc[mt][gi][c] = __fmaf_rn(r.dd, d1[ch][mt][gi][c], acc[mt][gi][c]);
                acc[mt][gi][c] = __fmaf_rn(r.dm, d2[c], acc[mt][gi][c]);
            }
        }
    }
}

// Q6_K: A = q - 32 (exact), one MMA per 16-weight scale group (C = 0), the
// group's int8 scale applied in fp32 (accs += sc * D), the block's d once per
// super-block (acc += d * accs).  Rows sit at byte offset boff[mt][rr] of
// their row in shared memory (row pitch RB); ALIGNED: every such block start
// is 4-byte aligned, so plain 32-bit loads read it.
template <int MT, int G, bool ALIGNED, bool ODD>
__device__ __forceinline__ void q6k_body(uint32_t wsl, int RB, uint32_t xsl, int xtok, int g, int t,
                                         int ntok, const int (&boff)[MT][2],
                                         float (&acc)[MT][G][4])
{
    uint32_t xb[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) xb[gi] = xsl + min(8 * gi + g, ntok - 1) * xtok;
    auto ld = [&](uint32_t a) -> uint32_t { return ALIGNED ? lds32(a) : lds32_any(a); };
    uint32_t sw[MT][2][4];  // int8 scales, 4 per word
    float dq[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t ba = wsl + (mt * 16 + g + 8 * rr) * RB + boff[mt][rr];
#pragma unroll
            for (int i = 0; i < 4; ++i) sw[mt][rr][i] = ld(ba + 192 + 4 * i);
            dq[mt][rr] = __half2float(__ushort_as_half((unsigned short)(ld(ba + 208) & 0xffffu)));
        }
    }
    float accs[MT][G][4];
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
                    ql0[mt][rr] = ld(ba + lo);
                    ql1[mt][rr] = ld(ba + lo + 32);
                    qh[mt][rr] = ld(ba + 128 + 32 * h + 16 * i + 4 * t);
                }
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                uint2 B[G];
                // unit (h, s, t) holds the 4-groups i = 0 and 1
#pragma unroll
                for (int gi = 0; gi < G; ++gi)
                    B[gi] = lds64(xb[gi] + ((h * 4 + s) * 4 + t) * 16 + 8 * i);
                const int grp = 8 * h + i + 2 * s;  // scale index
                const bool first = (h == 0 && i == 0 && s == 0);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a[2][2];
                    float scf[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        q6_decode((s & 1) ? ql1[mt][rr] : ql0[mt][rr], qh[mt][rr], s, a[rr][0],
                                  a[rr][1]);
                        scf[rr] = (float)(int8_t)((sw[mt][rr][grp >> 2] >> (8 * (grp & 3))) & 0xffu);
                    }
#pragma unroll
                    for (int gi = 0; gi < G; ++gi) {
                        float d[4];
                        mma16816_zc(d, a[0][0], a[1][0], a[0][1], a[1][1], B[gi].x, B[gi].y);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (!ODD && (c & 1)) continue;
                            accs[mt][gi][c] = first ? __fmul_rn(scf[c >> 1], d[c])
                                                    : __fmaf_rn(scf[c >> 1], d[c], accs[mt][gi][c]);
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (!ODD && (c & 1)) continue;
                acc[mt][gi][c] = __fmaf_rn(dq[mt][c >> 1], accs[mt][gi][c], acc[mt][gi][c]);
            }
}

template <int MT, int G, bool ODD>
__device__ __forceinline__ void compute_q6k(uint32_t wsl, int RB, uint32_t xsl, int xtok, int g,
                                            int t, int ntok, const int (&boff)[MT][2],
                                            float (&acc)[MT][G][4])
{
    bool al = true;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) al = al && (((wsl + (mt * 16 + g + 8 * rr) * RB +
                                                      boff[mt][rr]) & 3u) == 0);
    if (__all_sync(0xffffffffu, al))
        q6k_body<MT, G, true, ODD>(wsl, RB, xsl, xtok, g, t, ntok, boff, acc);
    else
        q6k_body<MT, G, false, ODD>(wsl, RB, xsl, xtok, g, t, ntok, boff, acc);
}

// NVFP4: acc is [2][MT][G][4] (two chains: even and odd steps).
// Code row r of the warp's tiles at cbase + r * cp (128 bytes), its 16 scale
// bytes at sbase + r * sp.
template <int MT, int G>
__device__ __forceinline__ void compute_fp4(uint32_t cbase, int cp, uint32_t sbase, int sp,
                                            uint32_t xsl, int xtok, int g, int t, int ntok,
                                            float (&acc)[2][MT][G][4])
{
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint4 cw[MT][2];
        uint32_t sA[MT][2], sB[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = mt * 16 + g + 8 * rr;
                cw[mt][rr] = lds128(cbase + r * cp + 64 * hf + 16 * t);
                fp4_scales(lds32(sbase + r * sp + 8 * hf + 4 * (t >> 1)), t, sA[mt][rr],
                           sB[mt][rr]);
            }
        }
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
            uint4 B[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi)
                B[gi] = lds128(xsl + min(8 * gi + g, ntok - 1) * xtok +
                               ((hf * 4 + sp) * 4 + t) * 16);
            // word sp of the thread's 16 code bytes feeds steps 2 sp (bytes 0,
            // 1) and 2 sp + 1 (bytes 2, 3): the values fp4_decode gives, with
            // the four conversions reading the word's bytes directly
            uint32_t hw[MT][2][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
                    e2m1x8_to_h2x4(word_of(cw[mt][rr], sp), hw[mt][rr][0], hw[mt][rr][1],
                                   hw[mt][rr][2], hw[mt][rr][3]);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int s = 2 * sp + jj;  // step: bytes 2s, 2s+1 of the thread's 16
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a[2][2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const uint32_t sc = (s < 4) ? sA[mt][rr] : sB[mt][rr];
                        a[rr][0] = hmul2(hw[mt][rr][2 * jj], sc);
                        a[rr][1] = hmul2(hw[mt][rr][2 * jj + 1], sc);
                    }
#pragma unroll
                    for (int gi = 0; gi < G; ++gi)
                        mma16816(acc[jj][mt][gi], a[0][0], a[1][0], a[0][1], a[1][1],
                                 jj ? B[gi].z : B[gi].x, jj ? B[gi].w : B[gi].y);
                }
            }
        }
    }
}

// FP8 block-scaled (TandemLLM "Kernels", FP8 matrix products: e4m3 codes, one
// bf16 scale per 128 x 128 block).  A super-block is two 128-wide scale
// blocks c; block c of the warp's rows sits in shared memory as a plane of
// 128-byte rows written by a tensor copy with 128-byte swizzle (16-byte chunk
// q of row r at chunk q ^ (r & 7)), plane c at cbase + c * plane.  Thread t
// owns bytes 32t .. 32t + 31 of each row of a block: MMA step j (0..7) takes
// its word j, elements 32t + 4j .. + 3, as fragment columns (2t, 2t + 1) and
// (2t + 8, 2t + 9) -- the staged x (NVFP4 order) gives x in the same order.
// Per block: eight MMAs in one chain from C = 0, then acc = fma(scale, D, acc),
// block 0 then block 1.  sc: the two scales as fp32.
template <int MT, int G, bool ODD>
__device__ __forceinline__ void compute_fp8(uint32_t cbase, int plane, uint32_t xsl, int xtok,
                                            int g, int t, int ntok, const float (&sc)[2],
                                            float (&acc)[MT][G][4])
{
    uint32_t xb[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) xb[gi] = xsl + min(8 * gi + g, ntok - 1) * xtok;
    float d[2][MT][G][4];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint4 w[MT][2][2];  // [mt][row g / g + 8][chunk 2t / 2t + 1]
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = mt * 16 + g + 8 * rr;
                const uint32_t ra = cbase + c * plane + r * 128;
                w[mt][rr][0] = lds128(ra + ((uint32_t)((2 * t) ^ (r & 7)) << 4));
                w[mt][rr][1] = lds128(ra + ((uint32_t)((2 * t + 1) ^ (r & 7)) << 4));
            }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 B[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi) B[gi] = lds128(xb[gi] + ((c * 4 + q) * 4 + t) * 16);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * q + jj;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    fp8_decode(word_of(w[mt][0][j >> 2], j & 3), a0, a2);
                    fp8_decode(word_of(w[mt][1][j >> 2], j & 3), a1, a3);
#pragma unroll
                    for (int gi = 0; gi < G; ++gi) {
                        const uint32_t b0 = jj ? B[gi].z : B[gi].x, b1 = jj ? B[gi].w : B[gi].y;
                        if (j == 0)
                            mma16816_zc(d[c][mt][gi], a0, a1, a2, a3, b0, b1);
                        else
                            mma16816(d[c][mt][gi], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int gi = 0; gi < G; ++gi)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (!ODD && (e & 1)) continue;
                    acc[mt][gi][e] = __fmaf_rn(sc[c], d[c][mt][gi][e], acc[mt][gi][e]);
                }
}

// Per-CTA accumulator set: K-quants fold into one [MT][G][4]; NVFP4 keeps two
// chains.  `finish` returns the rank partial sum of element (mt, gi, c).
template <int T, int MT, int G>
struct Acc {
    float a[(T == T_FP4) ? 2 : 1][MT][G][4];
    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int e = 0; e < ((T == T_FP4) ? 2 : 1); ++e)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int gi = 0; gi < G; ++gi)
#pragma unroll
                    for (int c = 0; c < 4; ++c) a[e][mt][gi][c] = 0.0f;
    }
    __device__ __forceinline__ float partial(int mt, int gi, int c) const
    {
        if (T == T_FP4) return __fadd_rn(a[0][mt][gi][c], a[1][mt][gi][c]);
        return a[0][mt][gi][c];
    }
};

// wsl: the warp's first weight row; for NVFP4 the codes use pitch `cp` and
// the scales start at `fsc` with a 16-byte pitch when fsc != 0 (else they
// follow each code row at +128 with the same pitch).
template <int T, int MT, int G, bool ODD = true>
__device__ __forceinline__ void compute_sb(Acc<T, MT, G> &A, uint32_t wsl, uint32_t xsl, int xtok,
                                           int g, int t, int ntok, const Mat &m, int row_w, int sb,
                                           const KSel &ksel, int cp = Fmt<T>::RB,
                                           uint32_t fsc = 0, int sb0q = -1)
{
    if (sb0q < 0) sb0q = sb;
    if (T == T_Q4K || T == T_Q5K) {
        compute_kquant<T, MT, G, ODD>(wsl, xsl, xtok, g, t, ntok, ksel, A.a[0]);
        (void)cp;  // K-quant rows use the same pitch in both kernels
    } else if (T == T_Q6K) {
        // The slot row holds the 16-byte aligned superset of a run of blocks
        // starting at block sb0q; this block sits (address & 15) + (sb - sb0q)
        // * 210 bytes into it.
        int boff[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = min(row_w + mt * 16 + g + 8 * rr, m.M - 1);
                boff[mt][rr] =
                    (int)((uintptr_t)(m.w + (int64_t)row * m.row_bytes + (int64_t)sb0q * 210) &
                          15) +
                    (sb - sb0q) * 210;
            }
        compute_q6k<MT, G, ODD>(wsl, cp, xsl, xtok, g, t, ntok, boff, A.a[0]);
    } else if (T == T_FP8) {
        // wsl: the warp's rows in the super-block's first scale-block plane;
        // cp: the plane stride; fsc: the CTA's row of bf16 scales in shared
        // memory (two per super-block)
        const uint32_t sw = lds32(fsc + 4 * sb);
        const float sc[2] = {bf16_to_f32(sw & 0xffffu), bf16_to_f32(sw >> 16)};
        compute_fp8<MT, G, ODD>(wsl, cp, xsl, xtok, g, t, ntok, sc, A.a[0]);
    } else {
        compute_fp4<MT, G>(wsl, cp, fsc ? fsc : wsl + 128, fsc ? 16 : cp, xsl, xtok, g, t, ntok,
                           *reinterpret_cast<float(*)[2][MT][G][4]>(&A.a));
    }
}

// Epilogue of one output element: NVFP4 global scale, residual (fp32 add
// before the single rounding), fp16 RN or fp32 store.
template <int T>
__device__ __forceinline__ void store_out(const Params &p, const Mat &m, int row, int tok, float val)
{
    if (row >= m.M || tok >= p.N) return;
    if (T == T_FP4) val = val * m.gscale;
    const int64_t o = (int64_t)tok * m.M + row;
    if (m.res) val = __fadd_rn(__half2float(m.res[o]), val);
    if (p.out_f32)
        reinterpret_cast<float *>(m.y)[o] = val;
    else
        reinterpret_cast<__half *>(m.y)[o] = __float2half_rn(val);
}

// The epilogue of four consecutive rows row .. row + 3 of token tok: one
// 8-byte (fp16) or 16-byte (fp32) store when all four rows exist and the y
// (and residual) addresses are aligned for it, else four scalar stores.
template <int T>
__device__ __forceinline__ void store_out4(const Params &p, const Mat &m, int row, int tok,
                                           float4 v)
{
    if (tok >= p.N) return;
    const int64_t o = (int64_t)tok * m.M + row;
    const uintptr_t ya = p.out_f32 ? (uintptr_t)(reinterpret_cast<float *>(m.y) + o)
                                   : (uintptr_t)(reinterpret_cast<__half *>(m.y) + o);
    const bool vec = row + 3 < m.M && (ya & (p.out_f32 ? 15u : 7u)) == 0 &&
                     (!m.res || ((uintptr_t)(m.res + o) & 7u) == 0);
    if (vec) {
        float a[4] = {v.x, v.y, v.z, v.w};
        if (T == T_FP4)
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] = a[e] * m.gscale;
        if (m.res) {
            const uint2 r = *reinterpret_cast<const uint2 *>(m.res + o);
            const __half2 r01 = *reinterpret_cast<const __half2 *>(&r.x);
            const __half2 r23 = *reinterpret_cast<const __half2 *>(&r.y);
            a[0] = __fadd_rn(__low2float(r01), a[0]);
            a[1] = __fadd_rn(__high2float(r01), a[1]);
            a[2] = __fadd_rn(__low2float(r23), a[2]);
            a[3] = __fadd_rn(__high2float(r23), a[3]);
        }
        if (p.out_f32) {
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(m.y) + o) =
                make_float4(a[0], a[1], a[2], a[3]);
        } else {
            const __half2 h01 = __halves2half2(__float2half_rn(a[0]), __float2half_rn(a[1]));
            const __half2 h23 = __halves2half2(__float2half_rn(a[2]), __float2half_rn(a[3]));
            uint2 u;
            u.x = *reinterpret_cast<const uint32_t *>(&h01);
            u.y = *reinterpret_cast<const uint32_t *>(&h23);
            *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(m.y) + o) = u;
        }
        return;
    }
    store_out<T>(p, m, row, tok, v.x);
    store_out<T>(p, m, row + 1, tok, v.y);
    store_out<T>(p, m, row + 2, tok, v.z);
    store_out<T>(p, m, row + 3, tok, v.w);
}

// SwiGLU epilogue of the gate/up pair (reflex-llm "docs/kernels.md", SwiGLU
// section): h = silu(g) * u, silu(v) = v / (1 + exp(-v)), in fp32 from the two
// products' finished fp32 values, then one rounding to the output type.
__device__ __forceinline__ float qg_silu(float v) { return __fdiv_rn(v, __fadd_rn(1.0f, expf(-v))); }

__device__ __forceinline__ void store_h(const Params &p, const Mat &m, int row, int tok, float g,
                                        float u)
{
    if (row >= m.M || tok >= p.N) return;
    const float h = __fmul_rn(qg_silu(g), u);
    const int64_t o = (int64_t)tok * m.M + row;
    if (p.out_f32)
        reinterpret_cast<float *>(m.y)[o] = h;
    else
        reinterpret_cast<__half *>(m.y)[o] = __float2half_rn(h);
}

// Rank-ordered K-split reduction through distributed shared memory, then the
// epilogue.  Every rank publishes its partial tile in `red` (free shared
// memory of at least ncons * MT * G * 4 floats); after a cluster barrier rank
// q sums the q-th 1/ks of the tile over ranks 0, 1, .., ks-1 in that order
// (all ks remote loads in flight at once, so one distributed-shared-memory
// round trip instead of one per rank) and stores it; a second, relaxed
// barrier keeps every rank's shared memory alive until all reads are done.  The sum order
// per element is the same for every rank split and every N.  Every thread of
// every CTA in the cluster must call this.  cid/ncons: this thread's index
// among the consumer threads; row_cta: the tile's first row (consumer warp w
// holds rows row_cta + 16 MT w ..).
//
// SwiGLU pair (role 0: the gate CTA, 1: the up CTA of the same row tile; -1:
// no SwiGLU): the cluster is [ks gate ranks | ks up ranks]; each up rank
// keeps its finished share (global scale applied) in shared memory and the
// gate rank of the same index reads it through distributed shared memory and
// stores h = silu(g) * u.  g and u get exactly the sums they get in a plain
// pair call.
template <int T, int MT, int G>
__device__ __forceinline__ void reduce_and_store(const Acc<T, MT, G> &A, float *red, int rank,
                                                 int ks, int cid, int ncons, bool consumer,
                                                 const Params &p, const Mat &m, int row_cta,
                                                 int tok0, int g, int t, int role = -1)
{
    constexpr int E = MT * G * 4;  // partial floats per consumer thread
    const uint32_t rank_base = (role == 1) ? (uint32_t)ks : 0u;
    if (ks > 1) {
        // partials published token-major, [token][row] of the tile, so that
        // a float4 of the share is four consecutive rows of one token
        const int nrows = (ncons >> 5) * MT * 16;
        if (consumer) {
            const int rw = (cid >> 5) * MT * 16;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int gi = 0; gi < G; ++gi)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        red[(8 * gi + 2 * t + (c & 1)) * nrows + rw + mt * 16 + g + 8 * (c >> 1)] =
                            A.partial(mt, gi, c);
        }
        cluster_sync();
        const int per = E * ncons / ks;  // floats of this rank's share (a multiple of 4)
        const uint32_t rbase = smem_u32(red);
        for (int q4 = threadIdx.x; 4 * q4 < per; q4 += blockDim.x) {
            const int idx0 = rank * per + 4 * q4;
            float4 part[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < ks)
                    part[r] = ld_dsmem_v4(map_shared_rank(rbase + 4 * idx0, rank_base + (uint32_t)r));
            float4 sum = part[0];
#pragma unroll
            for (int r = 1; r < 8; ++r) {
                if (r < ks) {
                    sum.x += part[r].x;
                    sum.y += part[r].y;
                    sum.z += part[r].z;
                    sum.w += part[r].w;
                }
            }
            const int tl = idx0 / nrows, rl = idx0 - tl * nrows;
            if (role < 0) {
                store_out4<T>(p, m, row_cta + rl, tok0 + tl, sum);
            } else {
                // this rank's finished share, after the partials it read
                if (T == T_FP4) {
                    sum.x *= m.gscale;
                    sum.y *= m.gscale;
                    sum.z *= m.gscale;
                    sum.w *= m.gscale;
                }
                *reinterpret_cast<float4 *>(red + E * ncons + 4 * q4) = sum;
            }
        }
        if (role >= 0) {
            cluster_sync();  // every rank's share is in place
            if (role == 0) {
                const uint32_t xb = smem_u32(red + E * ncons);
                for (int q4 = threadIdx.x; 4 * q4 < per; q4 += blockDim.x) {
                    const int idx0 = rank * per + 4 * q4;
                    const float4 gv = *reinterpret_cast<const float4 *>(red + E * ncons + 4 * q4);
                    const float4 uv =
                        ld_dsmem_v4(map_shared_rank(xb + 16 * q4, (uint32_t)(rank + ks)));
                    const int tl = idx0 / nrows, rl = idx0 - tl * nrows;
                    store_h(p, m, row_cta + rl, tok0 + tl, gv.x, uv.x);
                    store_h(p, m, row_cta + rl + 1, tok0 + tl, gv.y, uv.y);
                    store_h(p, m, row_cta + rl + 2, tok0 + tl, gv.z, uv.z);
                    store_h(p, m, row_cta + rl + 3, tok0 + tl, gv.w, uv.w);
                }
            }
        }
        // every remote read has returned (its value was summed): the other
        // CTAs may exit once all have arrived; the y stores need no wait
        cluster_arrive_relaxed();
        cluster_wait();
        return;
    }
    if (role >= 0) {
        // no K split: the up CTA (cluster rank 1) publishes its values, indexed
        // [element][consumer thread], for the gate CTA (rank 0)
        if (consumer && role == 1) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int gi = 0; gi < G; ++gi)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v = A.partial(mt, gi, c);
                        if (T == T_FP4) v = v * m.gscale;
                        red[((mt * G + gi) * 4 + c) * ncons + cid] = v;
                    }
        }
        cluster_sync();
        if (consumer && role == 0) {
            const int row_w = row_cta + (cid >> 5) * MT * 16;
            const uint32_t xb = smem_u32(red);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int gi = 0; gi < G; ++gi)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float gv = A.partial(mt, gi, c);
                        if (T == T_FP4) gv = gv * m.gscale;
                        const float uv = ld_dsmem_f32(map_shared_rank(
                            xb + 4 * (((mt * G + gi) * 4 + c) * ncons + cid), 1u));
                        store_h(p, m, row_w + mt * 16 + g + 8 * (c >> 1),
                                tok0 + 8 * gi + 2 * t + (c & 1), gv, uv);
                    }
        }
        cluster_sync();  // the up CTA's values stay readable until read
        return;
    }
    if (!consumer) return;
    const int row_w = row_cta + (cid >> 5) * MT * 16;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int gi = 0; gi < G; ++gi)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                store_out<T>(p, m, row_w + mt * 16 + g + 8 * (c >> 1),
                             tok0 + 8 * gi + 2 * t + (c & 1), A.partial(mt, gi, c));
}

// FP8: the bf16 scales of the CTA's 128-row block (K/128 of them, K/256
// 32-bit words) into shared memory at dst, by threads tid0.. of `nthr`.
__device__ __forceinline__ void load_fp8_scales(const Mat &m, int K, int row0, uint32_t *dst,
                                                int tid, int nthr)
{
    const uint32_t *src = reinterpret_cast<const uint32_t *>(m.sc + (int64_t)(row0 >> 7) *
                                                                         m.sc_row_bytes);
    for (int i = tid; i < K / 256; i += nthr) dst[i] = __ldg(src + i);
}

// Shared memory of an FP8 launch: barriers in [0, 64), the scale row in
// [128, 1024) (K <= 57,344), the weight ring from the first 1024-byte
// boundary at or after offset 1024 (the 128-byte swizzle of the tensor copies
// needs 1024-byte aligned slots); the host adds 1024 bytes of slack.
constexpr int kFp8RingOffset = 2048;  // bytes the ring may start after the base
constexpr int kFp8MaxK = (1024 - 128) * 64;
__device__ __forceinline__ uint32_t fp8_ring(uint32_t sbase) { return (sbase + 1024 + 1023) & ~1023u; }

__device__ __forceinline__ int select_mat(const Params &p, int tile)
{
    int mi = 0;
    if (p.nmat > 1 && tile >= p.mat[1].tile_begin) mi = 1;
    if (p.nmat > 2 && tile >= p.mat[2].tile_begin) mi = 2;
    return mi;
}

// ===========================================================================
// qg_n8_kernel (N <= 8): warp 0 produces, warps 1..CW consume (16 rows each).
// Shared memory: [full[STAGES], empty[STAGES] mbarriers | STAGES weight slots
// of rows_cta * RB bytes | x region: N tokens x (this rank's super-blocks) x
// 576 bytes, token stride p.xtok].
// ===========================================================================
constexpr int kGemvStagesMax = 4;
constexpr int kGemvCW = 8;        // consumer warps per CTA
constexpr int kGemvRows = 16 * kGemvCW;  // rows per CTA when kw == 1

// Bytes of one stage row for Q6_K: the 16-byte aligned superset of kw
// consecutive 210-byte blocks.
__host__ __device__ inline int q6_pitch(int kw) { return ((14 + 210 * kw) + 15) & ~15; }

// Slot layout of one stage (R = 128 / kw rows, kw super-blocks: one per slice):
//   Q4_K / Q5_K : [kw][R][BB]                 one 3-D tensor copy
//   NVFP4       : [kw][R][128] codes, then [kw][R][16] scales (two copies)
//   Q6_K        : [R][q6_pitch(kw)]          one 1-D bulk copy per row
// Consumer warp c takes row tile c / kw and K slice c % kw.
template <int T>
__device__ __forceinline__ int gemv_stage_bytes(int kw)
{
    const int R = kGemvRows / kw;
    if (T == T_Q6K) return R * q6_pitch(kw);
    if (T == T_FP4) return kw * R * (128 + 16);
    return kw * R * Fmt<T>::BB;
}

// One stage of the N <= 8 weight ring: super-blocks i*kw .. i*kw + kw - 1 of
// rows row0 .. row0 + R - 1 into the slot at shared address dst (generic
// pointer dstp), completing on the full barrier fb.  stage_bytes must be
// exactly the bytes the tensor copies deliver (gemv_stage_bytes<T>(kw)): the
// barrier's phase completes when that many have landed.  Called by the
// whole producer warp.  The weights are read once per call: evict-first in L2.
template <int T>
__device__ __forceinline__ void gemv_produce(const Mat &m, int kw, int R, int row0, int nb, int i,
                                             uint32_t dst, uint8_t *dstp, uint32_t fb,
                                             int stage_bytes, uint64_t wpol, int lane)
{
    const int sbq = i * kw;
    if (T != T_Q6K) {
        if (lane == 0) {
            mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
            if (T == T_FP4) {
                tma_load_3d_ef(dst, &m.tmw, 0, row0, sbq, fb, wpol);
                tma_load_3d_ef(dst + kw * R * 128, &m.tms, 0, row0, sbq, fb, wpol);
            } else if (T == T_FP8) {
                // planes of 128 codes: two per super-block
                tma_load_3d_ef(dst, &m.tmw, 0, row0, 2 * sbq, fb, wpol);
            } else {
                tma_load_3d_ef(dst, &m.tmw, 0, row0, sbq, fb, wpol);
            }
        }
        return;
    }
    // Q6_K: per row, the aligned superset of the stage's blocks; anything
    // past the end of the matrix is not read.
    const int nv = min(kw, nb - sbq);
    const int pitch = q6_pitch(kw);
    const uint8_t *end = m.w + m.w_bytes;
    uint32_t bytes = 0;
    for (int r = lane; r < R; r += 32) {
        const int row = row0 + r;
        if (row >= m.M) continue;
        const uint8_t *blk = m.w + (int64_t)row * m.row_bytes + (int64_t)sbq * 210;
        const uint8_t *al = (const uint8_t *)((uintptr_t)blk & ~(uintptr_t)15);
        const uint8_t *stop = blk + 210 * nv;
        uint32_t n = (uint32_t)(((stop - al) + 15) & ~(int64_t)15);
        if (al + n > end) {
            n = (uint32_t)((end - al) & ~(int64_t)15);
            uint8_t *d = dstp + r * pitch;
            for (uint32_t b = n; al + b < stop; ++b) d[b] = al[b];
        }
        bytes += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
    __syncwarp();
    for (int r = lane; r < R; r += 32) {
        const int row = row0 + r;
        if (row >= m.M) continue;
        const uint8_t *blk = m.w + (int64_t)row * m.row_bytes + (int64_t)sbq * 210;
        const uint8_t *al = (const uint8_t *)((uintptr_t)blk & ~(uintptr_t)15);
        const uint8_t *stop = blk + 210 * nv;
        uint32_t n = (uint32_t)(((stop - al) + 15) & ~(int64_t)15);
        if (al + n > end) n = (uint32_t)((end - al) & ~(int64_t)15);
        if (n) bulk_g2s_ef(dst + r * pitch, al, n, fb, wpol);
    }
}

template <int T, bool ODD>
__device__ __forceinline__ void gemv_tile(const Params &p, const Mat &m, int rtile, uint8_t *smem,
                                          int role)
{
    using F = Fmt<T>;
    constexpr bool TMA = (T != T_Q6K);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int kw = m.kw;
    const int R = kGemvRows / kw;
    const int STAGES = p.stages;
    const int nst = (p.nb + kw - 1) / kw;      // stages of this CTA
    const int ntok = p.N;                      // <= 8
    const int row0 = rtile * R;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase, bar_empty = sbase + 8 * kGemvStagesMax;
    const int slot_bytes = gemv_stage_bytes<T>(kw);
    const uint32_t slots = (T == T_FP8) ? fp8_ring(sbase) : sbase + 128;
    const uint32_t xreg = slots + STAGES * slot_bytes;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kGemvCW);
        }
        mbar_fence_init();
    }
    if (TMA && warp == 0 && lane == 0) {
        prefetch_tmap(&m.tmw);
        if (T == T_FP4) prefetch_tmap(&m.tms);
    }
    __syncthreads();

    // Producer: fill slot `slot` with stage i (super-blocks i*kw .. i*kw + kw - 1).
    const uint64_t wpol = l2_evict_first_policy();
    auto produce = [&](int i, int slot) {
        const uint32_t dst = slots + slot * slot_bytes;
        gemv_produce<T>(m, kw, R, row0, p.nb, i, dst, smem + (dst - sbase), bar_full + 8 * slot,
                        slot_bytes, wpol, lane);
    };

    unsigned int err = 0;
    if (warp == 0) {
        for (int i = 0; i < STAGES && i < nst; ++i) produce(i, i);
    } else if (T == T_FP8) {
        // the block scales, like the weights, need nothing from earlier kernels
        load_fp8_scales(m, p.K, row0, reinterpret_cast<uint32_t *>(smem + 128), threadIdx.x - 32,
                        32 * kGemvCW);
    }

    // x for the whole K range, staged after the programmatic dependency (x
    // may be written by the previous kernel): by every warp, except that the
    // Q6_K producer (still issuing its per-row copies) leaves it to the
    // consumer warps.
    pdl_wait();
    {
        // Loads for up to four items are in flight at once (one L2 round trip
        // per four items instead of one per item).
        // Item it = n * nb + sb; staging warp xw takes it = xw, xw + nwarps,
        // ... and steps (n, sb) without dividing.
        constexpr int XU = 4;
        constexpr int W0 = TMA ? 0 : 1;  // first staging warp
        const int nwarps = (blockDim.x >> 5) - W0;
        const int xw = warp - W0;
        const int nb = p.nb;
        const int total = xw < 0 ? 0 : ntok * nb;
        int n = 0, sb = xw < 0 ? 0 : xw;
        while (sb >= nb) {
            sb -= nb;
            ++n;
        }
        for (int base = xw; base < total; base += XU * nwarps) {
            uint4 v[XU];
            uint32_t dst[XU];
#pragma unroll
            for (int u = 0; u < XU; ++u) {
                if (base + u * nwarps < total) {
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(p.x + (int64_t)n * p.K +
                                                                 256 * sb + 8 * lane));
                    dst[u] = (uint32_t)(n * p.xtok + sb * kXTok);
                }
                sb += nwarps;
                while (sb >= nb) {
                    sb -= nb;
                    ++n;
                }
            }
#pragma unroll
            for (int u = 0; u < XU; ++u) {
                if (base + u * nwarps < total) {
                    uint8_t *d = smem + (xreg - sbase) + dst[u];
                    stage_sb(v[u], lane, F::XL == XL_Q4 ? d : nullptr,
                             F::XL == XL_Q6 ? d : nullptr, F::XL == XL_FP4 ? d : nullptr);
                }
            }
        }
    }
    // x is staged.  The Q6_K producer took no part in it and may still be
    // issuing its first stages' per-row copies: only the consumers meet.
    if (TMA)
        __syncthreads();
    else if (warp > 0)
        bar_sync_named(1, 32 * kGemvCW);

    Acc<T, 1, 1> A;
    A.zero();
    const int c = warp - 1;
    const int mg = c / kw, ks = c - mg * kw;
    const int row_w = row0 + 16 * mg;
    const KSel ksel = k_sel(t);
    if (warp == 0) {
        // stage i reuses slot i % STAGES after its consumers released it
        int slot = 0;
        uint32_t par = 0;
        for (int i = STAGES; i < nst; ++i) {
            if (!mbar_wait(bar_empty + 8 * slot, par)) {
                err |= ERR_EMPTY_TIMEOUT;
                break;
            }
            produce(i, slot);
            if (++slot == STAGES) {
                slot = 0;
                par ^= 1u;
            }
        }
    } else {
        int slot = 0;
        uint32_t par = 0;
        const uint32_t wrow = (T == T_Q6K) ? (uint32_t)(16 * mg * q6_pitch(kw))
                            : (T == T_FP4) ? (uint32_t)((ks * R + 16 * mg) * 128)
                            : (T == T_FP8) ? (uint32_t)((2 * ks * R + 16 * mg) * 128)
                                           : (uint32_t)((ks * R + 16 * mg) * F::BB);
        const uint32_t srow = (uint32_t)(kw * R * 128 + (ks * R + 16 * mg) * 16);
        for (int i = 0; i < nst; ++i) {
            if (!mbar_wait(bar_full + 8 * slot, par)) {
                err |= ERR_FULL_TIMEOUT;
                break;
            }
            const int sb = i * kw + ks;
            if (sb < p.nb) {
                const uint32_t sl = slots + slot * slot_bytes;
                const uint32_t xsl = xreg + sb * kXTok;
                if (T == T_FP4) {
                    compute_sb<T, 1, 1, ODD>(A, sl + wrow, xsl, p.xtok, g, t, ntok, m, row_w, sb,
                                             ksel, 128, sl + srow);
                } else if (T == T_FP8) {
                    compute_sb<T, 1, 1, ODD>(A, sl + wrow, xsl, p.xtok, g, t, ntok, m, row_w, sb,
                                             ksel, R * 128, sbase + 128);
                } else if (T == T_Q6K) {
                    compute_sb<T, 1, 1, ODD>(A, sl + wrow, xsl, p.xtok, g, t, ntok, m, row_w, sb,
                                             ksel, q6_pitch(kw), 0u, i * kw);
                } else {
                    compute_sb<T, 1, 1, ODD>(A, sl + wrow, xsl, p.xtok, g, t, ntok, m, row_w, sb,
                                             ksel);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
            if (++slot == STAGES) {
                slot = 0;
                par ^= 1u;
            }
        }
    }
    if (err && p.err) atomicOr(p.err, err);
    __syncthreads();

    // Slice partials: slices 1..kw-1 publish, slice 0 adds them in slice order.
    float *red = reinterpret_cast<float *>(smem + 128);
    float v[4];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) v[cc] = A.partial(0, 0, cc);
    if (warp > 0 && ks > 0) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) red[(c * 4 + cc) * 32 + lane] = v[cc];
    }
    __syncthreads();
    const bool fin = warp > 0 && ks == 0;  // slice-0 warps finish their rows
    if (fin) {
        for (int q = 1; q < kw; ++q) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) v[cc] += red[((c + q) * 4 + cc) * 32 + lane];
        }
    }
    if (role >= 0) {
        // SwiGLU pair: the up CTA (cluster rank 1) hands its finished values
        // to the gate CTA (rank 0) of the same rows, which stores
        // h = silu(g) * u; both get exactly the sums of a plain pair call.
        float *xb = red + kGemvCW * 4 * 32;
        if (fin && role == 1) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                xb[(c * 4 + cc) * 32 + lane] = (T == T_FP4) ? v[cc] * m.gscale : v[cc];
        }
        cluster_sync();
        if (fin && role == 0) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const float u = ld_dsmem_f32(
                    map_shared_rank(smem_u32(xb + (c * 4 + cc) * 32 + lane), 1u));
                store_h(p, m, row_w + g + 8 * (cc >> 1), 2 * t + (cc & 1),
                        (T == T_FP4) ? v[cc] * m.gscale : v[cc], u);
            }
        }
        cluster_sync();  // the up CTA's values stay readable until read
        return;
    }
    if (!fin) return;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int row = row_w + g + 8 * (cc >> 1);
        const int tok = 2 * t + (cc & 1);
        if (row >= m.M || tok >= p.N) continue;
        float val = v[cc];
        if (T == T_FP4) val = val * m.gscale;
        const int64_t o = (int64_t)tok * m.M + row;
        if (m.res) val = __fadd_rn(__half2float(m.res[o]), val);
        if (p.out_f32)
            reinterpret_cast<float *>(m.y)[o] = val;
        else
            reinterpret_cast<__half *>(m.y)[o] = __float2half_rn(val);
    }
}

// ONE: N == 1, so only the even token column of each accumulator pair is
// folded (the odd columns are never stored; the even ones get the same
// arithmetic as for any other N).
template <int TSET, bool ONE>
__global__ void __launch_bounds__(32 * (kGemvCW + 1)) qg_n8_kernel(const __grid_constant__ Params p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_trigger();
    const int tile = blockIdx.y;
    const int mi = p.swiglu ? (tile & 1) : select_mat(p, tile);
    const Mat &m = p.mat[mi];
    const int rtile = p.swiglu ? (tile >> 1) : tile - m.tile_begin;
    const int role = p.swiglu ? mi : -1;
    if constexpr ((TSET & TS_Q4K) != 0)
        if (m.type == T_Q4K) return gemv_tile<T_Q4K, !ONE>(p, m, rtile, smem, role);
    if constexpr ((TSET & TS_Q5K) != 0)
        if (m.type == T_Q5K) return gemv_tile<T_Q5K, !ONE>(p, m, rtile, smem, role);
    if constexpr ((TSET & TS_Q6K) != 0)
        if (m.type == T_Q6K) return gemv_tile<T_Q6K, !ONE>(p, m, rtile, smem, role);
    if constexpr ((TSET & TS_FP4) != 0)
        if (m.type == T_FP4) return gemv_tile<T_FP4, !ONE>(p, m, rtile, smem, role);
    if constexpr ((TSET & TS_FP8) != 0)
        if (m.type == T_FP8) return gemv_tile<T_FP8, !ONE>(p, m, rtile, smem, role);
}

// Dynamic shared memory of qg_n8_kernel: barriers, `stages` ring slots of
// `stage_bytes`, and the x region of N tokens x nb super-blocks.
__host__ __device__ inline int gemv_xtok(int nb) { return nb * kXTok + ((nb & 1) ? 0 : 64); }
__host__ __device__ inline int gemv_smem_bytes(int stage_bytes, int stages, int N, int nb,
                                               bool fp8 = false)
{
    const int body = stages * stage_bytes + N * gemv_xtok(nb);
    const int red = 2 * kGemvCW * 4 * 32 * 4;  // slice partials (+ SwiGLU exchange) overlay the ring
    return (fp8 ? kFp8RingOffset : 128) + (body > red ? body : red);
}

}  // namespace qg

namespace qg {

// ===========================================================================
// qg_sk_kernel (N > 8, and N <= 8 when x does not fit qg_n8_kernel's shared
// memory or the matrix is a Q4_K/Q5_K one of at most 4096 rows): warp 0
// streams, per super-block of this cluster rank's K slice,
// the weights of 128 rows (one 3-D tensor copy; Q6_K rows are loaded by
// their consumer warp with 16-byte cp.async) and the staged x of up to 32
// tokens (one 2-D tensor copy) into an mbarrier ring; warps 1..8 each decode
// and multiply 16 rows against G column groups.  The slices and their
// rank-order sum through distributed shared memory follow the same plan as
// qg_n8_kernel's in-CTA slices, so every row gets the same bits on either.
// Shared memory: [full[4], empty[4] | ring | (after the loop) rank partials].
// ===========================================================================
constexpr int kSkCons = 8;
constexpr int kSkRows = 16 * kSkCons;
constexpr int kSkThreads = 32 * (kSkCons + 1);
constexpr int kSkStagesMax = 4;

__host__ __device__ inline int sk_wbytes(int type)
{
    return kSkRows * (type == T_FP8 ? 256 : type == T_Q6K ? 224 : type == T_Q5K ? 176 : 144);
}
// Bytes of one ring slot: the stage's bytes (weights only when x is staged in
// the kernel), rounded up to 1024 for FP8 (swizzled tensor copies).
__host__ __device__ inline int sk_slot_bytes(bool fp8, int stage_with_x, int wbytes)
{
    const int b = stage_with_x ? stage_with_x : wbytes;
    return fp8 ? ((b + 1023) & ~1023) : b;
}
__host__ __device__ inline int sk_stage_bytes(int wbytes, int G) { return wbytes + 8 * G * kXTok; }
__host__ __device__ inline int sk_smem_bytes(int wbytes, int G, int stages, bool fp8 = false)
{
    const int ring = stages * sk_slot_bytes(fp8, sk_stage_bytes(wbytes, G), wbytes);
    if (fp8) {
        const int red = kSkCons * 32 * G * 4 * 4;
        return kFp8RingOffset + (ring > red ? ring : red);
    }
    const int red = kSkCons * 32 * G * 4 * 4;
    return 128 + (ring > red ? ring : red);
}

template <int T, int G, bool XIN>
__device__ __forceinline__ void sk_tile(const Params &p, const Mat &m, int rtile, uint8_t *smem,
                                        int wbytes, int role)
{
    using F = Fmt<T>;
    constexpr int WP = (T == T_Q6K) ? 224 : (T == T_FP4) ? 128 : F::BB;  // weight row pitch
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rank = blockIdx.x, ks = p.ks;
    const int nsb = (p.nb - rank + ks - 1) / ks;  // super-blocks rank, rank + ks, ...
    const int tok0 = p.tok_base + blockIdx.z * kTokChunk;
    const int ntok = min(8 * G, p.N - tok0);
    const int row0 = rtile * kSkRows;
    const int STAGES = p.stages;
    // xin: this rank's x, for all its super-blocks, is staged by the consumer
    // warps into a region after the ring (no staging launch); otherwise each
    // slot carries the stage's staged x, brought by TMA.
    constexpr bool xin = XIN;
    const int sbytes = sk_slot_bytes(T == T_FP8, xin ? 0 : wbytes + 8 * G * kXTok, wbytes);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase, bar_empty = sbase + 8 * kSkStagesMax;
    const uint32_t ring = (T == T_FP8) ? fp8_ring(sbase) : sbase + 128;
    const uint32_t xreg = ring + STAGES * sbytes;
    const uint32_t xbytes = xin ? 0u : (uint32_t)(8 * G * kXTok);
    (void)xreg;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kSkCons);
        }
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        if (T != T_Q6K) prefetch_tmap(&m.tmw1);
        if (T == T_FP4) prefetch_tmap(&m.tms1);
        if (!xin) prefetch_tmap(&p.xm[F::XL]);
    }
    __syncthreads();

    unsigned int err = 0;
    Acc<T, 1, G> A;
    A.zero();
    if (warp == 0) {
        if (lane == 0) {
            // Weights need nothing from earlier kernels: the first stages'
            // weight copies go out before the dependency wait, their x after.
            const int pre = min(STAGES, nsb);
            for (int i = 0; i < pre; ++i) {
                const int sb = rank + i * ks;
                const uint32_t dst = ring + i * sbytes, fb = bar_full + 8 * i;
                mbar_arrive_expect_tx(fb, (T == T_Q6K ? 0u : (uint32_t)sk_wbytes(T)) + xbytes);
                if (T != T_Q6K) tma_load_3d(dst, &m.tmw1, 0, row0, T == T_FP8 ? 2 * sb : sb, fb);
                if (T == T_FP4) tma_load_3d(dst + kSkRows * 128, &m.tms1, 0, row0, sb, fb);
            }
            pdl_wait();
            if (!xin)
                for (int i = 0; i < pre; ++i)
                    tma_load_2d(ring + i * sbytes + wbytes, &p.xm[F::XL], 72 * (rank + i * ks),
                                tok0, bar_full + 8 * i);
            int slot = 0;
            uint32_t par = 0;
            for (int i = STAGES; i < nsb; ++i) {
                if (!mbar_wait(bar_empty + 8 * slot, par)) {
                    err |= ERR_EMPTY_TIMEOUT;
                    break;
                }
                const int sb = rank + i * ks;
                const uint32_t dst = ring + slot * sbytes, fb = bar_full + 8 * slot;
                mbar_arrive_expect_tx(fb, (T == T_Q6K ? 0u : (uint32_t)sk_wbytes(T)) + xbytes);
                if (T != T_Q6K) tma_load_3d(dst, &m.tmw1, 0, row0, T == T_FP8 ? 2 * sb : sb, fb);
                if (T == T_FP4) tma_load_3d(dst + kSkRows * 128, &m.tms1, 0, row0, sb, fb);
                if (!xin) tma_load_2d(dst + wbytes, &p.xm[F::XL], 72 * sb, tok0, fb);
                if (++slot == STAGES) {
                    slot = 0;
                    par ^= 1u;
                }
            }
        }
    } else {
        const int cw = warp - 1;
        const int row_w = row0 + 16 * cw;
        const KSel ksel = k_sel(t);
        // Q6_K: this warp's 16 rows of stage i, each the 16-byte aligned
        // 224-byte superset of its 210-byte block (bytes past the end of the
        // matrix are zero-filled, not read).
        auto q6_issue = [&](int i) {
            const int sb = rank + i * ks;
            const uint32_t dst = ring + (i % STAGES) * sbytes + 16 * cw * 224;
            const uint8_t *end = m.w + m.w_bytes;
#pragma unroll 1
            for (int v = lane; v < 16 * 14; v += 32) {
                const int r = v / 14, c = v - r * 14;
                const int row = row_w + r;
                const uint8_t *src = m.w;
                int nbytes = 0;
                if (row < m.M) {
                    const uint8_t *blk = m.w + (int64_t)row * m.row_bytes + (int64_t)sb * 210;
                    src = (const uint8_t *)((uintptr_t)blk & ~(uintptr_t)15) + 16 * c;
                    const int64_t left = end - src;
                    nbytes = left >= 16 ? 16 : (left > 0 ? (int)left : 0);
                    if (!nbytes) src = m.w;
                }
                cp_async16(dst + r * 224 + 16 * c, src, nbytes);
            }
        };
        // Q6_K weights run STAGES - 1 (2 or 3) stages ahead of this warp; the
        // slot refilled is one this warp has finished with.
        const int q6_ahead = (STAGES >= 4) ? 3 : 2;
        if (T == T_Q6K) {
            for (int i = 0; i < q6_ahead; ++i) {
                if (i < nsb) q6_issue(i);
                cp_async_commit();
            }
        }
        if (T == T_FP8)  // the block scales need nothing from earlier kernels either
            load_fp8_scales(m, p.K, row0, reinterpret_cast<uint32_t *>(smem + 128), threadIdx.x - 32,
                            kSkCons * 32);
        // The weights need nothing from earlier kernels (their first stages
        // are on their way already); x, the residual and y may.
        pdl_wait();
        if constexpr (XIN) {
            // Items (j, n): super-block rank + j ks of token tok0 + n; four
            // loads in flight per warp, then the same staging as everywhere.
            constexpr int XU = 4;
            const int total = nsb * ntok;
            for (int base = cw; base < total; base += XU * kSkCons) {
                uint4 v[XU];
                uint32_t dst[XU];
#pragma unroll
                for (int u = 0; u < XU; ++u) {
                    const int it = base + u * kSkCons;
                    if (it < total) {
                        const int j = it / ntok, n = it - j * ntok;
                        v[u] = __ldg(reinterpret_cast<const uint4 *>(
                            p.x + (int64_t)(tok0 + n) * p.K + 256 * (rank + j * ks) + 8 * lane));
                        dst[u] = (uint32_t)((j * 8 * G + n) * kXTok);
                    }
                }
#pragma unroll
                for (int u = 0; u < XU; ++u) {
                    if (base + u * kSkCons < total) {
                        uint8_t *d = smem + (xreg - sbase) + dst[u];
                        stage_sb(v[u], lane, F::XL == XL_Q4 ? d : nullptr,
                                 F::XL == XL_Q6 ? d : nullptr, F::XL == XL_FP4 ? d : nullptr);
                    }
                }
            }
            bar_sync_named(3, kSkCons * 32);  // the consumer warps only
        }
        if (T == T_FP8) bar_sync_named(4, kSkCons * 32);  // the consumer warps' scale row
        int slot = 0;
        uint32_t par = 0;
#pragma unroll 1
        for (int i = 0; i < nsb; ++i) {
            const int sb = rank + i * ks;
            if (T == T_Q6K) {
                if (i + q6_ahead < nsb) q6_issue(i + q6_ahead);
                cp_async_commit();
                // stage i's group has landed
                if (q6_ahead == 3)
                    cp_async_wait<3>();
                else
                    cp_async_wait<2>();
            }
            if (!mbar_wait(bar_full + 8 * slot, par)) {
                err |= ERR_FULL_TIMEOUT;
                break;
            }
            if (T == T_Q6K) __syncwarp();
            const uint32_t sl = ring + slot * sbytes;
            const uint32_t xsl = xin ? xreg + (uint32_t)(i * 8 * G * kXTok) : sl + wbytes;
            if (T == T_FP4) {
                compute_sb<T, 1, G>(A, sl + 16 * cw * 128, xsl, kXTok, g, t, ntok, m, row_w, sb, ksel,
                                    128, sl + kSkRows * 128 + 16 * cw * 16);
            } else if (T == T_FP8) {
                compute_sb<T, 1, G>(A, sl + 16 * cw * 128, xsl, kXTok, g, t, ntok, m, row_w, sb, ksel,
                                    kSkRows * 128, sbase + 128);
            } else if (T == T_Q6K) {
                compute_sb<T, 1, G>(A, sl + 16 * cw * 224, xsl, kXTok, g, t, ntok, m, row_w, sb, ksel,
                                    224, 0u, sb);
            } else {
                compute_sb<T, 1, G>(A, sl + 16 * cw * WP, xsl, kXTok, g, t, ntok, m, row_w, sb, ksel);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
            if (++slot == STAGES) {
                slot = 0;
                par ^= 1u;
            }
        }
        if (T == T_Q6K) cp_async_wait<0>();
    }
    if (err && p.err) atomicOr(p.err, err);
    __syncthreads();
    reduce_and_store<T, 1, G>(A, reinterpret_cast<float *>(smem + 128), rank, ks,
                              threadIdx.x - 32, kSkCons * 32, warp > 0, p, m, row0, tok0, g, t,
                              role);
}

template <int TSET, int G, bool XIN = false>
__global__ void __launch_bounds__(kSkThreads) qg_sk_kernel(const __grid_constant__ Params p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_trigger();
    int wbytes = 0;
    for (int i = 0; i < p.nmat; ++i) wbytes = max(wbytes, sk_wbytes(p.mat[i].type));
    const int tile = blockIdx.y;
    const int mi = p.swiglu ? (tile & 1) : select_mat(p, tile);
    const Mat &m = p.mat[mi];
    const int rtile = p.swiglu ? (tile >> 1) : tile - m.tile_begin;
    const int role = p.swiglu ? mi : -1;
    if constexpr ((TSET & TS_Q4K) != 0)
        if (m.type == T_Q4K) return sk_tile<T_Q4K, G, XIN>(p, m, rtile, smem, wbytes, role);
    if constexpr ((TSET & TS_Q5K) != 0)
        if (m.type == T_Q5K) return sk_tile<T_Q5K, G, XIN>(p, m, rtile, smem, wbytes, role);
    if constexpr ((TSET & TS_Q6K) != 0)
        if (m.type == T_Q6K) return sk_tile<T_Q6K, G, XIN>(p, m, rtile, smem, wbytes, role);
    if constexpr ((TSET & TS_FP4) != 0)
        if (m.type == T_FP4) return sk_tile<T_FP4, G, XIN>(p, m, rtile, smem, wbytes, role);
    if constexpr ((TSET & TS_FP8) != 0)
        if (m.type == T_FP8) return sk_tile<T_FP8, G, XIN>(p, m, rtile, smem, wbytes, role);
}

}  // namespace qg
