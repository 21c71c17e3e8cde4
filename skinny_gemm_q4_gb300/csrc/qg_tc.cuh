// qg_tc_kernel: the K-quant products of prefill chunks (N >= 33) on the
// 5th-generation tensor core, for Q4_K, Q5_K and Q6_K weights.
//
// For N <= 32 every row must keep its bits whatever N is (TandemLLM
// "Kernels", Row invariance), so those calls stay on the mma.sync kernels;
// past 32 tokens that requirement is lifted and large MMAs pay: one
// tcgen05.mma of M 128 (weight rows) x N up to 128 (tokens) x K 16.  The
// weights are dequantized once per CTA for up to 128 tokens and shared by
// all of them (reflex-llm "docs/performance.md", Path E E5: several warps
// dequantize one A tile that serves every token stripe of the block).
//
// Per CTA: 128 weight rows, up to 128 tokens, one K slice (super-blocks
// rank, rank + ks, ...; the ks ranks of a row tile form a cluster and add
// their partials in rank order).  Warp roles, all running concurrently on a
// pipeline of mbarriers (every wait bounded):
//   * warp 8 (producer): the 128 packed rows of each super-block by one 3-D
//     tensor copy (Q4_K / Q5_K; Q6_K rows are fetched by the row threads) and
//     the staged x of the CTA's tokens by one bulk copy, into separate rings;
//   * warps 0..7 (two warpgroups, one thread per row): dequantize the row's
//     256 weights exactly into four 64-wide chunks of the A operand in tensor
//     memory (Q4_K / Q5_K: WG0 chunks 0, 2, WG1 chunks 1, 3 and the
//     sub-block mins into a small A tile in shared memory; Q6_K: WG0 chunks
//     0, 1, WG1 chunks 2, 3); then fold the previous super-block, each
//     warpgroup half of the tokens:
//       acc = fma(d', D1, acc) [; acc = fma(-dmin', D2, acc)]
//     with that super-block's d (and dmin) kept from its decode;
//   * warp 9 (MMA): per chunk, as soon as it is decoded, 4 MMAs into the
//     super-block's accumulator D1 (double-buffered in tensor memory); then
//     one MMA of the mins against the sub-block sums of x into D2.
// The decode of super-block i + 1 runs during the MMAs of i, and the fold
// of i - 1 after it, so decode, MMA and fold of successive super-blocks
// overlap.
//
// Exactness: Q4_K / Q5_K A = sc * q * 2^-22 and the mins m * 2^-24 (x32 for
// the hi sums) are exact fp16 values; D1, D2 are fp32 sums of exact
// products.  Q6_K A = s * (q - 32) (int8 scale s), exact below 2048 in
// magnitude and rounded once to fp16 above (fp16 has 11 significant bits).
#pragma once

#include "qg_kernels.cuh"

namespace qg {

constexpr int kTcRows = 128;
constexpr int kTcTok = 128;           // tokens per CTA (16 groups of 8)
constexpr int kTcGroups = kTcTok / 8;
constexpr int kTcXBlk = 4096 + 256;   // staged x per (super-block, 8-token group)
constexpr int kTcMinN = 33;           // smallest N served by qg_tc_kernel
constexpr int kTcThreads = 320;       // 2 row warpgroups, producer warp, MMA warp
constexpr int kTcCols = 512;          // tensor-memory columns (one CTA per SM)
constexpr int kTcHdr = 1024;          // barriers and the tensor-memory base
constexpr int kTcMinTile = 4096;      // mins A tile of one super-block: 128 rows x 16 fp16
constexpr int kTcMaxSmem = 226 * 1024;
constexpr int kTcMinSmem = 120 * 1024;  // more than half an SM: never two CTAs per SM
constexpr int kQ6Chunks = 14;         // 16-byte chunks of the aligned window of a Q6_K block

// Ring slot sizes: packed rows of one super-block (Q6_K: 14 chunks x 128
// rows, [chunk][row][16 B]) and the staged x of the CTA's G token groups.
__host__ __device__ constexpr int tc_wslot(int T)
{
    return T == T_Q6K ? kQ6Chunks * kTcRows * 16 : kTcRows * (T == T_Q5K ? 176 : 144);
}
__host__ __device__ constexpr int tc_xslot(int G) { return G * kTcXBlk; }
// Header and (Q4_K / Q5_K) two mins tiles.
__host__ __device__ constexpr int tc_fixed(int T) { return kTcHdr + (T == T_Q6K ? 0 : 2 * kTcMinTile); }
__host__ __device__ inline int tc_smem_bytes(int T, int G, int wstages, int xstages)
{
    const int body = wstages * tc_wslot(T) + xstages * tc_xslot(G);
    // overlay after the loop: rank partials of the cluster reduction, then the
    // output tile of the transposed stores
    const int red = (G + 7) * 4096 + 8 * G * kTcRows * 4;
    const int s = tc_fixed(T) + (body > red ? body : red);
    return s > kTcMinSmem ? s : kTcMinSmem;
}
// Staged x of qg_tc_kernel: [128-token chunk][super-block][16 groups x
// kTcXBlk, in two halves (see stage_tc4)].
__host__ __device__ inline int64_t tc_chunk_bytes(int nb) { return (int64_t)nb * kTcGroups * kTcXBlk; }

// ---------------------------------------------------------------------------
// x of one (token, super-block) into the tensor-core layout of the super-
// block's 128-token block `sbb` (16 groups of 8 tokens; token row `nrow` =
// token % 8 of group g), split in two halves so that the MMAs of chunks 0-1
// can start before the rest has landed:
//   half 0 at 0:      [group][2048 B]: k-step s = 0..7, core j (2): 8 token
//                     rows x 16 bytes at (2 s + j) * 128 + 16 nrow;
//   half 1 at 32768:  [group][2304 B]: k-steps 8..15 likewise at
//                     (2 (s - 8) + j) * 128, then at 2048 core 0: fp16 hi of
//                     the 8 sub-block sums, core 1: the lo parts.
// The row of k-step s, core j holds, for the 4-groups A = 16 c + w and A + 8
// (c = s / 4, w = 2 (s % 4) + j), the values (a0, a2, a1, a3, b0, b2, b1,
// b3) -- the order in which the decoders lay out word w of chunk c.
// Lane l holds x[256 sb + 8 l .. + 8].  Sub-block sums as in stage_sb
// (hi = fp16(S * 2^-5), lo = fp16(S - 32 hi)).
// ---------------------------------------------------------------------------
constexpr int kTcXHalf0 = 2048, kTcXHalf1 = 2304;  // bytes per group in each half
constexpr int kTcXHalf1Off = kTcGroups * kTcXHalf0;
__device__ __forceinline__ void stage_tc4(uint4 v, int lane, uint8_t *sbb, int g, int nrow)
{
    uint4 w;
    w.x = __shfl_down_sync(0xffffffffu, v.x, 4);
    w.y = __shfl_down_sync(0xffffffffu, v.y, 4);
    w.z = __shfl_down_sync(0xffffffffu, v.z, 4);
    w.w = __shfl_down_sync(0xffffffffu, v.w, 4);
    uint8_t *h1 = sbb + kTcXHalf1Off + g * kTcXHalf1;
    if ((lane & 7) < 4) {
        const int s = 4 * (lane >> 3) + (lane & 7);
        uint4 o0, o1;
        o0.x = __byte_perm(v.x, v.y, 0x5410);
        o0.y = __byte_perm(v.x, v.y, 0x7632);
        o0.z = __byte_perm(w.x, w.y, 0x5410);
        o0.w = __byte_perm(w.x, w.y, 0x7632);
        o1.x = __byte_perm(v.z, v.w, 0x5410);
        o1.y = __byte_perm(v.z, v.w, 0x7632);
        o1.z = __byte_perm(w.z, w.w, 0x5410);
        o1.w = __byte_perm(w.z, w.w, 0x7632);
        uint8_t *c0 = (s < 8) ? sbb + g * kTcXHalf0 + (2 * s) * 128 : h1 + (2 * (s - 8)) * 128;
        *reinterpret_cast<uint4 *>(c0 + 16 * nrow) = o0;
        *reinterpret_cast<uint4 *>(c0 + 128 + 16 * nrow) = o1;
    }
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    float sm = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        sm = __fadd_rn(sm, __half2float(__ushort_as_half((unsigned short)(w4[i] & 0xffffu))));
        sm = __fadd_rn(sm, __half2float(__ushort_as_half((unsigned short)(w4[i] >> 16))));
    }
    sm = __fadd_rn(sm, __shfl_xor_sync(0xffffffffu, sm, 1));
    sm = __fadd_rn(sm, __shfl_xor_sync(0xffffffffu, sm, 2));
    if ((lane & 3) == 0) {
        const int sbk = lane >> 2;
        const __half hi = __float2half_rn(__fmul_rn(sm, 0.03125f));
        const __half lo = __float2half_rn(__fsub_rn(sm, __fmul_rn(__half2float(hi), 32.0f)));
        *reinterpret_cast<__half *>(h1 + 2048 + 16 * nrow + 2 * sbk) = hi;
        *reinterpret_cast<__half *>(h1 + 2048 + 128 + 16 * nrow + 2 * sbk) = lo;
    }
}

// ---------------------------------------------------------------------------
// Decoders.  Chunk c of a super-block holds k = 64 c .. 64 c + 63; word w
// (0..7) of the chunk fills the 4 tensor-memory columns 4 w .. 4 w + 3 of the
// chunk with the 8 fp16 values of k = 64 c + 4 w + (0, 2, 1, 3) and
// 64 c + 32 + 4 w + (0, 2, 1, 3): the order stage_tc4 gives x.
// ---------------------------------------------------------------------------
// Q4_K / Q5_K row at ra (its 144- / 176-byte block in shared memory).
template <int T>
__device__ __forceinline__ void tc_chunk_kq(uint32_t ra, int c, uint32_t (&a)[32])
{
    const uint4 h = lds128(ra);
    // 6-bit scales of sub-blocks 2c (low nibbles) and 2c + 1 (high nibbles)
    const uint32_t sw = (c < 2) ? (h.y & 0x3f3f3f3fu)
                                : ((h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u));
    const uint32_t b0 = (uint32_t)(2 * c) & 3u, b1 = (uint32_t)(2 * c + 1) & 3u;
    const uint32_t slo = hsub2(__byte_perm(sw, 0x6C6Cu, 0x4040u | b0 | (b0 << 8)), 0x6C006C00u);
    const uint32_t shi =
        (T == T_Q4K) ? hsub2(__byte_perm(sw, 0x5C5Cu, 0x4040u | b1 | (b1 << 8)), 0x5C005C00u)
                     : hsub2(__byte_perm(sw, 0x6C6Cu, 0x4040u | b1 | (b1 << 8)), 0x6C006C00u);
    const uint32_t qsa = ra + ((T == T_Q4K) ? 16u : 48u) + 32u * (uint32_t)c;
    const uint4 qa = lds128(qsa), qb = lds128(qsa + 16);
    const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    uint32_t hq[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (T == T_Q5K) {
        const uint4 ha = lds128(ra + 16), hb = lds128(ra + 32);
        hq[0] = ha.x, hq[1] = ha.y, hq[2] = ha.z, hq[3] = ha.w;
        hq[4] = hb.x, hq[5] = hb.y, hq[6] = hb.z, hq[7] = hb.w;
    }
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        kq_decode<T>(q[w], hq[w], c, 0, slo, shi, a[4 * w + 0], a[4 * w + 1]);
        kq_decode<T>(q[w], hq[w], c, 1, slo, shi, a[4 * w + 2], a[4 * w + 3]);
    }
}

// Mins of a Q4_K / Q5_K row: (m_2i, m_2i+1) * 2^-24 as fp16 subnormals;
// hi[] carries the factor 32 (against the hi sums), lo[] not.
__device__ __forceinline__ void tc_mins_kq(uint32_t ra, uint4 &hi, uint4 &lo)
{
    const uint4 h = lds128(ra);
    const uint32_t mn03 = h.z & 0x3f3f3f3fu;
    const uint32_t mn47 = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
    lo.x = __byte_perm(mn03, 0u, 0x4140u);
    lo.y = __byte_perm(mn03, 0u, 0x4342u);
    lo.z = __byte_perm(mn47, 0u, 0x4140u);
    lo.w = __byte_perm(mn47, 0u, 0x4342u);
    hi.x = hmul2(lo.x, 0x50005000u);  // * 32
    hi.y = hmul2(lo.y, 0x50005000u);
    hi.z = hmul2(lo.z, 0x50005000u);
    hi.w = hmul2(lo.w, 0x50005000u);
}

// Words o[0..N) = bytes off + 4 i .. + 3 of the little-endian byte stream
// held in v[0..N+4) (off even, 0..14): a shift by 2 and 1 words chosen by
// bits 3 and 2 of off, then a 16-bit funnel shift for bit 1.
template <int N>
__device__ __forceinline__ void tc_realign(const uint32_t (&v)[N + 4], uint32_t off,
                                           uint32_t (&o)[N])
{
    uint32_t t[N + 2];
#pragma unroll
    for (int i = 0; i < N + 2; ++i) t[i] = (off & 8u) ? v[i + 2] : v[i];
    uint32_t u[N + 1];
#pragma unroll
    for (int i = 0; i < N + 1; ++i) u[i] = (off & 4u) ? t[i + 1] : t[i];
    const uint32_t sh = (off & 2u) ? 16u : 0u;
#pragma unroll
    for (int i = 0; i < N; ++i) o[i] = __funnelshift_r(u[i], u[i + 1], sh);
}

// The Q6_K data of half h (chunks 2h, 2h + 1) of one row from its window
// in the [chunk][row] slot (row address rs = slot + 16 row; the block starts
// `off` bytes into the window): ql bytes 64 h .. + 63, qh bytes 32 h .. + 31
// and the 8 int8 scales 8 h .. + 7.
struct Q6Half {
    uint32_t ql[16], qh[8], sc[2];
};
__device__ __forceinline__ void tc_q6_load(uint32_t rs, int h, uint32_t off, Q6Half &d)
{
    {
        uint32_t v[20];
#pragma unroll
        for (int j = 0; j < 5; ++j) {
            const uint4 x = lds128(rs + (uint32_t)(4 * h + j) * (kTcRows * 16));
            v[4 * j] = x.x, v[4 * j + 1] = x.y, v[4 * j + 2] = x.z, v[4 * j + 3] = x.w;
        }
        tc_realign<16>(v, off, d.ql);
    }
    {
        // qh of half h: window bytes 128 + 32 h + off ..: chunks 8 + 2h .. 10 + 2h
        uint32_t v[12];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const uint4 x = lds128(rs + (uint32_t)(8 + 2 * h + j) * (kTcRows * 16));
            v[4 * j] = x.x, v[4 * j + 1] = x.y, v[4 * j + 2] = x.z, v[4 * j + 3] = x.w;
        }
        tc_realign<8>(v, off, d.qh);
    }
    {
        // scales 8h .. 8h + 7: window bytes 192 + 8 h + off ..: chunks 12, 13
        // (words 2h .. of chunk 12 onwards)
        uint32_t v[8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint4 x = lds128(rs + (uint32_t)(12 + j) * (kTcRows * 16));
            v[4 * j] = x.x, v[4 * j + 1] = x.y, v[4 * j + 2] = x.z, v[4 * j + 3] = x.w;
        }
        uint32_t w6[6];
#pragma unroll
        for (int i = 0; i < 6; ++i) w6[i] = h ? v[i + 2] : v[i];
        tc_realign<2>(w6, off, d.sc);
    }
}

// Chunk c = 2 h + cc of a Q6_K row: A = s * (q - 32), q the 6-bit code of
// ql nibble cc and the qh bit pair (see the block layout: qh byte l holds
// the high bits of k = 128 h + l + 32 j in bits 2 j, 2 j + 1).
__device__ __forceinline__ void tc_chunk_q6(const Q6Half &d, int cc, uint32_t (&a)[32])
{
    // int8 scales of sub-blocks 4 c .. 4 c + 3 as fp16x2 broadcasts:
    // (0x6400 | (s ^ 0x80)) - (1024 + 128) = s
    const uint32_t sx = (cc ? d.sc[1] : d.sc[0]) ^ 0x80808080u;
    uint32_t s[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        s[j] = hsub2(__byte_perm(sx, 0x6464u, 0x4040u | (uint32_t)j | ((uint32_t)j << 8)),
                     0x64806480u);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t la = cc ? (d.ql[w] >> 4) : d.ql[w];
        const uint32_t lb = cc ? (d.ql[w + 8] >> 4) : d.ql[w + 8];
        const uint32_t ha = cc ? d.qh[w] : (d.qh[w] << 4);        // bits 4cc .. -> 4, 5
        const uint32_t hb = cc ? (d.qh[w] >> 2) : (d.qh[w] << 2);  // bits 4cc + 2 .. -> 4, 5
        const uint32_t va = (la & 0x0f0f0f0fu) | (ha & 0x30303030u);
        const uint32_t vb = (lb & 0x0f0f0f0fu) | (hb & 0x30303030u);
        const uint32_t sa = s[w >> 2], sb = s[2 + (w >> 2)];
        a[4 * w + 0] = hmul2(hsub2(__byte_perm(va, 0x6464u, 0x5240u), 0x64206420u), sa);
        a[4 * w + 1] = hmul2(hsub2(__byte_perm(va, 0x6464u, 0x5341u), 0x64206420u), sa);
        a[4 * w + 2] = hmul2(hsub2(__byte_perm(vb, 0x6464u, 0x5240u), 0x64206420u), sb);
        a[4 * w + 3] = hmul2(hsub2(__byte_perm(vb, 0x6464u, 0x5341u), 0x64206420u), sb);
    }
}

// Epilogue of one output element: residual (fp32 add before the single
// rounding), fp16 RN or fp32 store.  The output description is copied into
// registers first (TcOut), so that the stores need no reload of the kernel
// parameters they could otherwise alias.
struct TcOut {
    void *y;
    const __half *res;
    int M, N, f32;
};
__device__ __forceinline__ TcOut tc_out(const Params &p, const Mat &m)
{
    TcOut o;
    o.y = m.y;
    o.res = m.res;
    o.M = m.M;
    o.N = p.N;
    o.f32 = p.out_f32;
    return o;
}
__device__ __forceinline__ void tc_store(const TcOut &o, int row, int tok, float val)
{
    if (row >= o.M || tok >= o.N) return;
    const int64_t i = (int64_t)tok * o.M + row;
    if (o.res) val = __fadd_rn(__half2float(__ldg(o.res + i)), val);
    if (o.f32)
        reinterpret_cast<float *>(o.y)[i] = val;
    else
        reinterpret_cast<__half *>(o.y)[i] = __float2half_rn(val);
}
// Rows row .. row + 3 of token tok: one 8-byte (fp16) or 16-byte (fp32)
// store when all four rows exist and the addresses are aligned.
__device__ __forceinline__ void tc_store4(const TcOut &o, int row, int tok, float4 v)
{
    if (tok >= o.N || row >= o.M) return;
    const int64_t i = (int64_t)tok * o.M + row;
    const uintptr_t ya = o.f32 ? (uintptr_t)(reinterpret_cast<float *>(o.y) + i)
                               : (uintptr_t)(reinterpret_cast<__half *>(o.y) + i);
    const bool vec = row + 3 < o.M && (ya & (o.f32 ? 15u : 7u)) == 0 &&
                     (!o.res || ((uintptr_t)(o.res + i) & 7u) == 0);
    if (!vec) {
        tc_store(o, row, tok, v.x);
        tc_store(o, row + 1, tok, v.y);
        tc_store(o, row + 2, tok, v.z);
        tc_store(o, row + 3, tok, v.w);
        return;
    }
    if (o.res) {
        const uint2 rr = __ldg(reinterpret_cast<const uint2 *>(o.res + i));
        const __half2 r01 = *reinterpret_cast<const __half2 *>(&rr.x);
        const __half2 r23 = *reinterpret_cast<const __half2 *>(&rr.y);
        v.x = __fadd_rn(__low2float(r01), v.x);
        v.y = __fadd_rn(__high2float(r01), v.y);
        v.z = __fadd_rn(__low2float(r23), v.z);
        v.w = __fadd_rn(__high2float(r23), v.w);
    }
    if (o.f32) {
        *reinterpret_cast<float4 *>(ya) = v;
    } else {
        const __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t *>(&h01);
        u.y = *reinterpret_cast<const uint32_t *>(&h23);
        *reinterpret_cast<uint2 *>(ya) = u;
    }
}
// The row threads' results through a shared-memory tile [token][128 rows]
// (fp32 at `tile`): each thread writes its row's values, then the tile goes
// out four rows per thread (one 256-byte token row per warp store).
// nt: tokens in the tile, tok0: the first one.
__device__ __forceinline__ void tc_tile_out(const TcOut &o, const float *tile, int nt, int row0,
                                            int tok0, int tid, int nthr)
{
    for (int q = tid; q < nt * (kTcRows / 4); q += nthr) {
        const int t = q / (kTcRows / 4), c = q % (kTcRows / 4);
        const float4 v = *reinterpret_cast<const float4 *>(tile + t * kTcRows + 4 * c);
        tc_store4(o, row0 + 4 * c, tok0 + t, v);
    }
}

// ---------------------------------------------------------------------------
// Shared memory: [barriers, tensor-memory base (1 KB) | Q4_K / Q5_K: two
// mins tiles (2 x 4 KB) | weight ring (p.stages slots) | x ring (p.xstages
// slots)]; after the loop the rank partials [8 G][128] overlay the rings.
// Tensor memory (512 columns): A chunks 0..127 (chunk c at 32 c), D1 buffers
// at 128 + 8 G b (b = 0, 1), D2 at 128 + 16 G (single: the mins MMA of
// super-block i waits until the fold of i - 1 has read it).
// ---------------------------------------------------------------------------
template <int T, int G>
__device__ __forceinline__ void tc_body(const Params &p, const Mat &m, const int rtile)
{
    static_assert(G % 2 == 0 && G >= 2 && G <= kTcGroups, "MMA N = 8 G must be a multiple of 16");
    constexpr bool KQ = (T != T_Q6K);  // Q4_K / Q5_K: the mins term
    constexpr int WSLOT = tc_wslot(T);
    constexpr uint32_t XSLOT = (uint32_t)tc_xslot(G);
    constexpr int BB = Fmt<T>::BB;
    constexpr int G0 = (G + 1) / 2;  // token groups folded by WG0; WG1 folds the rest
    constexpr uint32_t kIdesc = tc_idesc_f16(8 * G);
    constexpr uint32_t kD1 = 128, kD2 = 128 + 16 * G;

    extern __shared__ __align__(1024) uint8_t smem_tc[];
    uint8_t *const smem = smem_tc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = blockIdx.x, ks = p.ks;
    const int nsb = (p.nb - rank + ks - 1) / ks;  // super-blocks rank, rank + ks, ...
    // token tile blockIdx.z: 8 G tokens, groups goff .. goff + G - 1 of the
    // staged 128-token chunk zch
    const int tz = blockIdx.z * 8 * G;
    const int zch = tz / kTcTok, goff = (tz % kTcTok) / 8;
    const int tok0 = p.tok_base + tz;
    const int ntok = min(8 * G, p.N - tok0);
    const int row0 = rtile * kTcRows;
    const int WS = p.stages, XS = p.xstages;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t b_wfull = sbase, b_wempty = sbase + 32, b_xfull = sbase + 64,
                   b_xempty = sbase + 96, b_afull = sbase + 128, b_aempty = sbase + 160,
                   b_dfull = sbase + 192, b_dfree = sbase + 208, b_xfull2 = sbase + 224;
    const uint32_t amin = sbase + kTcHdr;  // Q4_K / Q5_K mins tiles [2][4096]
    const uint32_t wring = sbase + tc_fixed(T);
    const uint32_t xring = wring + (uint32_t)(WS * WSLOT);

    if (threadIdx.x == 0) {
        for (int s = 0; s < WS; ++s) {
            mbar_init(b_wfull + 8 * s, KQ ? 1 : 256);  // Q6_K: every decoder thread's copies
            mbar_init(b_wempty + 8 * s, 8);            // the 8 decoder warps
        }
        for (int s = 0; s < XS; ++s) {
            mbar_init(b_xfull + 8 * s, 1);   // x half 0 (k-steps 0..7)
            mbar_init(b_xfull2 + 8 * s, 1);  // x half 1 (k-steps 8..15, sub-block sums)
            mbar_init(b_xempty + 8 * s, 1);
        }
        for (int c = 0; c < 4; ++c) {  // per A chunk (decoded by one warpgroup)
            mbar_init(b_afull + 8 * c, kTcRows);
            mbar_init(b_aempty + 8 * c, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_dfull + 8 * b, 1);
            mbar_init(b_dfree + 8 * b, 8);  // the 8 row warps
        }
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(sbase + 256, kTcCols);
    if (KQ && warp == 8 && lane == 0) prefetch_tmap(&m.tmw1);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(smem + 256);

    unsigned int err = 0;
    float acc[G0][8];  // row threads: WG0 groups 0..G0-1, WG1 groups G0..G-1
#pragma unroll
    for (int g = 0; g < G0; ++g)
#pragma unroll
        for (int n = 0; n < 8; ++n) acc[g][n] = 0.0f;

    if (warp == 8) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint8_t *xs =
                p.xs[XL_TC4] + (int64_t)zch * p.xs_tok_stride;
            auto load_w = [&](int i) {
                const uint32_t fb = b_wfull + 8 * (i % WS);
                mbar_arrive_expect_tx(fb, (uint32_t)WSLOT);
                tma_load_3d(wring + (i % WS) * WSLOT, &m.tmw1, 0, row0, rank + i * ks, fb);
            };
            const int wpre = KQ ? min(WS, nsb) : 0, xpre = min(XS, nsb);
            for (int i = 0; i < wpre; ++i) load_w(i);  // weights need nothing earlier
            pdl_wait();  // the staged x is written by the kernel just before
            auto load_x = [&](int i) {
                const int xsl = i % XS;
                const uint8_t *src = xs + (int64_t)(rank + i * ks) * (kTcGroups * kTcXBlk);
                const uint32_t dst = xring + xsl * XSLOT;
                mbar_arrive_expect_tx(b_xfull + 8 * xsl, (uint32_t)(G * kTcXHalf0));
                bulk_g2s(dst, src + goff * kTcXHalf0, (uint32_t)(G * kTcXHalf0), b_xfull + 8 * xsl);
                mbar_arrive_expect_tx(b_xfull2 + 8 * xsl, (uint32_t)(G * kTcXHalf1));
                bulk_g2s(dst + G * kTcXHalf0, src + kTcXHalf1Off + goff * kTcXHalf1,
                         (uint32_t)(G * kTcXHalf1), b_xfull2 + 8 * xsl);
            };
            for (int i = 0; i < xpre; ++i) load_x(i);
            // Refills in the order the slots free up: the decoders finish
            // super-block i before its MMAs complete.  Blocking waits
            // (try_wait suspends), so this warp takes no issue slots from the
            // decoders while it waits.
            for (int i = 0; i < nsb; ++i) {
                if (KQ && i + WS < nsb) {
                    if (!mbar_wait(b_wempty + 8 * (i % WS), (uint32_t)((i / WS) & 1))) {
                        err |= ERR_EMPTY_TIMEOUT;
                        break;
                    }
                    load_w(i + WS);
                }
                if (i + XS < nsb) {
                    if (!mbar_wait(b_xempty + 8 * (i % XS), (uint32_t)((i / XS) & 1))) {
                        err |= ERR_EMPTY_TIMEOUT;
                        break;
                    }
                    load_x(i + XS);
                }
            }
        }
    } else if (warp == 9) {
        // ---------------- MMA issue ----------------
        // One thread.  The tensor core idles while this thread is not issuing,
        // so the phase needed next is probed inside each batch of 4 MMAs
        // (tc_mma4_probe) and only waited for (try_wait, suspending: no issue
        // slots taken from the decoders) when not yet complete.
        int issued = 0;
        if (lane == 0) {
            bool ready = false;  // x half 0, D1[b] and chunk 0, probed in the previous batch
            for (int i = 0; i < nsb; ++i) {
                const int b = i & 1, xsl = i % XS;
                const uint32_t px = (uint32_t)((i / XS) & 1), pa = (uint32_t)(i & 1);
                // x half 0 landed; D1[b] read back by the folds of super-block i - 2;
                // chunk 0 decoded
                if (!ready &&
                    (!mbar_wait(b_xfull + 8 * xsl, px) ||
                     (i >= 2 && !mbar_wait(b_dfree + 8 * b, (uint32_t)(((i >> 1) - 1) & 1))) ||
                     !mbar_wait(b_afull, pa))) {
                    err |= ERR_FULL_TIMEOUT;
                    break;
                }
                const uint32_t xb = xring + xsl * XSLOT, xb1 = xb + G * kTcXHalf0;
                const uint32_t d1 = tbase + kD1 + 8 * G * b;
                bool ok = true;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    tc_fence_after();
                    // next: chunk c + 1 (and x half 1 before chunk 2); after
                    // chunk 3: the folds of i - 1 (D2, next D1) and the next
                    // super-block's x half 0
                    uint32_t q1 = b_afull + 8 * (c + 1), p1 = pa, q2 = q1, p2 = pa;
                    if (c == 1) q2 = b_xfull2 + 8 * xsl, p2 = px;
                    if (c == 3) {
                        const int ni = (i + 1 < nsb) ? i + 1 : i;
                        q1 = (i >= 1) ? b_dfree + 8 * ((i - 1) & 1) : b_xfull + 8 * xsl;
                        p1 = (i >= 1) ? (uint32_t)(((i - 1) >> 1) & 1) : px;
                        q2 = b_xfull + 8 * (ni % XS), p2 = (uint32_t)((ni / XS) & 1);
                    }
                    const uint64_t bd = (c < 2) ? smem_desc2(xb + 1024 * c, 128, kTcXHalf0)
                                                : smem_desc2(xb1 + 1024 * (c - 2), 128, kTcXHalf1);
                    const uint32_t r = tc_mma4_probe(d1, tbase + 32 * c, bd, kIdesc, c ? 1u : 0u,
                                                     q1, p1, q2, p2);
                    tc_commit(b_aempty + 8 * c);
                    if (c < 3 && !r && (!mbar_wait(q1, p1) || (c == 1 && !mbar_wait(q2, p2)))) {
                        ok = false;
                        break;
                    }
                    if (c == 3) ready = r;
                }
                // D2 is single-buffered: the folds of super-block i - 1 must
                // have read it.
                if (ok && !ready && KQ && i >= 1 &&
                    !mbar_wait(b_dfree + 8 * ((i - 1) & 1), (uint32_t)(((i - 1) >> 1) & 1)))
                    ok = false;
                if (!ok) {
                    err |= ERR_FULL_TIMEOUT;
                    break;
                }
                if (KQ)
                    tc_mma_ss(tbase + kD2, smem_desc2(amin + kTcMinTile * b, 128, 256),
                              smem_desc2(xb1 + 2048, 128, kTcXHalf1), kIdesc, 0u);
                tc_commit(b_dfull + 8 * b);
                tc_commit(b_xempty + 8 * xsl);
                ++issued;
                // the probe after chunk 3 covered x half 0 and the folds, not
                // the next chunk 0: wait for that one at the top
                if (ready && i + 1 < nsb && !mbar_wait(b_afull, (uint32_t)((i + 1) & 1))) {
                    err |= ERR_FULL_TIMEOUT;
                    break;
                }
            }
            // Nothing of this CTA may still run on the tensor core when its
            // tensor memory is released (matters only after a timeout).
            if (issued > 0)
                mbar_wait_spin(b_dfull + 8 * ((issued - 1) & 1), (uint32_t)(((issued - 1) >> 1) & 1));
        }
    } else {
        // ---------------- row threads: WG0 = warps 0..3, WG1 = 4..7 ----------------
        // Per super-block i: decode this WG's two chunks of i (WG1 also the
        // mins), then fold super-block i - 1 into this WG's token groups.
        const int wg = warp >> 2;
        const int r = threadIdx.x & 127;  // row within the tile; tensor-memory lane
        const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
        const int row = row0 + r;
        const bool rvalid = row < m.M;
        const int gbeg = wg ? G0 : 0, gcnt = wg ? G - G0 : G0;
        // Q6_K: this thread's 16-byte chunks (WG0 0..6, WG1 7..13) of its row's
        // aligned 224-byte window; bytes past the end of the matrix are
        // zero-filled, rows past M fetch nothing.
        auto q6_issue = [&](int i) {
            const int slot = i % WS;
            const uint32_t dst = wring + slot * WSLOT + 16 * r;
            const uint8_t *end = m.w + m.w_bytes;
            const uint8_t *base = m.w;
            if (rvalid)
                base = (const uint8_t *)((uintptr_t)(m.w + (int64_t)row * m.row_bytes +
                                                     (int64_t)(rank + i * ks) * 210) &
                                         ~(uintptr_t)15);
#pragma unroll
            for (int c = 7 * wg; c < 7 * wg + 7; ++c) {
                const uint8_t *src = base + 16 * c;
                const int64_t left = end - src;
                int nbytes = rvalid ? (left >= 16 ? 16 : (left > 0 ? (int)left : 0)) : 0;
                if (!nbytes) src = m.w;
                cp_async16(dst + (uint32_t)c * (kTcRows * 16), src, nbytes);
            }
            cp_async_mbar_arrive(b_wfull + 8 * slot);
        };
        // Fold super-block j (its D buffer) into this thread's token groups;
        // dw: its d (and dmin) as read by this thread's decode of j.
        auto fold = [&](int j, uint32_t dw) -> bool {
            const int b = j & 1;
            if (!mbar_wait(b_dfull + 8 * b, (uint32_t)((j >> 1) & 1))) return false;
            tc_fence_after();
            const float d = __half2float(__ushort_as_half((unsigned short)(dw & 0xffffu)));
            const float dd = KQ ? d * 4194304.0f : d;
            const float dm = -__half2float(__ushort_as_half((unsigned short)(dw >> 16))) * 16777216.0f;
            const uint32_t c1 = tl + kD1 + 8 * G * b + 8 * gbeg, c2 = tl + kD2 + 8 * gbeg;
#pragma unroll
            for (int g = 0; g < G0; g += 4) {
                if (g >= gcnt || 8 * (gbeg + g) >= ntok) break;
                if (g + 4 <= G0 && g + 4 <= gcnt) {
                    // four groups (32 columns) per load, one wait
                    uint32_t v1[32], v2[32];
                    tmem_ld32(c1 + 8 * g, v1);
                    if (KQ) tmem_ld32(c2 + 8 * g, v2);
                    tc_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (g + q >= G0) break;
#pragma unroll
                        for (int n = 0; n < 8; ++n) {
                            acc[g + q][n] = __fmaf_rn(dd, __uint_as_float(v1[8 * q + n]), acc[g + q][n]);
                            if (KQ)
                                acc[g + q][n] =
                                    __fmaf_rn(dm, __uint_as_float(v2[8 * q + n]), acc[g + q][n]);
                        }
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int gg = g + q;
                        if (gg >= G0 || gg >= gcnt || 8 * (gbeg + gg) >= ntok) break;
                        uint32_t v1[8], v2[8];
                        tmem_ld8(c1 + 8 * gg, v1);
                        if (KQ) tmem_ld8(c2 + 8 * gg, v2);
                        tc_wait_ld();
#pragma unroll
                        for (int n = 0; n < 8; ++n) {
                            acc[gg][n] = __fmaf_rn(dd, __uint_as_float(v1[n]), acc[gg][n]);
                            if (KQ) acc[gg][n] = __fmaf_rn(dm, __uint_as_float(v2[n]), acc[gg][n]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_dfree + 8 * b);
            return true;
        };
        int q6_next = 0;
        if (!KQ)
            for (; q6_next < WS - 1 && q6_next < nsb; ++q6_next) q6_issue(q6_next);
        uint32_t dprev = 0;
        bool ok = true;
        for (int i = 0; i < nsb && ok; ++i) {
            const int slot = i % WS;
            if (!KQ && q6_next < nsb) {
                // the slot refilled was last used by super-block q6_next - WS
                const int j = q6_next;
                if (j >= WS && !mbar_wait(b_wempty + 8 * (j % WS), (uint32_t)(((j / WS) - 1) & 1))) {
                    ok = false;
                    break;
                }
                q6_issue(j);
                ++q6_next;
            }
            if (!mbar_wait(b_wfull + 8 * slot, (uint32_t)((i / WS) & 1))) {
                ok = false;
                break;
            }
            const uint32_t ws = wring + slot * WSLOT;
            Q6Half q6;
            uint32_t dcur;  // d | dmin << 16 (Q6_K: d) of this row in super-block i
            if (KQ) {
                dcur = lds32(ws + (uint32_t)(r * BB));
            } else {
                const uint32_t off =
                    rvalid ? (uint32_t)((uintptr_t)(m.w + (int64_t)row * m.row_bytes +
                                                    (int64_t)(rank + i * ks) * 210) &
                                        15)
                           : 0u;
                tc_q6_load(ws + 16 * r, wg, off, q6);
                // d: window bytes 208 + off, 209 + off (chunk 13)
                dcur = lds16(ws + 13u * (kTcRows * 16) + 16 * r + off);
            }
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                // K-quants: WG0 chunks 0, 2 and WG1 chunks 1, 3 (interleaved, so a
                // chunk's decode has three chunks of MMAs to hide behind); Q6_K:
                // WG h the two chunks of block half h (one realigned load)
                const int c = KQ ? wg + 2 * cc : 2 * wg + cc;
                // chunk c of super-block i - 1 must have left the tensor core
                if (i > 0 && !mbar_wait(b_aempty + 8 * c, (uint32_t)((i - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t a[32];
                if (KQ)
                    tc_chunk_kq<T>(ws + (uint32_t)(r * BB), c, a);
                else
                    tc_chunk_q6(q6, cc, a);
                tmem_st32(tl + 32 * c, a);
                if (KQ && c == 3) {
                    // mins tile of this super-block: core (k-core kc, rows 8 g..)
                    // at 256 g + 128 kc + 16 (r % 8); free since super-block
                    // i - 2's MMAs completed before chunk 3 of i - 1 did
                    uint4 hi, lo;
                    tc_mins_kq(ws + (uint32_t)(r * BB), hi, lo);
                    const uint32_t t0 = amin + kTcMinTile * (i & 1) + 256 * (r >> 3) + 16 * (r & 7);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(t0), "r"(hi.x),
                                 "r"(hi.y), "r"(hi.z), "r"(hi.w)
                                 : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(t0 + 128),
                                 "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w)
                                 : "memory");
                    fence_proxy_async_smem();
                }
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(b_afull + 8 * c);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(b_wempty + 8 * slot);
            if (i > 0 && !fold(i - 1, dprev)) {
                ok = false;
                break;
            }
            dprev = dcur;
        }
        if (ok && nsb > 0 && !fold(nsb - 1, dprev)) ok = false;
        if (!KQ) cp_async_wait<0>();
        if (!ok) err |= ERR_FULL_TIMEOUT;
    }
    if (err && p.err) atomicOr(p.err, err);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tbase, kTcCols);
    pdl_wait();  // y and the residual belong to earlier kernels too

    // Rank partials through distributed shared memory, added in rank order.
    // Rank q owns token groups [q gpr, (q + 1) gpr); every rank pushes its
    // partials of those groups into rank q's shared memory (slot [source
    // rank][group][half][row] of 4 floats), then each owner adds the ks
    // slots in rank order and stores.  The first cluster barrier makes sure
    // no rank still uses its rings; the second publishes the pushes.
    float *red = reinterpret_cast<float *>(smem + tc_fixed(T));
    float *otile = reinterpret_cast<float *>(smem + tc_fixed(T) + (G + 7) * 4096);
    const TcOut out = tc_out(p, m);
    const bool foldt = warp < 8;
    const int r = threadIdx.x & 127;
    const int wgr = warp >> 2;
    const int gbeg = wgr ? G0 : 0, gcnt = wgr ? G - G0 : G0;
    if (ks > 1) {
        const int gpr = (G + ks - 1) / ks;
        const uint32_t rbase = smem_u32(red);
        cluster_sync();
        if (foldt) {
#pragma unroll
            for (int g = 0; g < G0; ++g) {
                if (g >= gcnt) break;
                const int gg = gbeg + g, q = gg / gpr, gl = gg - q * gpr;
                const uint32_t dst =
                    map_shared_rank(rbase + (uint32_t)(((rank * gpr + gl) * 2 * kTcRows + r) * 16),
                                    (uint32_t)q);
                st_dsmem_v4(dst, acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
                st_dsmem_v4(dst + kTcRows * 16, acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
            }
        }
        cluster_sync();
        if (!foldt) return;
        const int owned = min(G, (rank + 1) * gpr) - rank * gpr;
        for (int gl = wgr; gl < owned; gl += 2) {
            float v[8];
#pragma unroll 1
            for (int q = 0; q < ks; ++q) {
                const uint32_t a = rbase + (uint32_t)(((q * gpr + gl) * 2 * kTcRows + r) * 16);
                const uint4 lo = lds128(a), hi = lds128(a + kTcRows * 16);
                const float w[8] = {__uint_as_float(lo.x), __uint_as_float(lo.y),
                                    __uint_as_float(lo.z), __uint_as_float(lo.w),
                                    __uint_as_float(hi.x), __uint_as_float(hi.y),
                                    __uint_as_float(hi.z), __uint_as_float(hi.w)};
#pragma unroll
                for (int n = 0; n < 8; ++n) v[n] = q ? __fadd_rn(v[n], w[n]) : w[n];
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) otile[(8 * gl + n) * kTcRows + r] = v[n];
        }
        bar_sync_named(1, 256);  // the row threads
        tc_tile_out(out, otile, max(owned, 0) * 8, row0, tok0 + 8 * rank * gpr, threadIdx.x, 256);
        return;
    }
    if (!foldt) return;
#pragma unroll
    for (int g = 0; g < G0; ++g) {
        if (g >= gcnt) break;
#pragma unroll
        for (int n = 0; n < 8; ++n) otile[(8 * (gbeg + g) + n) * kTcRows + r] = acc[g][n];
    }
    bar_sync_named(1, 256);  // the row threads
    tc_tile_out(out, otile, 8 * G, row0, tok0, threadIdx.x, 256);
}

template <int T, int G>
__global__ void __launch_bounds__(kTcThreads, 1) qg_tc_kernel(const __grid_constant__ Params p)
{
    pdl_trigger();
    const Mat &m = p.mat[select_mat(p, blockIdx.y)];
    tc_body<T, G>(p, m, blockIdx.y - m.tile_begin);
}

// Q4_K and Q6_K matrices of one call (the QKV triple) in one launch: each
// CTA runs the pipeline of its tile's format; the launch's shared memory and
// ring depths fit both formats (a cluster's CTAs share a tile, so a format).
template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) qg_tc_mixed_kernel(const __grid_constant__ Params p)
{
    pdl_trigger();
    const Mat &m = p.mat[select_mat(p, blockIdx.y)];
    if (m.type == T_Q6K)
        tc_body<T_Q6K, G>(p, m, blockIdx.y - m.tile_begin);
    else
        tc_body<T_Q4K, G>(p, m, blockIdx.y - m.tile_begin);
}

}  // namespace qg
