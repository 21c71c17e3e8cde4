// qg_tc_kernel: the Q4_K product for prefill chunks (N >= 33) on the
// 5th-generation tensor core.
//
// For N <= 32 every row must keep its bits whatever N is (TandemLLM
// "Kernels", Row invariance), so those calls stay on the mma.sync kernels;
// past 32 tokens that requirement is lifted and the tensor core's large MMAs
// pay: one tcgen05.mma of M 128 (weight rows) x N 64 (tokens) x K 16 costs
// about what an N = 8 one does on this GPU.
//
// Per CTA: 128 weight rows, up to 64 tokens, one K slice (super-blocks rank,
// rank + ks, ...; the ks ranks of a row tile form a cluster and add their
// partials in rank order).  Per super-block:
//   * warp 8 brings the 128 packed rows by one 3-D tensor copy and the staged
//     x of the CTA's tokens by one bulk copy;
//   * warps 0..3 (WG0) and 4..7 (WG1), one thread per row, decode the row's
//     256 weights exactly to fp16, A = sc*q*2^-22 (reflex-llm
//     "docs/kernels.md": dequantize in registers), WG0 qs chunks 0-1, WG1
//     chunks 2-3 and the 6-bit mins (m*2^-24), into tensor memory;
//   * warp 9 issues 16 MMAs for D1 = A.x and one for D2 = mins.(sub-block sums
//     of x, S = 32 hi + lo), N = all the CTA's tokens;
//   * the row threads read D1, D2 back (double-buffered) and fold
//       acc = fma(d * 2^22, D1, acc); acc = fma(-dmin * 2^24, D2, acc),
//     WG0 the first half of the token groups, WG1 the rest.
// x arrives in the tensor core's K-major core-matrix layout (stage_tc4).
#pragma once

#include "qg_kernels.cuh"

namespace qg {

constexpr int kTcRows = 128;
constexpr int kTcTok = 64;            // tokens per CTA (8 groups of 8)
constexpr int kTcXBlk = 4096 + 256;   // staged x per (super-block, 8-token group)
constexpr int kTcStagesMax = 4;
constexpr int kTcMinN = 33;           // smallest N served by qg_tc_kernel

// ---------------------------------------------------------------------------
// x of one (token, super-block) into the tensor-core layout of its 8-token
// group block `blk` (kTcXBlk bytes; token row `nrow` = token % 8):
//   [0, 4096)   k-step s (16), core j (2): 8 token rows x 16 bytes at
//               (2 s + j) * 128 + 16 nrow; the row holds, for the 4-groups
//               A = 16 c + w and A + 8 (c = s / 4, w = 2 (s % 4) + j), the
//               values (a0, a2, a1, a3, b0, b2, b1, b3) -- the order in
//               which a weight row's qs word w of chunk c is decoded;
//   [4096, 4352) core 0: fp16 hi of the 8 sub-block sums, core 1: the lo parts.
// Lane l holds x[256 sb + 8 l .. + 8].  Sub-block sums as in stage_sb
// (hi = fp16(S * 2^-5), lo = fp16(S - 32 hi)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void stage_tc4(uint4 v, int lane, uint8_t *blk, int nrow)
{
    uint4 w;
    w.x = __shfl_down_sync(0xffffffffu, v.x, 4);
    w.y = __shfl_down_sync(0xffffffffu, v.y, 4);
    w.z = __shfl_down_sync(0xffffffffu, v.z, 4);
    w.w = __shfl_down_sync(0xffffffffu, v.w, 4);
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
        *reinterpret_cast<uint4 *>(blk + (2 * s) * 128 + 16 * nrow) = o0;
        *reinterpret_cast<uint4 *>(blk + (2 * s + 1) * 128 + 16 * nrow) = o1;
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
        *reinterpret_cast<__half *>(blk + 4096 + 16 * nrow + 2 * sbk) = hi;
        *reinterpret_cast<__half *>(blk + 4096 + 128 + 16 * nrow + 2 * sbk) = lo;
    }
}

// ---------------------------------------------------------------------------
// Half H of one Q4_K row (the 144-byte block at ra in shared memory) ->
// tensor memory at ta (this thread's lane): qs chunks 2H, 2H + 1 to columns
// 64 H .. 64 H + 63 (column (8 c + w) * 4 + q for chunk c, qs word w: q = 0
// the low nibbles of bytes 0, 2; 1 of bytes 1, 3; 2, 3 the high nibbles --
// the k order stage_tc4 gives x).  Half 0 returns d * 2^22 and -dmin * 2^24;
// half 1 also writes the mins (m_2i, m_2i+1) to columns 128..135 (read by
// the last MMA of the super-block): times 2^-19 against the hi sums (columns
// 128..131), times 2^-24 (subnormals) against the lo sums (132..135).
// ---------------------------------------------------------------------------
template <int H>
__device__ __forceinline__ void tc_decode_q4k(uint32_t ra, uint32_t ta, float &dd, float &dm)
{
    const uint4 h = lds128(ra);
    // sub-blocks 4H .. 4H + 3: scales of chunks 2H (2 sub-blocks) and 2H + 1
    const uint32_t sw = (H == 0) ? (h.y & 0x3f3f3f3fu)
                                 : ((h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u));
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * H + cc;
        // sub-blocks 2c (low nibbles, 4 sc) and 2c + 1 (high nibbles, sc / 4)
        const uint32_t b0 = (2 * c) & 3, b1 = (2 * c + 1) & 3;
        const uint32_t slo = hsub2(__byte_perm(sw, 0x6C6Cu, 0x4040u | b0 | (b0 << 8)), 0x6C006C00u);
        const uint32_t shi = hsub2(__byte_perm(sw, 0x5C5Cu, 0x4040u | b1 | (b1 << 8)), 0x5C005C00u);
        const uint4 qa = lds128(ra + 16 + 32 * c), qb = lds128(ra + 32 + 32 * c);
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        uint32_t a[32];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            kq_decode<T_Q4K>(q[w], 0u, 0, 0, slo, shi, a[4 * w + 0], a[4 * w + 1]);
            kq_decode<T_Q4K>(q[w], 0u, 0, 1, slo, shi, a[4 * w + 2], a[4 * w + 3]);
        }
        tmem_st32(ta + 32 * c, a);
    }
    if (H == 0) {
        dd = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu))) * 4194304.0f;
        dm = -__half2float(__ushort_as_half((unsigned short)(h.x >> 16))) * 16777216.0f;
    } else {
        const uint32_t mn03 = h.z & 0x3f3f3f3fu;
        const uint32_t mn47 = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
        uint32_t mn[8];
        mn[0] = __byte_perm(mn03, 0u, 0x4140u);
        mn[1] = __byte_perm(mn03, 0u, 0x4342u);
        mn[2] = __byte_perm(mn47, 0u, 0x4140u);
        mn[3] = __byte_perm(mn47, 0u, 0x4342u);
        mn[4] = mn[0];
        mn[5] = mn[1];
        mn[6] = mn[2];
        mn[7] = mn[3];
#pragma unroll
        for (int i = 0; i < 4; ++i) mn[i] = hmul2(mn[i], 0x50005000u);  // * 32.0
        tmem_st8(ta + 128, mn);
    }
}

// ---------------------------------------------------------------------------
// Shared memory: [barriers, tmem base | ring of `stages` slots: 128 weight
// rows (18,432 B) + the staged x of G token groups (G x kTcXBlk)]; after the
// loop the rank partials [8 G][128] overlay the ring.  Tensor memory (512
// columns): A 0..127, mins 128..135, then two buffers of (D1: 8 G, D2: 8 G).
// ---------------------------------------------------------------------------
constexpr int kTcThreads = 320;  // WG0, WG1, producer warp, MMA warp
constexpr int kTcCols = 512;
__host__ __device__ inline int tc_slot_bytes(int G) { return kTcRows * 144 + G * kTcXBlk; }
__host__ __device__ inline int tc_smem_bytes(int G, int stages)
{
    const int body = stages * tc_slot_bytes(G);
    const int red = kTcRows * 8 * G * 4;
    return 256 + (body > red ? body : red);
}
// Staged x of qg_tc_kernel: [64-token chunk][super-block][8 groups][kTcXBlk].
__host__ __device__ inline int64_t tc_chunk_bytes(int nb) { return (int64_t)nb * 8 * kTcXBlk; }

// Epilogue of one output element: residual (fp32 add before the single
// rounding), fp16 RN or fp32 store.
__device__ __forceinline__ void tc_store(const Params &p, const Mat &m, int row, int tok, float val)
{
    if (row >= m.M || tok >= p.N) return;
    const int64_t o = (int64_t)tok * m.M + row;
    if (m.res) val = __fadd_rn(__half2float(m.res[o]), val);
    if (p.out_f32)
        reinterpret_cast<float *>(m.y)[o] = val;
    else
        reinterpret_cast<__half *>(m.y)[o] = __float2half_rn(val);
}

template <int G>
__global__ void __launch_bounds__(kTcThreads) qg_tc_kernel(const __grid_constant__ Params p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    pdl_trigger();
    const Mat &m = p.mat[select_mat(p, blockIdx.y)];
    const int rtile = blockIdx.y - m.tile_begin;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = blockIdx.x, ks = p.ks;
    const int nsb = (p.nb - rank + ks - 1) / ks;  // super-blocks rank, rank + ks, ...
    const int tok0 = p.tok_base + blockIdx.z * kTcTok;
    const int ntok = min(8 * G, p.N - tok0);
    const int row0 = rtile * kTcRows;
    const int STAGES = p.stages;
    const int slot_bytes = tc_slot_bytes(G);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase, bar_empty = sbase + 32;
    const uint32_t bar_a0 = sbase + 64, bar_a1 = sbase + 72, bar_f0 = sbase + 80;
    const uint32_t bar_d = sbase + 88;       // [2]: D buffer b complete (also: A half 1 free)
    const uint32_t bar_dfree = sbase + 104;  // [2]: D buffer b read back by all row threads
    const uint32_t ring = sbase + 256;
    const uint32_t xbytes = (uint32_t)(G * kTcXBlk);
    constexpr uint32_t kIdesc = tc_idesc_f16(8 * G);
    constexpr int G0 = (G + 1) / 2;  // token groups folded by WG0; WG1 folds the rest

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 4);  // WG0's warps release a slot after its fold
        }
        mbar_init(bar_a0, kTcRows);
        mbar_init(bar_a1, kTcRows);
        mbar_init(bar_f0, 1);
        mbar_init(bar_d, 1);
        mbar_init(bar_d + 8, 1);
        mbar_init(bar_dfree, 2 * kTcRows);
        mbar_init(bar_dfree + 8, 2 * kTcRows);
        mbar_fence_init();
    }
    if (warp == 9) tmem_alloc(sbase + 128, kTcCols);
    if (warp == 8 && lane == 0) prefetch_tmap(&m.tmw1);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *reinterpret_cast<volatile uint32_t *>(smem + 128);
    auto colD1 = [&](int b, int g) { return (uint32_t)(136 + 16 * G * b + 8 * g); };
    auto colD2 = [&](int b, int g) { return (uint32_t)(136 + 16 * G * b + 8 * G + 8 * g); };

    unsigned int err = 0;
    float acc[G0][8];  // WG0: groups 0..G0-1; WG1: groups G0..G-1 (the first G-G0 entries)
#pragma unroll
    for (int g = 0; g < G0; ++g)
#pragma unroll
        for (int n = 0; n < 8; ++n) acc[g][n] = 0.0f;

    if (warp == 8) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const int pre = min(STAGES, nsb);
            for (int i = 0; i < pre; ++i) {
                const uint32_t fb = bar_full + 8 * i;
                mbar_arrive_expect_tx(fb, (uint32_t)(kTcRows * 144) + xbytes);
                tma_load_3d(ring + i * slot_bytes, &m.tmw1, 0, row0, rank + i * ks, fb);
            }
            pdl_wait();  // the staged x is written by the kernel just before
            const uint8_t *xs = p.xs[XL_TC4] + (int64_t)(tok0 / kTcTok) * p.xs_tok_stride;
            for (int i = 0; i < pre; ++i)
                bulk_g2s(ring + i * slot_bytes + kTcRows * 144,
                         xs + (int64_t)(rank + i * ks) * (8 * kTcXBlk), xbytes, bar_full + 8 * i);
            int slot = 0;
            uint32_t par = 0;
            for (int i = STAGES; i < nsb; ++i) {
                if (!mbar_wait(bar_empty + 8 * slot, par)) {
                    err |= ERR_EMPTY_TIMEOUT;
                    break;
                }
                const int sb = rank + i * ks;
                const uint32_t dst = ring + slot * slot_bytes, fb = bar_full + 8 * slot;
                mbar_arrive_expect_tx(fb, (uint32_t)(kTcRows * 144) + xbytes);
                tma_load_3d(dst, &m.tmw1, 0, row0, sb, fb);
                bulk_g2s(dst + kTcRows * 144, xs + (int64_t)sb * (8 * kTcXBlk), xbytes, fb);
                if (++slot == STAGES) {
                    slot = 0;
                    par ^= 1u;
                }
            }
        }
    } else if (warp == 9) {
        // ---------------- MMA issue (one MMA of N = 8 G per k-step) ----------------
        int issued = 0;
        if (lane == 0) {
            int slot = 0;
            uint32_t par = 0;
            for (int i = 0; i < nsb && !err; ++i) {
                const int b = i & 1;
                if (!mbar_wait(bar_full + 8 * slot, par) ||  // staged x
                    (i >= 2 && !mbar_wait(bar_dfree + 8 * b, (uint32_t)(((i >> 1) - 1) & 1))) ||
                    !mbar_wait(bar_a0, (uint32_t)(i & 1))) {
                    err |= ERR_FULL_TIMEOUT;
                    break;
                }
                tc_fence_after();
                const uint32_t xb = ring + slot * slot_bytes + kTcRows * 144;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    tc_mma(tbase + colD1(b, 0), tbase + 8 * s, smem_desc2(xb + 256 * s, 128, kTcXBlk),
                           kIdesc, s > 0 ? 1u : 0u);
                tc_commit(bar_f0);  // A half 0 free once these complete
                if (!mbar_wait(bar_a1, (uint32_t)(i & 1))) {
                    err |= ERR_FULL_TIMEOUT;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int s = 8; s < 16; ++s)
                    tc_mma(tbase + colD1(b, 0), tbase + 8 * s, smem_desc2(xb + 256 * s, 128, kTcXBlk),
                           kIdesc, 1u);
                tc_mma(tbase + colD2(b, 0), tbase + 128, smem_desc2(xb + 4096, 128, kTcXBlk), kIdesc,
                       0u);
                tc_commit(bar_d + 8 * b);
                ++issued;
                if (++slot == STAGES) {
                    slot = 0;
                    par ^= 1u;
                }
            }
            // Nothing of this CTA may still run on the tensor core when its
            // tensor memory is released (matters only after a timeout).
            if (issued > 0)
                mbar_wait(bar_d + 8 * ((issued - 1) & 1), (uint32_t)(((issued - 1) >> 1) & 1));
        }
    } else {
        // ---------------- row threads: WG0 = warps 0..3, WG1 = warps 4..7 ----------------
        pdl_wait();  // y and the residual belong to earlier kernels too
        const int wg = warp >> 2;
        const int r = threadIdx.x & 127;  // row within the tile; tensor-memory lane
        const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
        const int gbeg = wg ? G0 : 0, gend = wg ? G : G0;
        // Fold super-block i (its D buffer) into this thread's token groups.
        auto fold = [&](int i, float dd, float dm) -> bool {
            const int b = i & 1;
            if (!mbar_wait(bar_d + 8 * b, (uint32_t)((i >> 1) & 1))) return false;
            tc_fence_after();
#pragma unroll
            for (int g = 0; g < G0; ++g) {
                const int gg = gbeg + g;
                if (gg >= gend || 8 * gg >= ntok) break;
                uint32_t d1[8], d2[8];
                tmem_ld8(tl + colD1(b, gg), d1);
                tmem_ld8(tl + colD2(b, gg), d2);
                tc_wait_ld();
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    if (8 * gg + n >= ntok) continue;
                    acc[g][n] = __fmaf_rn(dd, __uint_as_float(d1[n]), acc[g][n]);
                    acc[g][n] = __fmaf_rn(dm, __uint_as_float(d2[n]), acc[g][n]);
                }
            }
            tc_fence_before();
            mbar_arrive(bar_dfree + 8 * b);
            return true;
        };
        int slot = 0, pslot = 0;
        uint32_t par = 0;
        float pdd = 0.f, pdm = 0.f;
        bool ok = true;
        for (int i = 0; i < nsb && ok; ++i) {
            if (!mbar_wait(bar_full + 8 * slot, par)) {
                ok = false;
                break;
            }
            const uint32_t ra = ring + slot * slot_bytes + r * 144;
            float dd = 0.f, dm = 0.f;
            if (wg == 0) {
                // A half 0 is free once super-block i - 1's first MMAs completed
                if (i > 0 && !mbar_wait(bar_f0, (uint32_t)((i - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tc_decode_q4k<0>(ra, tl, dd, dm);
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(bar_a0);
                if (i > 0) {
                    if (!fold(i - 1, pdd, pdm)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_empty + 8 * pslot);
                }
            } else {
                // A half 1 and the mins are free once super-block i - 1
                // completed; fold it first.
                if (i > 0 && !fold(i - 1, pdd, pdm)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tc_decode_q4k<1>(ra, tl, dd, dm);
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(bar_a1);
                // d, dmin of this super-block for its fold
                const uint32_t hx = lds32(ra);
                dd = __half2float(__ushort_as_half((unsigned short)(hx & 0xffffu))) * 4194304.0f;
                dm = -__half2float(__ushort_as_half((unsigned short)(hx >> 16))) * 16777216.0f;
            }
            pdd = dd;
            pdm = dm;
            pslot = slot;
            if (++slot == STAGES) {
                slot = 0;
                par ^= 1u;
            }
        }
        if (ok && nsb > 0) {
            if (!fold(nsb - 1, pdd, pdm)) ok = false;
            if (wg == 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * pslot);
            }
        }
        if (!ok) err |= ERR_FULL_TIMEOUT;
    }
    if (err && p.err) atomicOr(p.err, err);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tbase, kTcCols);

    // Rank partials through distributed shared memory, added in rank order:
    // every rank publishes its tile [group][token][row]; rank q then sums the
    // q-th 1/ks of it over ranks 0..ks-1 (all remote loads in flight at once)
    // and stores it.
    float *red = reinterpret_cast<float *>(smem + 256);
    const bool rowt = warp < 8;
    const int r = threadIdx.x & 127;
    const int gbeg = (warp >= 4) ? G0 : 0, gcnt = (warp >= 4) ? G - G0 : G0;
    if (ks > 1) {
        if (rowt) {
#pragma unroll
            for (int g = 0; g < G0; ++g)
                if (g < gcnt)
#pragma unroll
                    for (int n = 0; n < 8; ++n) red[((gbeg + g) * 8 + n) * kTcRows + r] = acc[g][n];
        }
        cluster_sync();
        const int per = G * 8 * kTcRows / ks;  // floats of this rank's share (a multiple of 4)
        const uint32_t rbase = smem_u32(red);
        for (int q4 = threadIdx.x; 4 * q4 < per; q4 += blockDim.x) {
            const int idx0 = rank * per + 4 * q4;
            float4 part[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < ks) part[q] = ld_dsmem_v4(map_shared_rank(rbase + 4 * idx0, (uint32_t)q));
            float4 sum = part[0];
#pragma unroll
            for (int q = 1; q < 8; ++q) {
                if (q < ks) {
                    sum.x = __fadd_rn(sum.x, part[q].x);
                    sum.y = __fadd_rn(sum.y, part[q].y);
                    sum.z = __fadd_rn(sum.z, part[q].z);
                    sum.w = __fadd_rn(sum.w, part[q].w);
                }
            }
            // four consecutive rows of one token
            store_out4<T_Q4K>(p, m, row0 + idx0 % kTcRows, tok0 + idx0 / kTcRows, sum);
        }
        cluster_arrive_relaxed();
        cluster_wait();
        return;
    }
    if (!rowt) return;
#pragma unroll
    for (int g = 0; g < G0; ++g) {
        if (g >= gcnt) break;
#pragma unroll
        for (int n = 0; n < 8; ++n) tc_store(p, m, row0 + r, tok0 + 8 * (gbeg + g) + n, acc[g][n]);
    }
}

}  // namespace qg
