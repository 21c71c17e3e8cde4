// Chain of decode calls in one persistent launch (N <= 8, K-quant weights):
// the calls of a transformer layer (QKV triple -> Wo + residual -> gate/up
// pair -> down) run back to back inside one grid that stays resident, so the
// weight ring keeps streaming across call boundaries instead of draining and
// refilling at every kernel boundary (reflex-llm "docs/performance.md",
// Level 4: persistent kernels that stay resident on the SMs).
//
// Order: call c reads its x and residual only after every CTA has stored its
// outputs of calls 0 .. c-1 (a device counter with release/acquire ordering),
// so any call may read what an earlier call wrote, exactly as the same calls
// issued one by one on a stream.  Weights never change during a chain, so the
// producer warp issues the next call's weights as soon as its own side has
// published (without waiting for the other CTAs).
//
// On GB300 the same calls as one launch each, chained by programmatic
// dependent launch, measured faster (the decode layer 29.0 vs 35.0 us), so
// this form is opt-in (QG_CHAIN_PERSISTENT).
//
// Placement: one CTA per SM holding two independent pipelines ("sides"),
// each a producer warp and 8 consumer warps with its own ring, staged x and
// partials, so that virtual CTA v = side * gridDim.x + blockIdx.x and the
// tiles t and t + gridDim.x of a call always share an SM while tiles
// t < gridDim.x are spread over every SM (with two CTAs per SM the hardware
// placed them unevenly: a 160-tile call ran on 80 SMs).
//
// Arithmetic: each row tile is computed by the same per-slice code as
// qg_n8_kernel (compute_sb, slices added in slice order), so every output has
// the bits of the single-call entry points.
#pragma once

#include "qg_kernels.cuh"

namespace qg {

constexpr int kChainMaxCalls = 4;
constexpr int kChainMaxMats = 3 * kChainMaxCalls;
enum { ERR_CHAIN_TIMEOUT = 4 };

constexpr int kChainSlots = 8;  // barrier pairs of a side's ring
constexpr int kChainHdr = 256;  // barriers of a side: full[8], empty[8], published

struct ChainCall {
    int mat0, nmat;      // matrices mat0 .. mat0 + nmat - 1 of ChainParams::mat
    int tiles;           // row tiles of the call; Mat::tile_begin is relative to the call
    int stages;          // ring slots of this call (<= kChainSlots)
    int slot_bytes;      // bytes of one slot (the call's largest stage)
    int N, K, nb, xtok;  // tokens, K, super-blocks, token stride of the staged x
    int out_f32;
    const __half *x;     // [N][K]
};

constexpr int kChainSideThreads = 32 * (kGemvCW + 1);  // one side: producer + 8 consumers
constexpr int kChainThreads = 2 * kChainSideThreads;

struct ChainParams {
    Mat mat[kChainMaxMats];
    ChainCall call[kChainMaxCalls];
    int ncalls;
    int side_bytes;      // shared memory of one side (the second starts there)
    int xoff, redoff;    // offsets (within a side) of the staged x and the slice partials
    unsigned int *err;   // error word (timeouts)
    unsigned int *ctr;   // [0] calls finished, summed over CTAs; [1] CTAs done waiting
    int hold_publish;    // test hook: virtual CTA 0 never publishes (the others' waits run out)
};

// Longest wait for the earlier calls' outputs before a side gives up (sets
// ERR_CHAIN_TIMEOUT and goes on): far beyond any call's duration.
constexpr unsigned long long kChainWaitNs = 500ull * 1000 * 1000;

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint4 ld_cg_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned short ld_cg_u16(const void *p)
{
    unsigned short v;
    asm volatile("ld.global.cg.u16 %0, [%1];\n" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned int *p, unsigned int v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int chain_mat(const ChainParams &p, const ChainCall &cl, int tile)
{
    int mi = cl.mat0;
    for (int j = 1; j < cl.nmat; ++j)
        if (tile >= p.mat[cl.mat0 + j].tile_begin) mi = cl.mat0 + j;
    return mi;
}

// The ring of one side is re-cut at every call into cl.stages slots of
// cl.slot_bytes (more slots for the smaller Q4_K stages), starting at byte
// kChainHdr.  Barrier pair i (full at 8 i, empty at 64 + 8 i) belongs to slot
// i; phase bits are kept per slot.  The producer starts a call only after
// every slot of the previous call has been released, so a re-cut never
// overwrites unread data, and only after its side has published the previous
// call's outputs (barrier at 128): the release waits for the side's stores,
// which would otherwise queue behind the burst of weight copies.
struct ChainProd {
    uint32_t k;      // stages of the current call issued
    uint32_t epar;   // per slot: parity of the next empty phase to wait for
    uint32_t used;   // slots holding a stage not yet waited free
    uint32_t fiss;   // per slot: parity of the last full phase issued
};

__device__ __forceinline__ bool chain_release_all(uint32_t sbase, ChainProd &r)
{
    for (int i = 0; i < kChainSlots; ++i) {
        if (!((r.used >> i) & 1u)) continue;
        if (!__all_sync(0xffffffffu, mbar_wait(sbase + 64 + 8 * i, (r.epar >> i) & 1u)))
            return false;
        r.epar ^= 1u << i;
    }
    r.used = 0;
    return true;
}

// Producer warp: every stage of one row tile into the ring.
template <int T>
__device__ __forceinline__ bool chain_produce(const ChainCall &cl, const Mat &m, int rtile,
                                              uint8_t *smem, ChainProd &r, uint64_t wpol,
                                              int lane)
{
    const int kw = m.kw, R = kGemvRows / kw;
    const int nst = (cl.nb + kw - 1) / kw;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t S = (uint32_t)cl.stages;
    for (int i = 0; i < nst; ++i, ++r.k) {
        const uint32_t slot = r.k % S;
        // (the lanes decide together: the Q6_K copies below shuffle across the warp)
        if ((r.used >> slot) & 1u) {
            if (!__all_sync(0xffffffffu, mbar_wait(sbase + 64 + 8 * slot, (r.epar >> slot) & 1u)))
                return false;
            r.epar ^= 1u << slot;
        }
        const uint32_t off = kChainHdr + slot * (uint32_t)cl.slot_bytes;
        // the stage's own bytes (a slot may be larger: it fits the call's largest stage)
        gemv_produce<T>(m, kw, R, rtile * R, cl.nb, i, sbase + off, smem + off, sbase + 8 * slot,
                        gemv_stage_bytes<T>(kw), wpol, lane);
        r.used |= 1u << slot;
        r.fiss ^= 1u << slot;
    }
    return true;
}

// x of one call in format T's staged layout, by the 8 consumer warps
// (coherent loads: an earlier call of the chain may have written x).
template <int T>
__device__ __forceinline__ void chain_stage_x(const ChainCall &cl, uint8_t *xr, int cw, int lane)
{
    using F = Fmt<T>;
    constexpr int XU = 4;
    const int nwarps = kGemvCW;
    const int nb = cl.nb, total = cl.N * nb;
    int n = 0, sb = cw;
    while (sb >= nb) {
        sb -= nb;
        ++n;
    }
    for (int base = cw; base < total; base += XU * nwarps) {
        uint4 v[XU];
        uint32_t dst[XU];
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            if (base + u * nwarps < total) {
                v[u] = ld_cg_v4(cl.x + (int64_t)n * cl.K + 256 * sb + 8 * lane);
                dst[u] = (uint32_t)(n * cl.xtok + sb * kXTok);
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
                uint8_t *d = xr + dst[u];
                stage_sb(v[u], lane, F::XL == XL_Q4 ? d : nullptr, F::XL == XL_Q6 ? d : nullptr,
                         nullptr);
            }
        }
    }
}

// Consumer warps: one row tile (all its stages), slice partials added in
// slice order, then the epilogue.  ok turns false when a wait of this warp
// runs out; from then on the warp neither waits for nor releases ring slots
// (a slot released without its data would let the producer re-arm a barrier
// whose phase never completed), but it still takes every named barrier, so
// the warps of the CTA stay in step and the kernel ends.
template <int T, bool ODD>
__device__ __forceinline__ void chain_tile(const ChainParams &p, const ChainCall &cl, const Mat &m,
                                           int rtile, uint8_t *smem, uint32_t &k, uint32_t &fpar,
                                           bool &ok, int tid, int bar)
{
    using F = Fmt<T>;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int kw = m.kw, R = kGemvRows / kw;
    const int nst = (cl.nb + kw - 1) / kw;
    const int c = warp - 1;
    const int mg = c / kw, ks = c - mg * kw;
    const int row_w = rtile * R + 16 * mg;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t S = (uint32_t)cl.stages;
    const uint32_t xreg = sbase + p.xoff;
    const KSel ksel = k_sel(t);
    const uint32_t wrow = (T == T_Q6K) ? (uint32_t)(16 * mg * q6_pitch(kw))
                                       : (uint32_t)((ks * R + 16 * mg) * F::BB);
    Acc<T, 1, 1> A;
    A.zero();
    for (int i = 0; i < nst && ok; ++i, ++k) {
        const uint32_t slot = k % S;
        // (the lanes decide together: the MMAs below need the whole warp)
        if (!__all_sync(0xffffffffu, mbar_wait(sbase + 8 * slot, (fpar >> slot) & 1u))) {
            ok = false;
            break;
        }
        fpar ^= 1u << slot;
        const int sb = i * kw + ks;
        if (sb < cl.nb) {
            const uint32_t sl = sbase + kChainHdr + slot * (uint32_t)cl.slot_bytes;
            const uint32_t xsl = xreg + sb * kXTok;
            if (T == T_Q6K)
                compute_sb<T, 1, 1, ODD>(A, sl + wrow, xsl, cl.xtok, g, t, cl.N, m, row_w, sb,
                                         ksel, q6_pitch(kw), 0u, i * kw);
            else
                compute_sb<T, 1, 1, ODD>(A, sl + wrow, xsl, cl.xtok, g, t, cl.N, m, row_w, sb,
                                         ksel);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sbase + 64 + 8 * slot);
    }

    // Slice partials: slices 1..kw-1 publish, slice 0 adds them in slice order.
    float *red = reinterpret_cast<float *>(smem + p.redoff);
    float v[4];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) v[cc] = A.partial(0, 0, cc);
    if (ks > 0) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) red[(c * 4 + cc) * 32 + lane] = v[cc];
    }
    bar_sync_named(bar, 32 * kGemvCW);
    if (ks == 0) {
        for (int qq = 1; qq < kw; ++qq) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) v[cc] += red[((c + qq) * 4 + cc) * 32 + lane];
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int row = row_w + g + 8 * (cc >> 1);
            const int tok = 2 * t + (cc & 1);
            if (row >= m.M || tok >= cl.N) continue;
            float val = v[cc];
            const int64_t o = (int64_t)tok * m.M + row;
            if (m.res) val = __fadd_rn(__half2float(__ushort_as_half(ld_cg_u16(m.res + o))), val);
            if (cl.out_f32)
                reinterpret_cast<float *>(m.y)[o] = val;
            else
                reinterpret_cast<__half *>(m.y)[o] = __float2half_rn(val);
        }
    }
    bar_sync_named(bar, 32 * kGemvCW);  // red is free for the next tile
}

template <int TSET, bool ONE>
__global__ void __launch_bounds__(kChainThreads, 1) qg_chain_kernel(const __grid_constant__ ChainParams p)
{
    extern __shared__ __align__(128) uint8_t smem_all[];
    pdl_trigger();
    const int side = threadIdx.x >= kChainSideThreads ? 1 : 0;
    const int tid = threadIdx.x - side * kChainSideThreads;
    const int warp = tid >> 5, lane = tid & 31;
    uint8_t *smem = smem_all + side * p.side_bytes;
    const uint32_t sbase = smem_u32(smem);
    const int bar = 1 + side;  // this side's consumer barrier
    const int G = 2 * gridDim.x, b = side * gridDim.x + blockIdx.x;  // virtual CTAs
    if (tid == 0) {
        for (int s = 0; s < kChainSlots; ++s) {
            mbar_init(sbase + 8 * s, 1);
            mbar_init(sbase + 64 + 8 * s, kGemvCW);
        }
        mbar_init(sbase + 128, 1);  // this side published a call's outputs
        mbar_fence_init();
    }
    __syncthreads();
    unsigned int err = 0;

    if (warp == 0) {
        // Producer: the weights of every tile of this side, in chain order; it
        // runs ahead of the consumers by the ring depth, across calls.
        const uint64_t wpol = l2_evict_first_policy();
        ChainProd r = {0u, 0u, 0u, 0u};
        bool ok = true;
        for (int c = 0; c < p.ncalls && ok; ++c) {
            const ChainCall &cl = p.call[c];
            if (b >= cl.tiles) continue;
            ok = chain_release_all(sbase, r);  // the ring is re-cut for this call
            if (ok && c > 0)  // the outputs of call c - 1 are published
                ok = __all_sync(0xffffffffu, mbar_wait(sbase + 128, (uint32_t)(c - 1) & 1u));
            r.k = 0;
            for (int tl = b; tl < cl.tiles && ok; tl += G) {
                const Mat &m = p.mat[chain_mat(p, cl, tl)];
                const int rtile = tl - m.tile_begin;
                if constexpr ((TSET & TS_Q4K) != 0)
                    if (m.type == T_Q4K) ok = chain_produce<T_Q4K>(cl, m, rtile, smem, r, wpol, lane);
                if constexpr ((TSET & TS_Q5K) != 0)
                    if (m.type == T_Q5K) ok = chain_produce<T_Q5K>(cl, m, rtile, smem, r, wpol, lane);
                if constexpr ((TSET & TS_Q6K) != 0)
                    if (m.type == T_Q6K) ok = chain_produce<T_Q6K>(cl, m, rtile, smem, r, wpol, lane);
            }
        }
        if (!ok) err |= ERR_EMPTY_TIMEOUT;
        // Wait (bounded) until the last stages' copies have landed, so no copy
        // is in flight when the CTA exits, whatever happened downstream.
        for (int i = 0; i < kChainSlots; ++i)
            if (((r.used >> i) & 1u) &&
                !mbar_wait(sbase + 8 * i, ((r.fiss >> i) & 1u) ^ 1u)) {
                err |= ERR_FULL_TIMEOUT;
                break;
            }
    } else {
        const int cw = warp - 1;
        pdl_wait();  // x, residuals and outputs of earlier kernels
        uint32_t fpar = 0;  // per slot: parity of the next full phase
        bool ok = true;
        for (int c = 0; c < p.ncalls; ++c) {
            const ChainCall &cl = p.call[c];
            uint32_t k = 0;     // stages of this call consumed
            if (c > 0) {
                // every side of every CTA has stored its outputs of calls 0 .. c-1
                if (tid == 32) {
                    const unsigned int target = (unsigned int)G * (unsigned int)c;
                    const unsigned long long t0 = globaltimer_ns();
                    while (ld_acquire_u32(p.ctr) < target) {
                        if (globaltimer_ns() - t0 > kChainWaitNs) {
                            err |= ERR_CHAIN_TIMEOUT;
                            break;
                        }
                    }
                }
                bar_sync_named(bar, 32 * kGemvCW);
            }
            int staged = -1;  // staged-x layout of this call in shared memory
            for (int tl = b; tl < cl.tiles; tl += G) {
                const Mat &m = p.mat[chain_mat(p, cl, tl)];
                const int rtile = tl - m.tile_begin;
                const int lay = (m.type == T_Q6K) ? XL_Q6 : XL_Q4;
                if (lay != staged) {
                    // (the last tile's closing barrier freed the x region)
                    if (lay == XL_Q6)
                        chain_stage_x<T_Q6K>(cl, smem + p.xoff, cw, lane);
                    else
                        chain_stage_x<T_Q4K>(cl, smem + p.xoff, cw, lane);
                    bar_sync_named(bar, 32 * kGemvCW);
                    staged = lay;
                }
                if constexpr ((TSET & TS_Q4K) != 0)
                    if (m.type == T_Q4K) chain_tile<T_Q4K, !ONE>(p, cl, m, rtile, smem, k, fpar, ok, tid, bar);
                if constexpr ((TSET & TS_Q5K) != 0)
                    if (m.type == T_Q5K) chain_tile<T_Q5K, !ONE>(p, cl, m, rtile, smem, k, fpar, ok, tid, bar);
                if constexpr ((TSET & TS_Q6K) != 0)
                    if (m.type == T_Q6K) chain_tile<T_Q6K, !ONE>(p, cl, m, rtile, smem, k, fpar, ok, tid, bar);
            }
            if (c + 1 < p.ncalls) {
                // this side's outputs of call c are stored: the named barrier
                // orders every consumer thread's stores before the release
                bar_sync_named(bar, 32 * kGemvCW);
                if (tid == 32) {
                    if (!(p.hold_publish && b == 0)) red_release_add(p.ctr, 1u);
                    mbar_arrive(sbase + 128);
                }
            }
        }
        if (!ok) err |= ERR_FULL_TIMEOUT;
        if (tid == 32 && p.ncalls > 1) {
            // The last side past its waits resets the counters for the next
            // launch (which reads them only after this grid has completed).
            if (atomicAdd(p.ctr + 1, 1u) == (unsigned int)G - 1) {
                atomicExch(p.ctr, 0u);
                atomicExch(p.ctr + 1, 0u);
            }
        }
    }
    if (err && p.err) atomicOr(p.err, err);
}

// Shared memory of one side of qg_chain_kernel: barriers, the ring, the
// staged x of the largest call and the slice partials (the CTA holds two).
__host__ __device__ inline int chain_side_bytes(int ring_bytes, int xbytes)
{
    return kChainHdr + ring_bytes + xbytes + kGemvCW * 4 * 32 * 4;
}

}  // namespace qg
