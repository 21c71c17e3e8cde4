// C ABI of the qgemv library: handles, launch plan, argument validation,
// staging + product launches, reference fallback and error reporting.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "qg_chain.cuh"
#include "qg_launch.cuh"
#include "qg_tc.cuh"
#include "qgemv.h"

using namespace qg;

namespace qg {
unsigned int *noalloc_error_word();  // qg_noalloc.cu (null on failure, message set)
}

struct qg_handle {
    qg_type type;
    int64_t M, K;
    int nb;
    const uint8_t *w;
    const uint8_t *sc;
    float gscale;
    int64_t row_bytes, sc_row_bytes, w_bytes;
    uint32_t flags;
    int max_tokens;
    int kw;        // K slices, fixed by (M, K)
    int layout;    // staged-x layout this format reads
    uint8_t *xs;   // staging buffer: max_tokens * nb * kXTok bytes
    unsigned int *err;  // device error word written by the kernels (timeouts)
    CUtensorMap tmw, tms;  // 3-D maps [block][row][bytes] for the N <= 8 kernel
    CUtensorMap tmw1, tms1;  // the same with a 128-row x 1-block box (qg_sk_kernel)
    CUtensorMap xmap[4];   // 2-D maps of this handle's staging buffer, box 8 (G) tokens
    int device;
    int sms = 0;           // SM count of that device
    void *hx;      // device buffers of the host-pointer entry point
    size_t hx_cap;
    void *hy;
    size_t hy_cap;
    bool owns_buffers;     // xs and err were allocated by qgemv_create
};

struct qg_chain {
    int device;
    int sms;
    uint32_t flags;       // QG_CHAIN_*
    unsigned int *words;  // [0] calls finished (summed over CTAs), [1] CTAs past their
                          // waits, [2] error word
};

namespace {

thread_local std::string g_err;

qg_status fail(qg_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

qg_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(QG_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool env_on(const char *name)
{
    const char *v = getenv(name);
    return v && *v && strcmp(v, "0") != 0;
}

bool fault_at(const char *site)
{
    const char *v = getenv("QGEMV_FAULT_INJECT");
    return v && strcmp(v, site) == 0;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int block_bytes(qg_type t)
{
    switch (t) {
    case QG_Q4_K: return 144;
    case QG_Q5_K: return 176;
    case QG_Q6_K: return 210;
    case QG_FP8_E4M3: return 256;  // codes of one 256-wide super-block of a row
    default: return 0;
    }
}

bool type_known(int t)
{
    return t == QG_Q4_K || t == QG_Q5_K || t == QG_Q6_K || t == QG_NVFP4_W4A16 ||
           t == QG_FP8_E4M3;
}

int layout_of(qg_type t)
{
    if (t == QG_Q6_K) return XL_Q6;
    if (t == QG_NVFP4_W4A16 || t == QG_FP8_E4M3) return XL_FP4;  // x in natural 16-byte units
    return XL_Q4;
}

int tset_bit(qg_type t)
{
    switch (t) {
    case QG_Q4_K: return TS_Q4K;
    case QG_Q5_K: return TS_Q5K;
    case QG_Q6_K: return TS_Q6K;
    case QG_FP8_E4M3: return TS_FP8;
    default: return TS_FP4;
    }
}

// K slices: the smallest power of two up to 8 that gives this matrix alone at least
// 120 row tiles of 128 / kw rows (about 0.8 CTA per SM of the N <= 8 kernel),
// and never more than the super-blocks.  Depends on (M, K) only, so every
// row's reduction order is fixed by the shape.  (The 120 rather than one per
// SM keeps Q 4096 x 2560 at 4 slices of 2-3 super-blocks instead of 8 slices
// of 1-2: measured N = 32 7.5 vs 17.0 us, the decode layer 29.7 vs 30.8 us.)
int plan_kw(int64_t M, int nb)
{
    int kw = 1;  // a power of two: kGemvRows / kw rows are whole 16-row tiles
    while (kw < 8 && 2 * kw <= nb && (M + kGemvRows / kw - 1) / (kGemvRows / kw) < 120) kw *= 2;
    return kw;
}

int groups_for(int64_t n) { return n >= 32 ? 4 : (int)((n + 7) / 8); }

// qg_n8_kernel keeps x for the whole K in shared memory; beyond about 48 KB of
// it the smaller ring costs more than qg_sk_kernel's per-stage x copies
// (measured crossover on the sweep shapes: 34-46 KB).
bool gemv_x_fits(int64_t n, int nb) { return n * nb * kXTok <= 48 * 1024; }

// Dynamic shared memory that keeps qg_sk_kernel at one CTA per SM (more than
// half of the 228 KB an SM has).
constexpr int kSkSpreadSmem = 120 * 1024;

// For N >= 2, Q4_K / Q5_K matrices of at most 4096 rows run faster on
// qg_sk_kernel than on qg_n8_kernel (measured at N = 2..8: Wo 2560 x 4096 5.2-5.4
// vs 6.2-7.7 us, K/V 1024 x 2560 4.5-4.8 vs 4.8-6.7 us, Q 4096 x 2560
// 5.9-6.0 vs 6.1-7.5 us, Q5_K 2560 x 9728 12.1-12.4 vs 12.2-12.6 us); the
// 9728-row matrices, Q6_K and NVFP4 do not.  Both kernels give the same
// bits, so this only moves time.
bool sk_preferred(const qg_handle *const *hs, int nh, int64_t n)
{
    if (n < 2) return false;
    for (int i = 0; i < nh; ++i)
        if ((hs[i]->type != QG_Q4_K && hs[i]->type != QG_Q5_K) || hs[i]->M > 4096) return false;
    return true;
}

// Stage bytes of the N <= 8 kernel for a format and slice count.
int gemv_stage_bytes_host(qg_type t, int kw)
{
    const int R = kGemvRows / kw;
    if (t == QG_Q6_K) return R * q6_pitch(kw);
    if (t == QG_NVFP4_W4A16) return kw * R * (128 + 16);
    return kw * R * block_bytes(t);
}

cudaError_t launch_gemv_tset(int tset, const Params &p, dim3 grid, int smem, cudaStream_t s)
{
    switch (tset) {
    case TS_Q4K: return launch_gemv_q4k(p, grid, smem, s);
    case TS_Q5K: return launch_gemv_q5k(p, grid, smem, s);
    case TS_Q6K: return launch_gemv_q6k(p, grid, smem, s);
    case TS_FP4: return launch_gemv_fp4(p, grid, smem, s);
    case TS_FP8: return launch_gemv_fp8(p, grid, smem, s);
    case TS_Q4K | TS_Q6K: return launch_gemv_q4k_q6k(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

Mat mat_of(const qg_handle *h, void *y, const __half *res)
{
    Mat m;
    memset(&m, 0, sizeof m);
    m.tmw = h->tmw;
    m.tms = h->tms;
    m.tmw1 = h->tmw1;
    m.tms1 = h->tms1;
    m.kw = h->kw;
    m.w = h->w;
    m.sc = h->sc;
    m.y = y;
    m.res = res;
    m.row_bytes = h->row_bytes;
    m.sc_row_bytes = h->sc_row_bytes;
    m.w_bytes = h->w_bytes;
    m.M = (int)h->M;
    m.type = (int)h->type;
    m.tile_begin = 0;
    m.gscale = h->gscale;
    return m;
}

bool tset_supported(int tset)
{
    return tset == TS_Q4K || tset == TS_Q5K || tset == TS_Q6K || tset == TS_FP4 ||
           tset == TS_FP8 || tset == (TS_Q4K | TS_Q6K);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
        else
            cudaGetLastError();
    }
    return fn;
}

// 3-D map of a matrix of `rows` rows (row stride row_bytes) made of blocks of
// `bb` bytes (viewed as 8-byte elements): dims (bytes of a block, row, block),
// box (bb, box_rows, box_blocks), so a copy lands as [block][row][bytes].
bool encode_blocks(CUtensorMap *m, const void *base, int64_t row_bytes, int64_t rows, int bb,
                   int box_rows, int box_blocks, bool swizzle128 = false)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)(bb / 8), (cuuint64_t)rows, (cuuint64_t)(row_bytes / bb)};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)bb};
    cuuint32_t box[3] = {(cuuint32_t)(bb / 8), (cuuint32_t)box_rows, (cuuint32_t)box_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map of the staging buffer: rows are tokens (stride nb * 576 bytes), a
// row is nb units of 576 bytes (72 8-byte elements); box = one unit x
// box_rows tokens.
bool encode_staged(CUtensorMap *m, const void *base, int nb, int64_t rows, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t unit = kXTok / 8;
    cuuint64_t dims[2] = {(cuuint64_t)nb * unit, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)nb * kXTok};
    cuuint32_t box[2] = {(cuuint32_t)unit, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sk_tset_smem(int wbytes, int G, bool q6, int *stages, bool fp8 = false)
{
    int st = kSkStagesMax;
    // Two CTAs per SM where the ring allows it; Q6_K (weights two stages
    // ahead, by cp.async from the consumers) needs at least three slots.
    while (st > 2 && sk_smem_bytes(wbytes, G, st, fp8) > 110 * 1024) --st;
    if (q6 && st < 3) st = 3;
    *stages = st;
    return sk_smem_bytes(wbytes, G, st, fp8);
}

// qg_sk_kernel with x staged inside (p.xin): ring of weights only, then this
// rank's x for all its super-blocks (ceil(nb / ks) x 8 G tokens x 576 B).
// Two CTAs per SM where the ring allows it, as above.  Returns 0 when the x
// region would be too large (the staging kernel is used instead).
constexpr int kSkXinMax = 100 * 1024;
bool sk_xin_ok(int64_t n, int nb, int kw)
{
    const int64_t nsb = (nb + kw - 1) / kw;  // super-blocks of the largest rank
    return n <= 8 && n * nsb <= 32 && nsb * 8 * groups_for(n) * kXTok <= kSkXinMax;
}
int sk_xin_smem(int wbytes, int G, bool q6, int nb, int ks, int *stages, bool fp8 = false)
{
    const int xreg = ((nb + ks - 1) / ks) * 8 * G * kXTok;
    if (xreg > kSkXinMax) return 0;
    const int red = kSkCons * 32 * G * 4 * 4;
    auto total = [&](int st) {
        const int body = st * sk_slot_bytes(fp8, 0, wbytes) + xreg;
        return (fp8 ? kFp8RingOffset : 128) + (body > red ? body : red);
    };
    int st = kSkStagesMax;
    while (st > 2 && total(st) > 110 * 1024) --st;
    if (q6 && st < 3) st = 3;
    *stages = st;
    return total(st);
}

cudaError_t launch_sk_tset(int tset, int G, const Params &p, dim3 grid, int smem, cudaStream_t s)
{
    switch (tset) {
    case TS_Q4K: return launch_sk_q4k(G, p, grid, smem, s);
    case TS_Q5K: return launch_sk_q5k(G, p, grid, smem, s);
    case TS_Q6K: return launch_sk_q6k(G, p, grid, smem, s);
    case TS_FP4: return launch_sk_fp4(G, p, grid, smem, s);
    case TS_FP8: return launch_sk_fp8(G, p, grid, smem, s);
    case TS_Q4K | TS_Q6K: return launch_sk_q4k_q6k(G, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

// The whole path for 1..3 handles that share x: staging, then one product
// launch per chunk of at most max_tokens rows (several launches only when the
// formats have no common kernel).
qg_status run_product_mma(qg_handle *const *hs, int nh, const __half *x, int64_t N,
                          void *const *ys, const __half *res, int out_f32, cudaStream_t s,
                          bool swiglu = false)
{
    const qg_handle *h0 = hs[0];
    uint32_t flags = 0;
    int max_tokens = h0->max_tokens;
    for (int i = 0; i < nh; ++i) {
        flags |= hs[i]->flags;
        if (hs[i]->max_tokens < max_tokens) max_tokens = hs[i]->max_tokens;
    }
    const bool force_ref = (flags & QG_FLAG_FORCE_REFERENCE) != 0;
    g_err.clear();

    int tset = 0;
    for (int i = 0; i < nh; ++i) tset |= tset_bit(hs[i]->type);
    const bool fp8 = (tset & TS_FP8) != 0;  // FP8 launches hold FP8 matrices only

    for (int64_t c0 = 0; c0 < N; c0 += max_tokens) {
        const int n = (int)((N - c0) < max_tokens ? (N - c0) : max_tokens);
        const __half *xc = x + c0 * h0->K;
        auto ref_fallback = [&](const Params &pp) -> qg_status {
            if (swiglu) {
                cudaError_t re = launch_ref_swiglu(pp.mat[0], pp.mat[1], (int)h0->K, xc, n,
                                                   out_f32, s);
                if (re != cudaSuccess) return cuda_fail(re, "reference kernel launch");
                return QG_OK;
            }
            for (int j = 0; j < pp.nmat; ++j) {
                cudaError_t re = launch_ref_gemv(pp.mat[j], (int)h0->K, xc, n, out_f32, s);
                if (re != cudaSuccess) return cuda_fail(re, "reference kernel launch");
            }
            return QG_OK;
        };
        if (force_ref && swiglu) {
            Params pp;
            memset(&pp, 0, sizeof pp);
            pp.nmat = 2;
            for (int i = 0; i < 2; ++i)
                pp.mat[i] = mat_of(hs[i], ys[i] ? (uint8_t *)ys[i] + c0 * hs[i]->M * (out_f32 ? 4 : 2)
                                                : nullptr,
                                   nullptr);
            const qg_status rs = ref_fallback(pp);
            if (rs != QG_OK) return rs;
            continue;
        }
        if (force_ref) {
            for (int i = 0; i < nh; ++i) {
                Mat m = mat_of(hs[i], (uint8_t *)ys[i] + c0 * hs[i]->M * (out_f32 ? 4 : 2),
                               res ? res + c0 * hs[i]->M : nullptr);
                cudaError_t e = launch_ref_gemv(m, (int)h0->K, xc, n, out_f32, s);
                if (e != cudaSuccess) return cuda_fail(e, "reference kernel launch");
            }
            continue;
        }
        // Groups of handles that one kernel serves.
        int groups[3][3];
        int gsize[3] = {0, 0, 0};
        int ng = 0;
        if (tset_supported(tset)) {
            for (int i = 0; i < nh; ++i) groups[0][gsize[0]++] = i;
            ng = 1;
        } else {
            for (int i = 0; i < nh; ++i) {
                groups[ng][0] = i;
                gsize[ng++] = 1;
            }
        }
        // N <= 8 with the whole x of the call fitting in shared memory: one
        // kernel per group, x staged inside the kernel.
        int gemv_smem = 0, gemv_stages = 1;
        if (n <= 8) {
            int sbytes = 0, nst = 1;
            for (int i = 0; i < nh; ++i) {
                const int b = gemv_stage_bytes_host(hs[i]->type, hs[i]->kw);
                if (b > sbytes) sbytes = b;
                const int st = (h0->nb + hs[i]->kw - 1) / hs[i]->kw;
                if (st > nst) nst = st;
            }
            gemv_stages = nst < kGemvStagesMax ? nst : kGemvStagesMax;
            // Two CTAs per SM when a shallower ring allows it: never below 3
            // stages, or 2 when the grid has more row tiles than SMs (one
            // CTA per SM would run it as two waves).
            int tiles = 0;
            for (int i = 0; i < nh; ++i) {
                const int R = kGemvRows / hs[i]->kw;
                tiles += (int)((hs[i]->M + R - 1) / R);
            }
            const int min_stages = (h0->sms > 0 && tiles > h0->sms) ? 2 : 3;
            while (gemv_stages > min_stages &&
                   gemv_smem_bytes(sbytes, gemv_stages, n, h0->nb, fp8) > 110 * 1024)
                --gemv_stages;
            gemv_smem = gemv_smem_bytes(sbytes, gemv_stages, n, h0->nb, fp8);
        }
        if (n <= 8 && gemv_smem <= kGemvMaxSmem && gemv_x_fits(n, h0->nb) &&
            !sk_preferred(hs, nh, n)) {
            for (int gidx = 0; gidx < ng; ++gidx) {
                Params p;
                memset(&p, 0, sizeof p);
                int gts = 0, tiles = 0;
                for (int j = 0; j < gsize[gidx]; ++j) {
                    const int idx = groups[gidx][j];
                    const qg_handle *h = hs[idx];
                    gts |= tset_bit(h->type);
                    p.mat[j] = mat_of(h, ys[idx] ? (uint8_t *)ys[idx] + c0 * h->M * (out_f32 ? 4 : 2)
                                                 : nullptr,
                                      res ? res + c0 * h->M : nullptr);
                    p.mat[j].tile_begin = tiles;
                    const int R = kGemvRows / h->kw;
                    tiles += (int)((h->M + R - 1) / R);
                }
                p.nmat = gsize[gidx];
                p.x = xc;
                p.N = n;
                p.K = (int)h0->K;
                p.nb = h0->nb;
                p.ks = 1;
                p.stages = gemv_stages;
                p.xtok = gemv_xtok(h0->nb);
                p.out_f32 = out_f32;
                p.err = h0->err;
                p.swiglu = swiglu ? 1 : 0;  // tiles interleaved: 2 tile + matrix
                const dim3 grid(1u, (unsigned)tiles, 1u);
                cudaError_t le = fault_at("launch") ? cudaErrorLaunchOutOfResources
                                                    : launch_gemv_tset(gts, p, grid, gemv_smem, s);
                if (le != cudaSuccess) {
                    cudaGetLastError();
                    if (flags & QG_FLAG_NO_FALLBACK) {
                        if (fault_at("launch"))
                            return fail(QG_EFAULT_INJECTED, "injected fault: product launch");
                        return cuda_fail(le, "product kernel launch");
                    }
                    const qg_status rs = ref_fallback(p);
                    if (rs != QG_OK) return rs;
                    fail(QG_OK, "fast path launch failed (%s); used the reference kernel",
                         cudaGetErrorName(le));
                }
            }
            continue;
        }
        // Stage x once per layout.
        uint8_t *xl[XL_COUNT] = {nullptr, nullptr, nullptr};
        const qg_handle *xh[XL_COUNT] = {nullptr, nullptr, nullptr};
        for (int i = 0; i < nh; ++i)
            if (!xl[hs[i]->layout]) {
                xl[hs[i]->layout] = hs[i]->xs;
                xh[hs[i]->layout] = hs[i];
            }
        const int G = groups_for(n);
        // N <= 8 with at most 32 (token, super-block) items per CTA: x staged
        // inside qg_sk_kernel (no staging launch; the smallest kw gives the
        // largest per-rank x).  With more items every CTA staging its slice
        // of x costs more than the launch it saves (measured: Q4_K 9728 x 2560
        // N = 16 9.5 vs 7.9 us, Q6_K 2560 x 9728 N = 8 16.2 vs 15.7 us; at
        // N = 2..8 it saves 0.2-1.0 us on the 1024-4096-row Q4_K matrices).
        int kw_min = 8;
        for (int i = 0; i < nh; ++i) kw_min = hs[i]->kw < kw_min ? hs[i]->kw : kw_min;
        const bool xin = sk_xin_ok(n, h0->nb, kw_min);
        if (fault_at("stage")) return fail(QG_EFAULT_INJECTED, "injected fault: staging launch");
        const int64_t tok_stride = (int64_t)h0->nb * kXTok;
        if (!xin) {
            cudaError_t e = launch_stage(xc, n, (int)h0->K, h0->nb, tok_stride, xl[XL_Q4],
                                         xl[XL_Q6], xl[XL_FP4], s);
            if (e != cudaSuccess) return cuda_fail(e, "staging kernel launch");
        }

        const int rows = kSkRows;
        // One launch serves handles of one cluster shape (equal kw): split
        // the group by kw, keeping the call order within each part.
        if (ng == 1) {
            int kws[3], nk = 0;
            for (int i = 0; i < nh; ++i) {
                bool seen = false;
                for (int q = 0; q < nk; ++q) seen = seen || kws[q] == hs[i]->kw;
                if (!seen) kws[nk++] = hs[i]->kw;
            }
            if (nk > 1) {
                ng = nk;
                for (int q = 0; q < nk; ++q) {
                    gsize[q] = 0;
                    for (int i = 0; i < nh; ++i)
                        if (hs[i]->kw == kws[q]) groups[q][gsize[q]++] = i;
                }
            }
        }
        for (int gidx = 0; gidx < ng; ++gidx) {
            Params p;
            memset(&p, 0, sizeof p);
            int tiles = 0, gts = 0;
            int wbytes = 0;
            bool q6 = false;
            for (int j = 0; j < gsize[gidx]; ++j) {
                const qg_handle *h = hs[groups[gidx][j]];
                const int idx = groups[gidx][j];
                p.mat[j] = mat_of(h, ys[idx] ? (uint8_t *)ys[idx] + c0 * h->M * (out_f32 ? 4 : 2)
                                             : nullptr,
                                  res ? res + c0 * h->M : nullptr);
                p.mat[j].tile_begin = tiles;
                tiles += (int)((h->M + rows - 1) / rows);
                gts |= tset_bit(h->type);
                const int wb = sk_wbytes((int)h->type);
                if (wb > wbytes) wbytes = wb;
                q6 = q6 || h->type == QG_Q6_K;
            }
            for (int l = 0; l < XL_COUNT; ++l)
                if (xh[l]) p.xm[l] = xh[l]->xmap[G - 1];
            int stages = 0;
            const int smem = xin ? sk_xin_smem(wbytes, G, q6, h0->nb,
                                               hs[groups[gidx][0]]->kw, &stages, fp8)
                                 : sk_tset_smem(wbytes, G, q6, &stages, fp8);
            p.stages = stages;
            p.xin = xin ? 1 : 0;
            p.x = xc;
            p.nmat = gsize[gidx];
            for (int l = 0; l < XL_COUNT; ++l) p.xs[l] = xl[l];
            p.xs_tok_stride = tok_stride;
            p.N = n;
            p.tok_base = 0;
            p.nb = h0->nb;
            p.ks = hs[groups[gidx][0]]->kw;
            p.K = (int)h0->K;
            p.out_f32 = out_f32;
            p.err = h0->err;
            p.swiglu = swiglu ? 1 : 0;  // tiles interleaved: 2 tile + matrix
            const dim3 grid((unsigned)p.ks, (unsigned)tiles, (unsigned)((n + kTokChunk - 1) / kTokChunk));
            // With no more CTAs than SMs, ask for more than half an SM's shared
            // memory: otherwise both CTAs of a cluster may be placed on one SM
            // and leave another idle (measured: Q4_K 9728 x 2560 at N = 9..16
            // 7.8 us with this, 7.9-9.8 us without, varying from run to run).
            const int64_t ctas = (int64_t)grid.x * grid.y * grid.z;
            const int smem_launch =
                (h0->sms > 0 && ctas <= h0->sms && smem < kSkSpreadSmem) ? kSkSpreadSmem : smem;
            cudaError_t le;
            if (fault_at("launch")) {
                le = cudaErrorLaunchOutOfResources;  // simulated, nothing was launched
            } else {
                le = launch_sk_tset(gts, G, p, grid, smem_launch, s);
            }
            if (le != cudaSuccess) {
                cudaGetLastError();  // launch-time errors are not sticky
                if (flags & QG_FLAG_NO_FALLBACK) {
                    if (fault_at("launch"))
                        return fail(QG_EFAULT_INJECTED, "injected fault: product launch");
                    return cuda_fail(le, "product kernel launch");
                }
                const qg_status rs = ref_fallback(p);
                if (rs != QG_OK) return rs;
                fail(QG_OK, "fast path launch failed (%s); used the reference kernel",
                     cudaGetErrorName(le));
            }
        }
    }
    return QG_OK;
}

// Plan of a qg_tc_kernel launch over `tiles` row tiles, n tokens and nb
// super-blocks: token tiles of 8 G tokens (G even, <= 16) and K slices ks
// (<= 8; <= nb), one CTA per SM.  A K split costs a cluster reduction at the
// end (rank partials through distributed shared memory) and is bounded by
// how many clusters of ks CTAs the GPU holds at once (a cluster lives in one
// GPC, so 7 or 8 CTA clusters leave SMs idle); a token split costs a second
// decode of the weights.  Estimated time: waves x (super-blocks per CTA x
// the time of one, about 1.2 us on GB300 and nearly independent of the tile
// width, + the epilogue, about 4 us with a cluster reduction and 2 us
// without); ties go to the wider tile, then to the smaller K split.
constexpr int kNumSMs = 152;
struct TcPlan {
    int G, zc, ks;
};
static TcPlan tc_plan(int tiles, int n, int nb)
{
    TcPlan best = {0, 0, 0};
    double best_t = 1e30;
    for (int w = 64; w <= kTcTok; w *= 2) {  // token tile width
        if (w == 64 && n <= 32) continue;
        const int nt = n < w ? n : w;
        const int G = 2 * ((nt + 15) / 16);
        const int zc = (n + 8 * G - 1) / (8 * G);
        const int clusters = tiles * zc;
        for (int ks = 8; ks >= 1; --ks) {
            if (ks > nb) continue;
            int cap = tc_cluster_capacity(ks);
            if (cap <= 0) cap = kNumSMs / ks;
            const int waves = (clusters + cap - 1) / cap;
            const double t =
                waves * ((double)((nb + ks - 1) / ks) * 1.2 + (ks > 1 ? 4.0 : 2.0));
            if (t < best_t - 1e-9 || (t <= best_t + 1e-9 && 8 * G >= 8 * best.G)) {
                best_t = t;
                best = {G, zc, ks};
            }
        }
    }
    return best;
}

// Ring depths of qg_tc_kernel: x ring 2..3 slots, weight ring 2..4 slots,
// within the shared-memory budget (x first: it is the larger copy).
static bool tc_stages(int T, int G, int *ws, int *xs)
{
    for (int x = 3; x >= 2; --x)
        for (int w = 4; w >= 2; --w)
            if (tc_smem_bytes(T, G, w, x) <= kTcMaxSmem && (x == 2 || w >= 3)) {
                *ws = w;
                *xs = x;
                return true;
            }
    return false;
}

static bool tc_type(qg_type t) { return t == QG_Q4_K || t == QG_Q5_K || t == QG_Q6_K; }

// K-quant handles sharing x, N >= 33, on the tensor core (qg_tc_kernel): x
// staged once per chunk by qg_stage_tc_kernel, one product launch per weight
// format (the matrices of a launch share its K split).
qg_status run_product_tc(qg_handle *const *hs, int nh, const __half *x, int64_t N,
                         void *const *ys, const __half *res, int out_f32, cudaStream_t s)
{
    const qg_handle *h0 = hs[0];
    uint32_t flags = 0;
    int max_tokens = h0->max_tokens;
    for (int i = 0; i < nh; ++i) {
        flags |= hs[i]->flags;
        if (hs[i]->max_tokens < max_tokens) max_tokens = hs[i]->max_tokens;
    }
    const int nb = h0->nb;
    const int64_t chunk_stride = tc_chunk_bytes(nb);
    for (int64_t c0 = 0; c0 < N; c0 += max_tokens) {
        const int n = (int)((N - c0) < max_tokens ? (N - c0) : max_tokens);
        const __half *xc = x + c0 * h0->K;
        if (fault_at("stage")) return fail(QG_EFAULT_INJECTED, "injected fault: staging launch");
        cudaError_t e = launch_stage_tc4(xc, n, (int)h0->K, nb, chunk_stride, h0->xs, s);
        if (e != cudaSuccess) return cuda_fail(e, "staging kernel launch");

        // One launch per format, except that Q4_K and Q6_K matrices of one
        // call (the QKV triple) share a launch of the mixed kernel.
        auto cls = [](qg_type ty) { return ty == QG_Q5_K ? 1 : 0; };
        bool done[3] = {false, false, false};
        for (int a = 0; a < nh; ++a) {
            if (done[a]) continue;
            const qg_type t = hs[a]->type;
            bool mixed = false;
            for (int j = a; j < nh; ++j)
                mixed = mixed || (!done[j] && cls(hs[j]->type) == cls(t) && hs[j]->type != t);
            Params p;
            memset(&p, 0, sizeof p);
            int tiles = 0;
            for (int j = a; j < nh; ++j) {
                if (done[j] || (mixed ? cls(hs[j]->type) != cls(t) : hs[j]->type != t)) continue;
                done[j] = true;
                const qg_handle *h = hs[j];
                Mat &m = p.mat[p.nmat++];
                m = mat_of(h, (uint8_t *)ys[j] + c0 * h->M * (out_f32 ? 4 : 2),
                           res ? res + c0 * h->M : nullptr);
                m.tile_begin = tiles;
                tiles += (int)((h->M + kTcRows - 1) / kTcRows);
            }
            const TcPlan pl = tc_plan(tiles, n, nb);
            const int G = pl.G, zc = pl.zc, ks = pl.ks;  // MMA N = 8 G, a multiple of 16
            p.xs[XL_TC4] = h0->xs;
            p.xs_tok_stride = chunk_stride;
            p.x = xc;
            p.N = n;
            p.tok_base = 0;
            p.K = (int)h0->K;
            p.nb = nb;
            p.ks = ks;
            p.out_f32 = out_f32;
            p.err = h0->err;
            int ws = 0, xs = 0, ws6 = 0, xs6 = 0;
            const int T = (t == QG_Q4_K) ? T_Q4K : (t == QG_Q5_K) ? T_Q5K : T_Q6K;
            cudaError_t le = cudaErrorInvalidValue;
            // mixed: ring depths both formats' layouts fit, the larger layout's bytes
            const bool staged = mixed ? (tc_stages(T_Q4K, G, &ws, &xs) &&
                                         tc_stages(T_Q6K, G, &ws6, &xs6))
                                      : tc_stages(T, G, &ws, &xs);
            if (staged) {
                if (mixed) {
                    ws = ws < ws6 ? ws : ws6;
                    xs = xs < xs6 ? xs : xs6;
                }
                p.stages = ws;
                p.xstages = xs;
                int smem = tc_smem_bytes(T, G, ws, xs);
                if (mixed) {
                    const int a4 = tc_smem_bytes(T_Q4K, G, ws, xs), a6 = tc_smem_bytes(T_Q6K, G, ws, xs);
                    smem = a4 > a6 ? a4 : a6;
                }
                const dim3 grid((unsigned)ks, (unsigned)tiles, (unsigned)zc);
                if (fault_at("launch"))
                    le = cudaErrorLaunchOutOfResources;
                else if (mixed)
                    le = launch_tc_q4k_q6k(G, p, grid, smem, s);
                else if (T == T_Q4K)
                    le = launch_tc_q4k(G, p, grid, smem, s);
                else if (T == T_Q5K)
                    le = launch_tc_q5k(G, p, grid, smem, s);
                else
                    le = launch_tc_q6k(G, p, grid, smem, s);
            }
            if (le != cudaSuccess) {
                cudaGetLastError();
                if (flags & QG_FLAG_NO_FALLBACK) {
                    if (fault_at("launch"))
                        return fail(QG_EFAULT_INJECTED, "injected fault: product launch");
                    return cuda_fail(le, "product kernel launch");
                }
                for (int j = 0; j < p.nmat; ++j) {
                    cudaError_t re = launch_ref_gemv(p.mat[j], (int)h0->K, xc, n, out_f32, s);
                    if (re != cudaSuccess) return cuda_fail(re, "reference kernel launch");
                }
                fail(QG_OK, "fast path launch failed (%s); used the reference kernel",
                     cudaGetErrorName(le));
            }
        }
    }
    return QG_OK;
}

// Every product call: Q4_K, Q5_K and Q6_K handles of calls with N >= 33
// (prefill chunks; rows need not keep their bits across N there) go to the
// tcgen05 engine
// unless QG_FLAG_MMA_SYNC_PREFILL is set; everything else runs on the
// mma.sync kernels.
qg_status run_product(qg_handle *const *hs, int nh, const __half *x, int64_t N, void *const *ys,
                      const __half *res, int out_f32, cudaStream_t s, bool swiglu = false)
{
    g_err.clear();
    uint32_t flags = 0;
    for (int i = 0; i < nh; ++i) flags |= hs[i]->flags;
    qg_handle *tc[3], *mm[3];
    void *ytc[3], *ymm[3];
    int ntc = 0, nmm = 0;
    for (int i = 0; i < nh; ++i) {
        if (tc_type(hs[i]->type) && N >= kTcMinN && !(flags & QG_FLAG_MMA_SYNC_PREFILL) &&
            !(flags & QG_FLAG_FORCE_REFERENCE) && !swiglu) {
            tc[ntc] = hs[i];
            ytc[ntc++] = ys[i];
        } else {
            mm[nmm] = hs[i];
            ymm[nmm++] = ys[i];
        }
    }
    qg_status st = QG_OK;
    std::string note;
    if (ntc) {
        st = run_product_tc(tc, ntc, x, N, ytc, res, out_f32, s);
        if (st != QG_OK) return st;
        note = g_err;
    }
    if (nmm) {
        st = run_product_mma(mm, nmm, x, N, ymm, res, out_f32, s, swiglu);
        if (st != QG_OK) return st;
        if (note.empty()) note = g_err;
    }
    g_err = note;
    if (flags & QG_FLAG_DEBUG_SYNC) {
        cudaError_t e = cudaStreamSynchronize(s);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "debug synchronize");
        for (int i = 0; i < nh; ++i) {
            unsigned int w = 0;
            e = cudaMemcpy(&w, hs[i]->err, sizeof w, cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return cuda_fail(e, "error word read");
            if (w) return fail(QG_ECUDA, "kernel reported a bounded-wait timeout (0x%x)", w);
        }
    }
    return QG_OK;
}

qg_status check_run_args(const qg_handle *h, const void *x, int64_t N, const void *y, qg_out ydt)
{
    if (!h) return fail(QG_EINVAL, "null handle");
    if (!x || !y) return fail(QG_EINVAL, "null x or y");
    if (N < 1) return fail(QG_EINVAL, "N must be >= 1 (got %lld)", (long long)N);
    if (N > (int64_t)1 << 24) return fail(QG_EUNSUPPORTED, "N too large");
    if (ydt != QG_OUT_F16 && ydt != QG_OUT_F32) return fail(QG_EINVAL, "bad output type");
    if (!aligned(x, 16)) return fail(QG_EALIGN, "x must be 16-byte aligned");
    if (!aligned(y, ydt == QG_OUT_F32 ? 4 : 2)) return fail(QG_EALIGN, "y misaligned");
    return QG_OK;
}

// Argument checks of a weight matrix, before any CUDA call (qgemv_create and
// the allocation-free entry point).
qg_status check_matrix(qg_type t, int64_t M, int64_t K, const void *w_dev, const void *scales_dev,
                       float global_scale)
{
    if (!type_known(t)) return fail(QG_EUNSUPPORTED, "unknown weight type %d", (int)t);
    if (M < 1) return fail(QG_EINVAL, "M must be >= 1");
    if (K < 256 || K % 256 != 0) return fail(QG_EUNSUPPORTED, "K must be a positive multiple of 256");
    if (M > (int64_t)1 << 30 || K > (int64_t)1 << 24) return fail(QG_EUNSUPPORTED, "shape too large");
    if (!w_dev) return fail(QG_EINVAL, "null weight pointer");
    if (!aligned(w_dev, 16)) return fail(QG_EALIGN, "weights must be 16-byte aligned");
    if (t == QG_NVFP4_W4A16) {
        if (!scales_dev) return fail(QG_EINVAL, "NVFP4 needs the e4m3 scale array");
        if (!aligned(scales_dev, 16)) return fail(QG_EALIGN, "scales must be 16-byte aligned");
        if (!std::isfinite(global_scale)) return fail(QG_EINVAL, "global scale must be finite");
    }
    if (t == QG_FP8_E4M3) {
        if (!scales_dev) return fail(QG_EINVAL, "FP8 needs the bf16 block-scale array");
        if (!aligned(scales_dev, 16)) return fail(QG_EALIGN, "scales must be 16-byte aligned");
        if (K > kFp8MaxK) return fail(QG_EUNSUPPORTED, "FP8 supports K up to %d", kFp8MaxK);
    }
    const int64_t rows_needed = (M + 63) / 64;
    if (rows_needed > 65535) return fail(QG_EUNSUPPORTED, "too many rows for one grid");
    return QG_OK;
}

// Everything of a handle that needs no device allocation: the plan (K
// slices, layout), the device's SM count and the tensor maps (encoded on the
// host) of the weights and of the given staging buffer xs; err is the device
// error word the kernels report to.
qg_status init_handle(qg_handle *h, qg_type t, int64_t M, int64_t K, const void *w_dev,
                      const void *scales_dev, float global_scale, uint32_t flags, int max_tokens,
                      uint8_t *xs, unsigned int *err)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const int nb = (int)(K / 256);
    h->type = t;
    h->M = M;
    h->K = K;
    h->nb = nb;
    h->w = (const uint8_t *)w_dev;
    h->sc = (const uint8_t *)scales_dev;
    h->gscale = (t == QG_NVFP4_W4A16) ? global_scale : 1.0f;
    h->row_bytes = qgemv_row_bytes(t, K);
    // NVFP4: e4m3 bytes per row; FP8: bf16 bytes per 128-row block
    h->sc_row_bytes = (t == QG_NVFP4_W4A16) ? K / 16 : (t == QG_FP8_E4M3) ? (K / 128) * 2 : 0;
    h->w_bytes = h->row_bytes * M;
    h->flags = flags;
    h->max_tokens = max_tokens;
    h->kw = plan_kw(M, nb);
    h->layout = layout_of(t);
    h->device = dev;
    h->xs = xs;
    h->err = err;
    if (cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        h->sms = 0;
    }
    if (t == QG_FP8_E4M3) {
        // planes of 128 codes (one bf16 scale block wide), 128-byte swizzle
        const int R = kGemvRows / h->kw;
        bool ok = encode_blocks(&h->tmw, w_dev, h->row_bytes, M, 128, R, 2 * h->kw, true);
        if (ok) ok = encode_blocks(&h->tmw1, w_dev, h->row_bytes, M, 128, kSkRows, 2, true);
        if (!ok) return fail(QG_ECUDA, "tensor map encoding failed");
    } else if (t != QG_Q6_K) {
        const int bb = (t == QG_NVFP4_W4A16) ? 128 : block_bytes(t);
        const int R = kGemvRows / h->kw;
        bool ok = encode_blocks(&h->tmw, w_dev, h->row_bytes, M, bb, R, h->kw);
        if (ok && t == QG_NVFP4_W4A16)
            ok = encode_blocks(&h->tms, scales_dev, h->sc_row_bytes, M, 16, R, h->kw);
        if (ok) ok = encode_blocks(&h->tmw1, w_dev, h->row_bytes, M, bb, kSkRows, 1);
        if (ok && t == QG_NVFP4_W4A16)
            ok = encode_blocks(&h->tms1, scales_dev, h->sc_row_bytes, M, 16, kSkRows, 1);
        if (!ok) return fail(QG_ECUDA, "tensor map encoding failed");
    }
    for (int G = 1; G <= 4; ++G)
        if (!encode_staged(&h->xmap[G - 1], xs, nb, max_tokens, 8 * G))
            return fail(QG_ECUDA, "tensor map encoding failed (staging buffer)");
    return QG_OK;
}

}  // namespace

namespace qg {
// The path of qgemv_run with caller-provided device memory and no handle
// (qgemv_run_noalloc, qg_noalloc.cu): the matrix is checked as qgemv_create
// checks it, a handle is filled on the stack (plan and host-encoded tensor
// maps; nothing is allocated), the staged x goes to the scratch memory that
// get_scratch() returns (at most scratch_bytes; called only after every
// argument check passed) in chunks of up to 32 tokens, and the kernels report
// bounded-wait timeouts to the word at scratch + err_offset.  Q4_K calls with N >= 33 stay on the
// mma.sync kernels (as with QG_FLAG_MMA_SYNC_PREFILL), so every row keeps
// the bits of an N <= 32 call.
qg_status run_with_scratch(qg_type t, int64_t M, int64_t K, const void *w_dev,
                           const void *scales_dev, float global_scale, const void *x, int64_t N,
                           void *y, qg_out ydt, cudaStream_t s, uint8_t *(*get_scratch)(),
                           size_t scratch_bytes, size_t err_offset)
{
    g_err.clear();
    qg_status st = check_matrix(t, M, K, w_dev, scales_dev, global_scale);
    if (st != QG_OK) return st;
    if (!x || !y) return fail(QG_EINVAL, "null x or y");
    if (N < 1) return fail(QG_EINVAL, "N must be >= 1 (got %lld)", (long long)N);
    if (N > (int64_t)1 << 24) return fail(QG_EUNSUPPORTED, "N too large");
    if (ydt != QG_OUT_F16 && ydt != QG_OUT_F32) return fail(QG_EINVAL, "bad output type");
    if (!aligned(x, 16)) return fail(QG_EALIGN, "x must be 16-byte aligned");
    if (!aligned(y, ydt == QG_OUT_F32 ? 4 : 2)) return fail(QG_EALIGN, "y misaligned");
    const size_t tok_bytes = (size_t)(K / 256) * kXTok;
    const size_t fit = scratch_bytes / tok_bytes;
    if (fit < 1)
        return fail(QG_EUNSUPPORTED,
                    "K too large: one token's staged x (%zu bytes) exceeds the %zu-byte scratch "
                    "array",
                    tok_bytes, scratch_bytes);
    const int chunk = (int)(fit < 32 ? fit : 32);
    // Every argument has been checked: now the device.
    uint8_t *scratch = get_scratch();
    if (!scratch) return QG_ECUDA;
    unsigned int *err_word = reinterpret_cast<unsigned int *>(scratch + err_offset);
    uint32_t flags = QG_FLAG_MMA_SYNC_PREFILL;
    if (env_on("QGEMV_FORCE_REFERENCE")) flags |= QG_FLAG_FORCE_REFERENCE;
    if (env_on("QGEMV_DEBUG_SYNC")) flags |= QG_FLAG_DEBUG_SYNC;
    qg_handle h = {};
    st = init_handle(&h, t, M, K, w_dev, scales_dev, global_scale, flags, chunk, scratch, err_word);
    if (st != QG_OK) return st;
    qg_handle *hp = &h;
    void *ys[1] = {y};
    return run_product(&hp, 1, (const __half *)x, N, ys, nullptr, ydt == QG_OUT_F32, s);
}

// Sets the calling thread's qgemv_last_error text (used by qg_noalloc.cu).
void set_last_error(const char *msg) { g_err = msg; }
}  // namespace qg

namespace {

int call_nh(int kind) { return kind == QG_CALL_PAIR ? 2 : kind == QG_CALL_TRIPLE ? 3 : 1; }

qg_status check_call(const qg_call &c)
{
    if (c.kind < QG_CALL_RUN || c.kind > QG_CALL_TRIPLE)
        return fail(QG_EINVAL, "bad chain call kind %d", (int)c.kind);
    const int nh = call_nh(c.kind);
    const qg_out ydt = c.kind == QG_CALL_RUN_ADD ? QG_OUT_F16 : (qg_out)c.out_dtype;
    if (c.kind == QG_CALL_RUN_ADD && c.out_dtype != QG_OUT_F16)
        return fail(QG_EINVAL, "a residual call writes fp16");
    for (int i = 0; i < nh; ++i) {
        const qg_status st = check_run_args(c.h[i], c.x, c.N, c.y[i], ydt);
        if (st != QG_OK) return st;
        if (c.h[i]->K != c.h[0]->K) return fail(QG_EINVAL, "the handles of a call must share K");
        for (int j = 0; j < i; ++j)
            if (c.y[i] == c.y[j]) return fail(QG_EINVAL, "the outputs of a call must differ");
    }
    if (c.kind == QG_CALL_RUN_ADD) {
        if (!c.residual) return fail(QG_EINVAL, "null residual");
        if (!aligned(c.residual, 2)) return fail(QG_EALIGN, "residual misaligned");
    }
    return QG_OK;
}

qg_status run_call(const qg_call &c, cudaStream_t s)
{
    void *sv = (void *)s;
    switch (c.kind) {
    case QG_CALL_RUN: return qgemv_run(c.h[0], c.x, c.N, c.y[0], (qg_out)c.out_dtype, sv);
    case QG_CALL_RUN_ADD: return qgemv_run_add(c.h[0], c.x, c.N, c.residual, c.y[0], sv);
    case QG_CALL_PAIR:
        return qgemv_pair_run(c.h[0], c.h[1], c.x, c.N, c.y[0], c.y[1], (qg_out)c.out_dtype, sv);
    default:
        return qgemv_triple_run(c.h[0], c.h[1], c.h[2], c.x, c.N, c.y[0], c.y[1], c.y[2],
                                (qg_out)c.out_dtype, sv);
    }
}

// Calls the persistent chain kernel serves: N <= 8 with x in shared memory,
// Q4_K / Q6_K handles on the chain's device, default arithmetic flags.
bool chain_ok(const qg_chain *ch, const qg_call &c)
{
    if (c.N > 8 || !gemv_x_fits(c.N, c.h[0]->nb)) return false;
    for (int i = 0; i < call_nh(c.kind); ++i) {
        const qg_handle *h = c.h[i];
        if (h->type != QG_Q4_K && h->type != QG_Q6_K) return false;
        if (h->flags & (QG_FLAG_FORCE_REFERENCE | QG_FLAG_DEBUG_SYNC)) return false;
        if (h->device != ch->device) return false;
    }
    return !env_on("QGEMV_FORCE_REFERENCE") && !env_on("QGEMV_DEBUG_SYNC");
}

// One persistent launch for calls[0 .. n-1] (all chain_ok).
qg_status launch_chain_calls(qg_chain *ch, const qg_call *calls, int n, cudaStream_t s)
{
    ChainParams p;
    memset(&p, 0, sizeof p);
    int nm = 0, xbytes = 0, maxtiles = 0;
    bool one = true;
    for (int c = 0; c < n; ++c) {
        const qg_call &q = calls[c];
        ChainCall &cl = p.call[c];
        const int nh = call_nh(q.kind);
        cl.mat0 = nm;
        cl.nmat = nh;
        int tiles = 0, slot = 0;
        for (int i = 0; i < nh; ++i) {
            const qg_handle *h = q.h[i];
            Mat m = mat_of(h, q.y[i], q.kind == QG_CALL_RUN_ADD ? (const __half *)q.residual
                                                                : nullptr);
            m.tile_begin = tiles;
            const int R = kGemvRows / h->kw;
            tiles += (int)((h->M + R - 1) / R);
            p.mat[nm++] = m;
            const int b = gemv_stage_bytes_host(h->type, h->kw);
            slot = b > slot ? b : slot;
        }
        const qg_handle *h0 = q.h[0];
        cl.tiles = tiles;
        cl.slot_bytes = slot;
        cl.N = (int)q.N;
        cl.K = (int)h0->K;
        cl.nb = h0->nb;
        cl.xtok = gemv_xtok(h0->nb);
        cl.out_f32 = (q.kind != QG_CALL_RUN_ADD && q.out_dtype == QG_OUT_F32) ? 1 : 0;
        cl.x = (const __half *)q.x;
        const int xb = (int)q.N * cl.xtok;
        xbytes = xb > xbytes ? xb : xbytes;
        maxtiles = tiles > maxtiles ? tiles : maxtiles;
        one = one && q.N == 1;
    }
    // Each side gets half of the CTA's shared memory; its ring is what the
    // barriers, the largest staged x and the partials leave, re-cut per call
    // into as many slots of the call's largest stage as fit.
    const int side = (chain_max_smem() / 2) & ~1023;
    const int ring = side - chain_side_bytes(0, xbytes);
    int ring_used = 0;
    for (int c = 0; c < n; ++c) {
        ChainCall &cl = p.call[c];
        int st = ring / cl.slot_bytes;
        st = st < kChainSlots ? st : kChainSlots;
        if (st < 2) return fail(QG_EUNSUPPORTED, "chain does not fit shared memory");
        cl.stages = st;
        ring_used = st * cl.slot_bytes > ring_used ? st * cl.slot_bytes : ring_used;
    }
    const int smem = 2 * side;
    const int per_sm = chain_ctas_per_sm(smem, one);
    if (per_sm < 1 || ch->sms < 1) return fail(QG_EUNSUPPORTED, "chain kernel does not fit an SM");
    // Every CTA must be resident at once (they wait for one another): one per
    // SM, each side a virtual CTA (tiles t and t + grid share an SM).
    int grid = per_sm * ch->sms;
    grid = grid < maxtiles ? grid : maxtiles;
    p.ncalls = n;
    p.side_bytes = side;
    p.xoff = kChainHdr + ring_used;
    p.redoff = p.xoff + xbytes;
    p.err = ch->words + 2;
    p.ctr = ch->words;
    p.hold_publish = fault_at("chain_publish") ? 1 : 0;
    const cudaError_t e = launch_chain(p, grid, smem, one, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail(e, "chain kernel launch");
    }
    return QG_OK;
}

}  // namespace

extern "C" {

int64_t qgemv_row_bytes(qg_type t, int64_t K)
{
    if (!type_known(t) || K < 256 || K % 256 != 0) return -1;
    if (t == QG_NVFP4_W4A16) return K / 2;
    if (t == QG_FP8_E4M3) return K;
    return (K / 256) * block_bytes(t);
}

const char *qgemv_last_error(void) { return g_err.c_str(); }

const char *qgemv_describe(void)
{
    static thread_local std::string d;
    const char *fi = getenv("QGEMV_FAULT_INJECT");
    d = std::string("qgemv: GB300 (sm_103a) fused 4-bit GEMV; formats Q4_K=12 Q5_K=13 Q6_K=14 "
                    "NVFP4_W4A16=256 FP8_E4M3=257; flags FORCE_REFERENCE=1 DEBUG_SYNC=2 NO_FALLBACK=4 "
                    "MMA_SYNC_PREFILL=8; ") +
        "env QGEMV_FORCE_REFERENCE=" + (env_on("QGEMV_FORCE_REFERENCE") ? "1" : "0") +
        " QGEMV_DEBUG_SYNC=" + (env_on("QGEMV_DEBUG_SYNC") ? "1" : "0") +
        " QGEMV_FAULT_INJECT=" + (fi ? fi : "") +
        "; staging " + std::to_string(kXTok) + " B per token per 256 columns; " +
        "K slices kw in {1,2,4,8} fixed by (M, K); Q4_K/Q5_K/Q6_K N >= 33 on the tcgen05 engine "
        "unless MMA_SYNC_PREFILL";
    return d.c_str();
}

qg_status qgemv_create(qg_handle **out, qg_type t, int64_t M, int64_t K, const void *w_dev,
                       const void *scales_dev, float global_scale, const qg_opts *opts)
{
    if (!out) return fail(QG_EINVAL, "null output handle pointer");
    *out = nullptr;
    qg_status st = check_matrix(t, M, K, w_dev, scales_dev, global_scale);
    if (st != QG_OK) return st;
    const int max_tokens = (opts && opts->max_tokens > 0) ? opts->max_tokens : 128;
    if (max_tokens > (1 << 20)) return fail(QG_EUNSUPPORTED, "max_tokens too large");
    uint32_t flags = opts ? opts->flags : 0u;
    if (env_on("QGEMV_FORCE_REFERENCE")) flags |= QG_FLAG_FORCE_REFERENCE;
    if (env_on("QGEMV_DEBUG_SYNC")) flags |= QG_FLAG_DEBUG_SYNC;
    if (fault_at("create")) return fail(QG_EFAULT_INJECTED, "injected fault: create");

    qg_handle *h = new (std::nothrow) qg_handle();
    if (!h) return fail(QG_ENOMEM, "host allocation failed");
    // staged x: [token][super-block][576] for the mma.sync kernels; K-quant
    // prefill chunks use the same buffer as [128-token chunk][super-block][16
    // groups][kTcXBlk] (qg_tc_kernel)
    const int nb = (int)(K / 256);
    size_t xs_bytes = (size_t)max_tokens * nb * kXTok;
    if (tc_type(t)) {
        const size_t tc = (size_t)((max_tokens + kTcTok - 1) / kTcTok) * tc_chunk_bytes(nb);
        if (tc > xs_bytes) xs_bytes = tc;
    }
    uint8_t *xs = nullptr;
    cudaError_t e = cudaMalloc((void **)&xs, xs_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return fail(QG_ENOMEM, "staging buffer allocation of %zu bytes failed", xs_bytes);
    }
    unsigned int *err = nullptr;
    e = cudaMalloc((void **)&err, sizeof(unsigned int));
    if (e == cudaSuccess) e = cudaMemset(err, 0, sizeof(unsigned int));
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (err) cudaFree(err);
        cudaFree(xs);
        delete h;
        return fail(QG_ENOMEM, "error word allocation failed");
    }
    st = init_handle(h, t, M, K, w_dev, scales_dev, global_scale, flags, max_tokens, xs, err);
    if (st != QG_OK) {
        cudaFree(xs);
        cudaFree(err);
        delete h;
        return st;
    }
    h->owns_buffers = true;
    *out = h;
    return QG_OK;
}

void qgemv_destroy(qg_handle *h)
{
    if (!h) return;
    if (h->owns_buffers && h->xs) cudaFree(h->xs);
    if (h->owns_buffers && h->err) cudaFree(h->err);
    if (h->hx) cudaFree(h->hx);
    if (h->hy) cudaFree(h->hy);
    delete h;
}

qg_status qgemv_run(qg_handle *h, const void *x, int64_t N, void *y, qg_out ydt, void *stream)
{
    qg_status st = check_run_args(h, x, N, y, ydt);
    if (st != QG_OK) return st;
    void *ys[1] = {y};
    return run_product(&h, 1, (const __half *)x, N, ys, nullptr, ydt == QG_OUT_F32,
                       (cudaStream_t)stream);
}

qg_status qgemv_run_add(qg_handle *h, const void *x, int64_t N, const void *residual, void *y,
                        void *stream)
{
    qg_status st = check_run_args(h, x, N, y, QG_OUT_F16);
    if (st != QG_OK) return st;
    if (!residual) return fail(QG_EINVAL, "null residual");
    if (!aligned(residual, 2)) return fail(QG_EALIGN, "residual misaligned");
    void *ys[1] = {y};
    return run_product(&h, 1, (const __half *)x, N, ys, (const __half *)residual, 0,
                       (cudaStream_t)stream);
}

qg_status qgemv_pair_run(qg_handle *a, qg_handle *b, const void *x, int64_t N, void *ya,
                         void *yb, qg_out ydt, void *stream)
{
    qg_status st = check_run_args(a, x, N, ya, ydt);
    if (st != QG_OK) return st;
    st = check_run_args(b, x, N, yb, ydt);
    if (st != QG_OK) return st;
    if (a->K != b->K) return fail(QG_EINVAL, "pair handles must share K");
    if (ya == yb) return fail(QG_EINVAL, "pair outputs must differ");
    qg_handle *hs[2] = {a, b};
    void *ys[2] = {ya, yb};
    return run_product(hs, 2, (const __half *)x, N, ys, nullptr, ydt == QG_OUT_F32,
                       (cudaStream_t)stream);
}

qg_status qgemv_triple_run(qg_handle *a, qg_handle *b, qg_handle *c, const void *x, int64_t N,
                           void *ya, void *yb, void *yc, qg_out ydt, void *stream)
{
    qg_status st = check_run_args(a, x, N, ya, ydt);
    if (st == QG_OK) st = check_run_args(b, x, N, yb, ydt);
    if (st == QG_OK) st = check_run_args(c, x, N, yc, ydt);
    if (st != QG_OK) return st;
    if (a->K != b->K || a->K != c->K) return fail(QG_EINVAL, "triple handles must share K");
    if (ya == yb || ya == yc || yb == yc) return fail(QG_EINVAL, "triple outputs must differ");
    qg_handle *hs[3] = {a, b, c};
    void *ys[3] = {ya, yb, yc};
    return run_product(hs, 3, (const __half *)x, N, ys, nullptr, ydt == QG_OUT_F32,
                       (cudaStream_t)stream);
}

qg_status qgemv_pair_swiglu_run(qg_handle *gate, qg_handle *up, const void *x, int64_t N,
                                void *h, qg_out hdt, void *stream)
{
    qg_status st = check_run_args(gate, x, N, h, hdt);
    if (st != QG_OK) return st;
    if (!up) return fail(QG_EINVAL, "null up handle");
    if (gate == up) return fail(QG_EINVAL, "gate and up must be different handles");
    if (gate->M != up->M || gate->K != up->K)
        return fail(QG_EINVAL, "gate and up must have the same shape");
    if (gate->type != up->type)
        return fail(QG_EUNSUPPORTED, "gate and up must have the same weight format");
    qg_handle *hs[2] = {gate, up};
    void *ys[2] = {h, nullptr};
    return run_product(hs, 2, (const __half *)x, N, ys, nullptr, hdt == QG_OUT_F32,
                       (cudaStream_t)stream, true);
}

qg_status qgemv_run_host(qg_handle *h, const void *x_host, int64_t N, void *y_host, qg_out ydt,
                         void *stream)
{
    if (!h) return fail(QG_EINVAL, "null handle");
    if (!x_host || !y_host) return fail(QG_EINVAL, "null host buffer");
    if (N < 1) return fail(QG_EINVAL, "N must be >= 1");
    if (ydt != QG_OUT_F16 && ydt != QG_OUT_F32) return fail(QG_EINVAL, "bad output type");
    cudaStream_t s = (cudaStream_t)stream;
    const size_t xb = (size_t)N * h->K * 2;
    const size_t yb = (size_t)N * h->M * (ydt == QG_OUT_F32 ? 4 : 2);
    cudaError_t e;
    if (h->hx_cap < xb) {
        if (h->hx) cudaFree(h->hx);
        h->hx = nullptr;
        h->hx_cap = 0;
        e = cudaMalloc(&h->hx, xb);
        if (e != cudaSuccess) return fail(QG_ENOMEM, "device x buffer allocation failed");
        h->hx_cap = xb;
    }
    if (h->hy_cap < yb) {
        if (h->hy) cudaFree(h->hy);
        h->hy = nullptr;
        h->hy_cap = 0;
        e = cudaMalloc(&h->hy, yb);
        if (e != cudaSuccess) return fail(QG_ENOMEM, "device y buffer allocation failed");
        h->hy_cap = yb;
    }
    e = cudaMemcpyAsync(h->hx, x_host, xb, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "copy of x to the device");
    qg_status st = qgemv_run(h, h->hx, N, h->hy, ydt, stream);
    if (st != QG_OK) return st;
    e = cudaMemcpyAsync(y_host, h->hy, yb, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "copy of y to the host");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    return QG_OK;
}

qg_status qgemv_dequantize(qg_handle *h, float *w_out, void *stream)
{
    if (!h) return fail(QG_EINVAL, "null handle");
    if (!w_out) return fail(QG_EINVAL, "null output");
    if (!aligned(w_out, 4)) return fail(QG_EALIGN, "output must be 4-byte aligned");
    Mat m = mat_of(h, nullptr, nullptr);
    // The product kernels' own decoders; FORCE_REFERENCE selects the simple
    // per-element reference decoder instead.
    cudaError_t e = (h->flags & QG_FLAG_FORCE_REFERENCE)
                        ? launch_dequant(m, (int)h->K, w_out, (cudaStream_t)stream)
                        : launch_dequant_fast(m, (int)h->K, w_out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "dequantize kernel launch");
    if (h->flags & QG_FLAG_DEBUG_SYNC) {
        e = cudaStreamSynchronize((cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "debug synchronize");
    }
    return QG_OK;
}

qg_status qgemv_device_status(qg_handle *h, uint32_t *flags_out, int clear)
{
    // NULL: the allocation-free entry point's error word on the current device.
    unsigned int *word = h ? h->err : noalloc_error_word();
    if (!word) return QG_ECUDA;
    unsigned int w = 0;
    cudaError_t e = cudaMemcpy(&w, word, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "error word read");
    if (clear && w) {
        e = cudaMemset(word, 0, sizeof(unsigned int));
        if (e != cudaSuccess) return cuda_fail(e, "error word reset");
    }
    if (flags_out) *flags_out = w;
    return QG_OK;
}

static bool gv_x_ok(const qg_handle *h, int64_t n)
{
    return gemv_smem_bytes(gemv_stage_bytes_host(h->type, h->kw), kGemvStagesMax, (int)n, h->nb) <=
               kGemvMaxSmem &&
           gemv_x_fits(n, h->nb) && !sk_preferred(&h, 1, n);
}

qg_status qgemv_plan_info(const qg_handle *h, int64_t N, int32_t *ksplit, int32_t *rows_cta,
                          int32_t *launches)
{
    if (!h) return fail(QG_EINVAL, "null handle");
    if (N < 1) return fail(QG_EINVAL, "N must be >= 1");
    const int64_t chunks = (N + h->max_tokens - 1) / h->max_tokens;
    const int64_t nfirst = N < h->max_tokens ? N : h->max_tokens;
    if (ksplit) *ksplit = h->kw;
    if (tc_type(h->type) && N >= kTcMinN && !(h->flags & QG_FLAG_MMA_SYNC_PREFILL) &&
        !(h->flags & QG_FLAG_FORCE_REFERENCE)) {
        // qg_tc_kernel: 128 rows per CTA, one staging launch per chunk
        const int tiles = (int)((h->M + kTcRows - 1) / kTcRows);
        if (ksplit) *ksplit = tc_plan(tiles, (int)nfirst, h->nb).ks;
        if (rows_cta) *rows_cta = kTcRows;
        if (launches) *launches = (int32_t)(2 * chunks);
        return QG_OK;
    }
    if (rows_cta) *rows_cta = kSkRows;
    if (launches) {
        int64_t l = 0;
        for (int64_t c = 0; c < chunks; ++c) {
            const int64_t n = (N - c * h->max_tokens) < h->max_tokens ? (N - c * h->max_tokens)
                                                                      : h->max_tokens;
            const bool gemv = n <= 8 && gv_x_ok(h, n);
            const bool xin = sk_xin_ok(n, h->nb, h->kw);
            l += ((h->flags & QG_FLAG_FORCE_REFERENCE) || gemv || xin) ? 1 : 2;
        }
        *launches = (int32_t)l;
    }
    if (rows_cta && nfirst <= 8 && gv_x_ok(h, nfirst) && !(h->flags & QG_FLAG_FORCE_REFERENCE))
        *rows_cta = kGemvRows / h->kw;
    return QG_OK;
}


qg_status qgemv_chain_create(qg_chain **out, uint32_t flags)
{
    if (!out) return fail(QG_EINVAL, "null out");
    *out = nullptr;
    if (flags & ~(uint32_t)QG_CHAIN_PERSISTENT) return fail(QG_EINVAL, "unknown chain flag");
    qg_chain *c = new qg_chain();
    c->flags = flags;
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "device query");
    }
    e = cudaMalloc(&c->words, 4 * sizeof(unsigned int));
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return fail(QG_ENOMEM, "chain counters: %s", cudaGetErrorName(e));
    }
    e = cudaMemset(c->words, 0, 4 * sizeof(unsigned int));
    if (e != cudaSuccess) {
        cudaFree(c->words);
        delete c;
        return cuda_fail(e, "chain counters reset");
    }
    *out = c;
    return QG_OK;
}

qg_status qgemv_chain_run(qg_chain *c, const qg_call *calls, int32_t ncalls, void *stream)
{
    g_err.clear();
    if (!c || !calls) return fail(QG_EINVAL, "null chain or calls");
    if (ncalls < 1) return fail(QG_EINVAL, "ncalls must be >= 1");
    for (int i = 0; i < ncalls; ++i) {
        const qg_status st = check_call(calls[i]);
        if (st != QG_OK) return st;
    }
    const cudaStream_t s = (cudaStream_t)stream;
    int i = 0;
    while (i < ncalls) {
        int j = i;
        if (c->flags & QG_CHAIN_PERSISTENT)
            while (j < ncalls && j - i < kChainMaxCalls && chain_ok(c, calls[j])) ++j;
        if (j - i >= 2) {
            const qg_status st = launch_chain_calls(c, calls + i, j - i, s);
            if (st == QG_OK) {
                i = j;
                continue;
            }
            if (st != QG_EUNSUPPORTED) return st;
        }
        // one call through its entry point
        const qg_status st = run_call(calls[i], s);
        if (st != QG_OK) return st;
        ++i;
    }
    return QG_OK;
}

// The address a kernel uses for a host buffer: its mapped device address if
// the buffer is page-locked and mapped, else null (copy-engine path).
static const void *mapped_device_ptr(const void *host)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// One host <-> device transfer of a chain step: by the SMs through the mapped
// host buffer when it is page-locked, mapped and the copy is whole 16-byte
// units, else by the copy engine.
static qg_status step_copy(const void *src, void *dst, size_t bytes, bool to_device,
                           cudaStream_t s)
{
    if (bytes == 0) return QG_OK;
    const void *hp = to_device ? src : dst;
    const void *mapped = mapped_device_ptr(hp);
    if (mapped && bytes % 16 == 0 && aligned(src, 16) && aligned(dst, 16) && aligned(mapped, 16)) {
        const cudaError_t e = to_device ? launch_copy16(mapped, dst, bytes, s)
                                        : launch_copy16(src, const_cast<void *>(mapped), bytes, s);
        if (e == cudaSuccess) return QG_OK;
        cudaGetLastError();
    }
    const cudaError_t e = cudaMemcpyAsync(dst, src, bytes,
                                          to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "step copy");
}

qg_status qgemv_chain_run_host(qg_chain *c, const qg_call *calls, int32_t ncalls,
                               const void *in_host, void *in_dev, size_t in_bytes,
                               const void *out_dev, void *out_host, size_t out_bytes,
                               void *stream)
{
    g_err.clear();
    if (!c || !calls) return fail(QG_EINVAL, "null chain or calls");
    if (ncalls < 1) return fail(QG_EINVAL, "ncalls must be >= 1");
    if ((in_bytes && (!in_host || !in_dev)) || (out_bytes && (!out_dev || !out_host)))
        return fail(QG_EINVAL, "null step buffer");
    for (int i = 0; i < ncalls; ++i) {
        const qg_status st = check_call(calls[i]);
        if (st != QG_OK) return st;
    }
    const cudaStream_t s = (cudaStream_t)stream;
    qg_status st = step_copy(in_host, in_dev, in_bytes, true, s);
    if (st == QG_OK) st = qgemv_chain_run(c, calls, ncalls, stream);
    if (st == QG_OK) st = step_copy(out_dev, out_host, out_bytes, false, s);
    if (st != QG_OK) return st;
    const cudaError_t e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "stream synchronize");
}

qg_status qgemv_chain_status(qg_chain *c, uint32_t *flags_out, int clear)
{
    if (!c) return fail(QG_EINVAL, "null chain");
    unsigned int w = 0;
    cudaError_t e = cudaMemcpy(&w, c->words + 2, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "chain error word read");
    if (clear && w) {
        e = cudaMemset(c->words + 2, 0, sizeof(unsigned int));
        if (e != cudaSuccess) return cuda_fail(e, "chain error word reset");
    }
    if (flags_out) *flags_out = w;
    return QG_OK;
}

void qgemv_chain_destroy(qg_chain *c)
{
    if (!c) return;
    cudaFree(c->words);
    delete c;
}

}  // extern "C"
