// qgemv_run_noalloc: the staging + product path of qgemv_run without any
// device allocation.  The staged x (B-fragment order and sub-block sums) that
// qgemv_run keeps in a buffer owned by the handle lives here in one fixed
// file-scope device array instead, so a caller needs no handle and this entry
// point never calls cudaMalloc / cudaFree or any allocating routine.
//
// Who needs it: programs that may not allocate device memory once they are
// running — for example a serving runtime that reserves all device memory in
// its own pool at start-up, or a library that must not change its host
// process's device-memory footprint — but still hold the weights, x and y in
// memory of their own.
//
// Limits and sharing rules:
//   * The array holds kNoallocScratchBytes (2 MiB).  A call stages
//     min(32, 2 MiB / (K/256 * 576 bytes)) tokens at a time and loops over N;
//     if not even one token fits (K above 931,840) the call is rejected with
//     QG_EUNSUPPORTED.
//   * Every call on a device uses the same array, and the array keeps the last
//     call's contents.  Nothing in it has to start at zero: each call writes
//     every staged byte it later reads.  Two calls whose kernels overlap on the
//     GPU (different streams, no ordering) race on the array and give wrong
//     results; order them on one stream.
//   * The first call on each device looks up the array's device address with
//     cudaGetSymbolAddress while that device is current; make that first call
//     before any stream capture on the device.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "qg_launch.cuh"
#include "qgemv.h"

namespace {

constexpr size_t kNoallocScratchBytes = 2u << 20;

// The scratch array.  In host code this name is only a host-side stand-in for
// the symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
uint8_t *g_scratch_ptr[kMaxDevices] = {nullptr};

}  // namespace

namespace qg {
void set_last_error(const char *msg);    // qg_api.cu: the text qgemv_last_error returns
int plan_k_slices(int64_t M, int nb);   // qg_api.cu: a handle's K slices for (M, K/256)
}

namespace {

qg_status noalloc_fail(qg_status s, const char *msg)
{
    char buf[320];
    snprintf(buf, sizeof buf, "qgemv_run_noalloc: %s", msg);
    qg::set_last_error(buf);
    return s;
}

cudaError_t launch_product(int tset, int G, const qg::Params &p, dim3 grid, cudaStream_t s)
{
    using namespace qg;
    switch (tset) {
    case TS_Q4K: return launch_skinny_q4k(G, p, grid, s);
    case TS_Q5K: return launch_skinny_q5k(G, p, grid, s);
    case TS_Q6K: return launch_skinny_q6k(G, p, grid, s);
    case TS_FP4: return launch_skinny_fp4(G, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

extern "C" qg_status qgemv_run_noalloc(qg_type t, int64_t M, int64_t K, const void *w_dev,
                                       const void *scales_dev, float global_scale, const void *x,
                                       int64_t N, void *y, qg_out ydt, void *stream)
{
    using namespace qg;
    set_last_error("");
    const int bb = (t == QG_Q4_K) ? 144 : (t == QG_Q5_K) ? 176 : (t == QG_Q6_K) ? 210 : 0;
    if (bb == 0 && t != QG_NVFP4_W4A16) return noalloc_fail(QG_EUNSUPPORTED, "unknown weight type");
    if (M < 1 || N < 1) return noalloc_fail(QG_EINVAL, "M and N must be >= 1");
    if (K < 256 || K % 256 != 0) return noalloc_fail(QG_EUNSUPPORTED, "K must be a positive multiple of 256");
    if (M > (int64_t)1 << 30 || K > (int64_t)1 << 24) return noalloc_fail(QG_EUNSUPPORTED, "shape too large");
    if (!w_dev || !x || !y) return noalloc_fail(QG_EINVAL, "null pointer");
    if (t == QG_NVFP4_W4A16 && !scales_dev) return noalloc_fail(QG_EINVAL, "NVFP4 needs the scale array");
    if (ydt != QG_OUT_F16 && ydt != QG_OUT_F32) return noalloc_fail(QG_EINVAL, "bad output type");
    if (((uintptr_t)w_dev | (uintptr_t)x) % 16 || (scales_dev && (uintptr_t)scales_dev % 16) ||
        (uintptr_t)y % (ydt == QG_OUT_F32 ? 4 : 2))
        return noalloc_fail(QG_EALIGN, "misaligned pointer (weights, scales, x: 16 bytes)");

    const int nb = (int)(K / 256);
    const size_t tok_bytes = (size_t)nb * kXTok;
    const int64_t fit = (int64_t)(kNoallocScratchBytes / tok_bytes);
    if (fit < 1)
        return noalloc_fail(QG_EUNSUPPORTED,
                            "K too large: one token's staged x exceeds the 2 MiB scratch array");
    const int chunk = (int)(fit < kTokChunk ? fit : kTokChunk);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return noalloc_fail(QG_ECUDA, "no usable current device");
    }
    uint8_t *scratch;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_scratch_ptr[dev]) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                cudaGetLastError();
                return noalloc_fail(QG_ECUDA, "cudaGetSymbolAddress of the scratch array failed");
            }
            g_scratch_ptr[dev] = (uint8_t *)p;
        }
        scratch = g_scratch_ptr[dev];
    }

    // Same plan as a handle for (t, M, K): K slices of 1, 2, 4 or 8, so the
    // results equal qgemv_run's bit for bit.
    const int kw = plan_k_slices(M, nb);

    cudaStream_t s = (cudaStream_t)stream;
    const int esize = (ydt == QG_OUT_F32) ? 4 : 2;
    const int layout = (t == QG_Q6_K) ? XL_Q6 : (t == QG_NVFP4_W4A16 ? XL_FP4 : XL_Q4);
    const int tset = (t == QG_Q4_K) ? TS_Q4K
                   : (t == QG_Q5_K) ? TS_Q5K
                   : (t == QG_Q6_K) ? TS_Q6K
                                    : TS_FP4;
    const int64_t row_bytes = (t == QG_NVFP4_W4A16) ? K / 2 : (int64_t)nb * bb;
    for (int64_t c0 = 0; c0 < N; c0 += chunk) {
        const int n = (int)((N - c0) < chunk ? (N - c0) : chunk);
        const __half *xc = (const __half *)x + c0 * K;
        uint8_t *xl[XL_COUNT] = {nullptr, nullptr, nullptr, nullptr};
        xl[layout] = scratch;
        cudaError_t e = launch_stage(xc, n, (int)K, nb, (int64_t)tok_bytes, xl[XL_Q4], xl[XL_Q6],
                                     xl[XL_FP4], s);
        if (e != cudaSuccess) return noalloc_fail(QG_ECUDA, cudaGetErrorString(e));
        Params p;
        memset(&p, 0, sizeof p);
        Mat &m = p.mat[0];
        m.w = (const uint8_t *)w_dev;
        m.sc = (const uint8_t *)scales_dev;
        m.y = (uint8_t *)y + c0 * M * esize;
        m.res = nullptr;
        m.row_bytes = row_bytes;
        m.sc_row_bytes = (t == QG_NVFP4_W4A16) ? K / 16 : 0;
        m.w_bytes = row_bytes * M;
        m.M = (int)M;
        m.type = (int)t;
        m.tile_begin = 0;
        m.kw = kw;
        m.gscale = (t == QG_NVFP4_W4A16) ? global_scale : 1.0f;
        p.nmat = 1;
        for (int l = 0; l < XL_COUNT; ++l) p.xs[l] = xl[l];
        p.xs_tok_stride = (int64_t)tok_bytes;
        p.N = n;
        p.tok_base = 0;
        p.K = (int)K;
        p.nb = nb;
        p.ks = kw;
        p.out_f32 = (ydt == QG_OUT_F32);
        p.err = nullptr;
        const int G = n >= 32 ? 4 : (n + 7) / 8;
        const int rows = (G <= 2) ? Cfg<1>::ROWS : Cfg<4>::ROWS;
        const dim3 grid((unsigned)kw, (unsigned)((M + rows - 1) / rows),
                        (unsigned)((n + kTokChunk - 1) / kTokChunk));
        e = launch_product(tset, G, p, grid, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return noalloc_fail(QG_ECUDA, cudaGetErrorString(e));
        }
    }
    return QG_OK;
}
