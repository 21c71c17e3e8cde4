// qgemv_run_noalloc: the product of qgemv_run without a handle and without
// any device allocation.  The staged x (B-fragment order and sub-block sums)
// that qgemv_run keeps in a buffer owned by the handle, and the kernels'
// error word, live in one fixed file-scope device array instead, so this
// entry point never calls cudaMalloc / cudaFree or any allocating routine;
// the launch plan and the tensor maps of a handle are built on the host, in
// a handle on the stack, for every call (qg::run_with_scratch, qg_api.cu).
//
// Who needs it: programs that may not allocate device memory once they are
// running -- for example a serving runtime that reserves all device memory in
// its own pool at start-up (any cudaMalloc behind its back can fail or
// fragment that pool), or a library that must not change its host process's
// device-memory footprint -- but still hold the weights, x and y in memory of
// their own.
//
// Limits and sharing rules:
//   * The array holds kNoallocScratchBytes (2 MiB): the last 256 bytes are the
//     error word, the rest staged x.  A call stages min(32, that / (K/256 * 576
//     bytes)) tokens at a time and loops over N; if not even one token fits (K
//     above 931,840) the call is rejected with QG_EUNSUPPORTED before any CUDA
//     call.  Calls with N <= 8 stage x inside the product kernel and use only
//     the error word.
//   * Every call on a device uses the same array, and the array keeps the last
//     call's contents.  The staged x needs no clearing: each call writes every
//     staged byte it later reads.  The error word starts at zero (static
//     device memory is zeroed when the library is loaded); kernels only OR
//     bits into it, and qgemv_device_status(NULL, ..) reads (and may clear)
//     it.  Two calls whose kernels overlap on the GPU (different streams, no
//     ordering) race on the array and give wrong results; order them on one
//     stream.
//   * The first call on each device (and the first qgemv_device_status(NULL,
//     ..) there) looks up the array's device address with
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
constexpr size_t kNoallocErrOffset = kNoallocScratchBytes - 256;

// The scratch array.  In host code this name is only a host-side stand-in for
// the symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
uint8_t *g_scratch_ptr[kMaxDevices] = {nullptr};

}  // namespace

namespace qg {
void set_last_error(const char *msg);  // qg_api.cu: the text qgemv_last_error returns
qg_status run_with_scratch(qg_type t, int64_t M, int64_t K, const void *w_dev,
                           const void *scales_dev, float global_scale, const void *x, int64_t N,
                           void *y, qg_out ydt, cudaStream_t s, uint8_t *(*get_scratch)(),
                           size_t scratch_bytes, size_t err_offset);

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).  Null on failure (message set).
uint8_t *noalloc_scratch()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        set_last_error("qgemv_run_noalloc: no usable current device");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            set_last_error("qgemv_run_noalloc: cudaGetSymbolAddress of the scratch array failed");
            return nullptr;
        }
        g_scratch_ptr[dev] = (uint8_t *)p;
    }
    return g_scratch_ptr[dev];
}

// The allocation-free path's error word on the current device (null on failure).
unsigned int *noalloc_error_word()
{
    uint8_t *s = noalloc_scratch();
    return s ? reinterpret_cast<unsigned int *>(s + kNoallocErrOffset) : nullptr;
}
}  // namespace qg

extern "C" qg_status qgemv_run_noalloc(qg_type t, int64_t M, int64_t K, const void *w_dev,
                                       const void *scales_dev, float global_scale, const void *x,
                                       int64_t N, void *y, qg_out ydt, void *stream)
{
    // Every argument is checked before the device is touched; the scratch
    // array's address is looked up only then.
    return qg::run_with_scratch(t, M, K, w_dev, scales_dev, global_scale, x, N, y, ydt,
                                (cudaStream_t)stream, qg::noalloc_scratch, kNoallocErrOffset,
                                kNoallocErrOffset);
}
