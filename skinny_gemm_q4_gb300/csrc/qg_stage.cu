// Activation staging: x[N][K] fp16 -> the B-fragment order each format's
// product kernel reads, plus (for Q4_K/Q5_K) the per-sub-block sums of x.
//
// One warp handles one (token, 256-wide super-block); lane l holds the eight
// values x[256*sb + 8l .. +8], i.e. the aligned 4-groups 2l and 2l+1.
//
// The per-(token, super-block) layouts (576 bytes each) are written by
// stage_sb in qg_kernels.cuh, the same function the N <= 8 kernel uses for
// its in-kernel staging, so both paths see identical x and sub-block sums.
#include "qg_kernels.cuh"
#include "qg_tc.cuh"

namespace qg {

__global__ void __launch_bounds__(128)
    qg_stage_kernel(const __half *__restrict__ x, int N, int K, int nb, int64_t tok_stride,
                   uint8_t *xq4, uint8_t *xq6, uint8_t *xfp4)
{
    pdl_trigger();
    // The buffers written here are read by the previous product kernel.
    pdl_wait();
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= N * nb) return;
    const int n = warp / nb, sb = warp - n * nb;
    const uint4 v = *reinterpret_cast<const uint4 *>(x + (int64_t)n * K + 256 * sb + 8 * lane);
    const int64_t base = (int64_t)n * tok_stride + (int64_t)sb * kXTok;
    stage_sb(v, lane, xq4 ? xq4 + base : nullptr, xq6 ? xq6 + base : nullptr,
             xfp4 ? xfp4 + base : nullptr);
}

cudaError_t launch_stage(const __half *x, int N, int K, int nb, int64_t tok_stride, uint8_t *xq4,
                         uint8_t *xq6, uint8_t *xfp4, cudaStream_t stream)
{
    const int warps = N * nb;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qg_stage_kernel, x, N, K, nb, tok_stride, xq4, xq6, xfp4);
}

// The same for qg_tc_kernel's layout: token n of a 128-token chunk goes to
// row n % 8 of 8-token group (n % 128) / 8 of its super-block block (two
// halves, see stage_tc4).
__global__ void __launch_bounds__(128)
    qg_stage_tc_kernel(const __half *__restrict__ x, int N, int K, int nb, int64_t chunk_stride,
                     uint8_t *out)
{
    pdl_trigger();
    pdl_wait();
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= N * nb) return;
    const int n = warp / nb, sb = warp - n * nb;
    const uint4 v = *reinterpret_cast<const uint4 *>(x + (int64_t)n * K + 256 * sb + 8 * lane);
    uint8_t *sbb = out + (int64_t)(n / kTcTok) * chunk_stride + (int64_t)sb * (kTcGroups * kTcXBlk);
    stage_tc4(v, lane, sbb, (n % kTcTok) / 8, n % 8);
}

cudaError_t launch_stage_tc4(const __half *x, int N, int K, int nb, int64_t chunk_stride,
                             uint8_t *out, cudaStream_t stream)
{
    const int warps = N * nb;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qg_stage_tc_kernel, x, N, K, nb, chunk_stride, out);
}

}  // namespace qg

namespace qg {

// Copy of n16 16-byte units by the SMs (host <-> device through mapped,
// page-locked host memory, for the small per-step buffers where a copy-engine
// transfer costs several microseconds of setup).  Ordered like the kernels
// around it: it waits for the previous kernel before touching either buffer.
__global__ void __launch_bounds__(256) qg_copy16_kernel(const uint4 *__restrict__ src,
                                                        uint4 *__restrict__ dst, int64_t n16)
{
    pdl_trigger();
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

cudaError_t launch_copy16(const void *src, void *dst, size_t bytes, cudaStream_t s)
{
    const int64_t n16 = (int64_t)(bytes / 16);
    if (n16 == 0) return cudaSuccess;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 304) blocks = 304;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qg_copy16_kernel, (const uint4 *)src, (uint4 *)dst, n16);
}

}  // namespace qg
