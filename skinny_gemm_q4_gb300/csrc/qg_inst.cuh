// Instantiation helper: defines launch_gemv_<NAME> and launch_sk_<NAME>(G, ...)
// for one type set.
#pragma once
#include "qg_launch.cuh"

namespace qg {

template <int TSET>
static cudaError_t launch_gemv_one(const Params &p, dim3 grid, int smem, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (smem > kGemvMaxSmem) return cudaErrorInvalidValue;
    if (!configured[dev]) {
        // Largest shared-memory carveout, so two ~110 KB CTAs share an SM.
        e = cudaFuncSetAttribute(qg_n8_kernel<TSET, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qg_n8_kernel<TSET, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qg_n8_kernel<TSET, false>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qg_n8_kernel<TSET, true>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32 * (kGemvCW + 1));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.swiglu) {
        // the gate and up CTAs of one row tile form a cluster (SwiGLU epilogue)
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 2;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (p.N == 1) return cudaLaunchKernelEx(&cfg, qg_n8_kernel<TSET, true>, p);
    return cudaLaunchKernelEx(&cfg, qg_n8_kernel<TSET, false>, p);
}

template <int TSET, int G, bool XIN = false>
static cudaError_t launch_sk_one(const Params &p, dim3 grid, int smem, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (smem > kGemvMaxSmem) return cudaErrorInvalidValue;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(qg_sk_kernel<TSET, G, XIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemvMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qg_sk_kernel<TSET, G, XIN>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        // SwiGLU pairs of 8-slice matrices use clusters of 16 CTAs
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qg_sk_kernel<TSET, G, XIN>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.ks > 1 || p.swiglu) {
        // K-split ranks along x; for a SwiGLU pair the gate and up tiles along y
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.ks;
        attr[na].val.clusterDim.y = p.swiglu ? 2u : 1u;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, qg_sk_kernel<TSET, G, XIN>, p);
}

}  // namespace qg

#define QG_DEFINE_TSET(NAME, TSET)                                                          \
    namespace qg {                                                                          \
    cudaError_t launch_gemv_##NAME(const Params &p, dim3 grid, int smem, cudaStream_t s)  \
    {                                                                                       \
        return launch_gemv_one<TSET>(p, grid, smem, s);                                     \
    }                                                                                       \
    cudaError_t launch_sk_##NAME(int G, const Params &p, dim3 grid, int smem, cudaStream_t s) \
    {                                                                                       \
        switch (G) {                                                                        \
        case 1: return p.xin ? launch_sk_one<TSET, 1, true>(p, grid, smem, s)                \
                             : launch_sk_one<TSET, 1>(p, grid, smem, s);                     \
        case 2: return launch_sk_one<TSET, 2>(p, grid, smem, s);                            \
        case 3: return launch_sk_one<TSET, 3>(p, grid, smem, s);                            \
        case 4: return launch_sk_one<TSET, 4>(p, grid, smem, s);                            \
        default: return cudaErrorInvalidValue;                                              \
        }                                                                                   \
    }                                                                                       \
    }
