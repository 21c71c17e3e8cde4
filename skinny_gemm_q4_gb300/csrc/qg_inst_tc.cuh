// Launchers of qg_tc_kernel (K-quant prefill chunks on the 5th-generation
// tensor core).  Each qg_inst_tc_*.cu defines QG_TC_TYPE and QG_TC_NAME and
// includes this file: one translation unit per weight format, so that they
// compile in parallel.  With QG_TC_MIXED the launcher runs
// qg_tc_mixed_kernel (Q4_K and Q6_K tiles in one launch).
#pragma once
#include "qg_launch.cuh"
#include "qg_tc.cuh"

namespace qg {

template <int T, int G>
static cudaError_t launch_tc_one(const Params &p, dim3 grid, int smem, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (smem > kTcMaxSmem) return cudaErrorInvalidValue;
#ifdef QG_TC_MIXED
    (void)T;
    auto fn = qg_tc_mixed_kernel<G>;
#else
    auto fn = qg_tc_kernel<T, G>;
#endif
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.ks > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.ks;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

#ifdef QG_TC_CAPACITY
// How many clusters of ks CTAs of qg_tc_kernel (one CTA per SM) the GPU runs
// at once: a cluster must fit in one GPC, so for ks > 2 this is less than
// 152 / ks.  Queried once per device and cluster size; 0 on failure.
int tc_cluster_capacity(int ks)
{
    static int cache[64][9];
    static bool filled[64][9];
    int dev = 0;
    if (ks < 1 || ks > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (filled[dev][ks]) return cache[dev][ks];
    auto fn = qg_tc_kernel<QG_TC_TYPE, 16>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (ks > 1 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                      cudaSuccess)
        cudaGetLastError();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ks, 152, 1);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcMinSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[dev][ks] = n;
    filled[dev][ks] = true;
    return n;
}
#endif

cudaError_t QG_TC_NAME(int G, const Params &p, dim3 grid, int smem, cudaStream_t s)
{
    constexpr int T = QG_TC_TYPE;
    switch (G) {
    case 2: return launch_tc_one<T, 2>(p, grid, smem, s);
    case 4: return launch_tc_one<T, 4>(p, grid, smem, s);
    case 6: return launch_tc_one<T, 6>(p, grid, smem, s);
    case 8: return launch_tc_one<T, 8>(p, grid, smem, s);
    case 10: return launch_tc_one<T, 10>(p, grid, smem, s);
    case 12: return launch_tc_one<T, 12>(p, grid, smem, s);
    case 14: return launch_tc_one<T, 14>(p, grid, smem, s);
    case 16: return launch_tc_one<T, 16>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
