// Launchers of qg_tc_kernel (Q4_K prefill chunks on the 5th-generation tensor core).
#include "qg_launch.cuh"
#include "qg_tc.cuh"

namespace qg {

template <int G>
static cudaError_t launch_tc_one(const Params &p, dim3 grid, int smem, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (smem > kGemvMaxSmem) return cudaErrorInvalidValue;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(qg_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemvMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qg_tc_kernel<G>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
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
    return cudaLaunchKernelEx(&cfg, qg_tc_kernel<G>, p);
}

cudaError_t launch_tc(int G, const Params &p, dim3 grid, int smem, cudaStream_t s)
{
    switch (G) {
    case 1: return launch_tc_one<1>(p, grid, smem, s);
    case 2: return launch_tc_one<2>(p, grid, smem, s);
    case 3: return launch_tc_one<3>(p, grid, smem, s);
    case 4: return launch_tc_one<4>(p, grid, smem, s);
    case 5: return launch_tc_one<5>(p, grid, smem, s);
    case 6: return launch_tc_one<6>(p, grid, smem, s);
    case 7: return launch_tc_one<7>(p, grid, smem, s);
    case 8: return launch_tc_one<8>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
