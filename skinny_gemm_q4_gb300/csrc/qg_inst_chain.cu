// The persistent decode-chain kernel (qg_chain.cuh) for the K-quant formats.
#include "qg_chain.cuh"
#include "qg_launch.cuh"

namespace qg {

constexpr int kChainTset = TS_Q4K | TS_Q6K;
constexpr int kChainMaxSmem = 227 * 1024;  // the most one CTA may opt into

template <bool ONE>
static cudaError_t chain_configure()
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(qg_chain_kernel<kChainTset, ONE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kChainMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qg_chain_kernel<kChainTset, ONE>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    return cudaSuccess;
}

int chain_max_smem() { return kChainMaxSmem; }

int chain_ctas_per_sm(int smem, bool one)
{
    int n = 0;
    cudaError_t e = one ? chain_configure<true>() : chain_configure<false>();
    if (e == cudaSuccess)
        e = one ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &n, qg_chain_kernel<kChainTset, true>, kChainThreads, smem)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                      &n, qg_chain_kernel<kChainTset, false>, kChainThreads, smem);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_chain(const ChainParams &p, int grid, int smem, bool one, cudaStream_t s)
{
    if (smem > kChainMaxSmem) return cudaErrorInvalidValue;
    cudaError_t e = one ? chain_configure<true>() : chain_configure<false>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kChainThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (one) return cudaLaunchKernelEx(&cfg, qg_chain_kernel<kChainTset, true>, p);
    return cudaLaunchKernelEx(&cfg, qg_chain_kernel<kChainTset, false>, p);
}

}  // namespace qg
