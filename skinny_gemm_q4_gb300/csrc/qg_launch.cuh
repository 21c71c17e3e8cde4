// Host-side launch entry points of the kernels (one translation unit per
// weight-format set, so the instantiations compile in parallel).
#pragma once
#include <cuda_runtime.h>
#include "qg_kernels.cuh"

namespace qg {

constexpr int kGemvMaxSmem = 200 * 1024;

cudaError_t launch_stage(const __half *x, int N, int K, int nb, int64_t tok_stride, uint8_t *xq4,
                         uint8_t *xq6, uint8_t *xfp4, cudaStream_t stream);
// Copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) by the
// SMs; either side may be mapped page-locked host memory (qg_stage.cu).
cudaError_t launch_copy16(const void *src, void *dst, size_t bytes, cudaStream_t s);
cudaError_t launch_stage_tc4(const __half *x, int N, int K, int nb, int64_t chunk_stride,
                             uint8_t *out, cudaStream_t stream);
cudaError_t launch_dequant(const Mat &m, int K, float *out, cudaStream_t stream);
// Dequantize through the product kernels' decoders (qg_dequant.cu).
cudaError_t launch_dequant_fast(const Mat &m, int K, float *out, cudaStream_t stream);
// qg_tc_kernel (Q4_K / Q5_K / Q6_K, N >= 33, on the tensor core; defined in
// qg_inst_tc*.cu); G = token groups of 8 per CTA (even, 2..16).
cudaError_t launch_tc_q4k(int G, const Params &p, dim3 grid, int smem, cudaStream_t s);
cudaError_t launch_tc_q5k(int G, const Params &p, dim3 grid, int smem, cudaStream_t s);
cudaError_t launch_tc_q6k(int G, const Params &p, dim3 grid, int smem, cudaStream_t s);
// Q4_K and Q6_K matrices of one call in one launch (qg_tc_mixed_kernel).
cudaError_t launch_tc_q4k_q6k(int G, const Params &p, dim3 grid, int smem, cudaStream_t s);
// Clusters of ks qg_tc_kernel CTAs the GPU holds at once (0: unknown).
int tc_cluster_capacity(int ks);
cudaError_t launch_ref_gemv(const Mat &m, int K, const __half *x, int N, int out_f32,
                            cudaStream_t stream);
// Reference SwiGLU pair: h = silu(x.gate^T) * (x.up^T) into gate.y.
cudaError_t launch_ref_swiglu(const Mat &gate, const Mat &up, int K, const __half *x, int N,
                              int out_f32, cudaStream_t stream);

// The persistent decode chain (qg_chain.cuh, defined in qg_inst_chain.cu):
// CTAs of `smem` bytes that one SM holds at once (0: unknown), and the launch.
struct ChainParams;
int chain_max_smem();
int chain_ctas_per_sm(int smem, bool one);
cudaError_t launch_chain(const ChainParams &p, int grid, int smem, bool one, cudaStream_t s);

// Per type-set launchers (defined in qg_inst_*.cu).
#define QG_DECLARE_TSET(NAME)                                                           \
    cudaError_t launch_gemv_##NAME(const Params &p, dim3 grid, int smem, cudaStream_t s); \
    cudaError_t launch_sk_##NAME(int G, const Params &p, dim3 grid, int smem, cudaStream_t s);
QG_DECLARE_TSET(q4k)
QG_DECLARE_TSET(q5k)
QG_DECLARE_TSET(q6k)
QG_DECLARE_TSET(fp4)
QG_DECLARE_TSET(fp8)
QG_DECLARE_TSET(q4k_q6k)
#undef QG_DECLARE_TSET

}  // namespace qg
