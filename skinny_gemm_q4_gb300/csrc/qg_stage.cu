// Activation staging: x[N][K] fp16 -> the B-fragment order each format's
// product kernel reads, plus (for Q4_K/Q5_K) the per-sub-block sums of x.
//
// One warp handles one (token, 256-wide super-block); lane l holds the eight
// values x[256*sb + 8l .. +8], i.e. the aligned 4-groups 2l and 2l+1.
//
// Layouts, per (token, super-block), 576 bytes:
//   Q4 (Q4_K, Q5_K): 4-group q = 16t + 8e + j (thread t, nibble half e, word
//       j) goes to 16-byte unit ((j/2)*2 + e)*4 + t, half (j & 1); each
//       4-group stored as (x0, x2, x1, x3).  Bytes 512..543: for t = 0..3 the
//       fp16 (hi[2t], hi[2t+1], lo[2t], lo[2t+1]) of the sub-block sums
//       S_s = sum of the 32 x of sub-block s (fp32, fixed order),
//       hi = fp16(S), lo = fp16(S - hi).
//   Q6 (Q6_K): 4-group q = 32h + 8s + 4i + t goes to 16-byte unit
//       (h*4 + s)*4 + t, half i; stored as (x0, x2, x1, x3).
//   FP4 (NVFP4): the raw 8 values of lane l go to unit
//       ((l/16)*4 + (l&3))*4 + ((l/4)&3), unpermuted.
#include "qg_kernels.cuh"

namespace qg {

__global__ void __launch_bounds__(128)
    stage_x_kernel(const __half *__restrict__ x, int N, int K, int nb, int64_t tok_stride,
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

    if (xq4) {
        uint4 o;
        o.x = __byte_perm(v.x, v.y, 0x5410);
        o.y = __byte_perm(v.x, v.y, 0x7632);
        o.z = __byte_perm(v.z, v.w, 0x5410);
        o.w = __byte_perm(v.z, v.w, 0x7632);
        const int u = ((lane & 3) * 2 + ((lane >> 2) & 1)) * 4 + (lane >> 3);
        *reinterpret_cast<uint4 *>(xq4 + base + 16 * u) = o;

        // Sub-block sums: sequential within the lane, then a fixed butterfly.
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s = __fadd_rn(s, __half2float(__ushort_as_half((unsigned short)(w4[i] & 0xffffu))));
            s = __fadd_rn(s, __half2float(__ushort_as_half((unsigned short)(w4[i] >> 16))));
        }
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2));
        const __half hi = __float2half_rn(s);
        const __half lo = __float2half_rn(__fsub_rn(s, __half2float(hi)));
        const uint32_t hib = __half_as_ushort(hi), lob = __half_as_ushort(lo);
        const uint32_t hin = __shfl_down_sync(0xffffffffu, hib, 4);
        const uint32_t lon = __shfl_down_sync(0xffffffffu, lob, 4);
        if ((lane & 7) == 0) {
            uint2 o2;
            o2.x = hib | (hin << 16);
            o2.y = lob | (lon << 16);
            *reinterpret_cast<uint2 *>(xq4 + base + 512 + 8 * (lane >> 3)) = o2;
        }
    }
    if (xq6) {
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            const int q = 2 * lane + hq;
            const int h = q >> 5, s = (q >> 3) & 3, i = (q >> 2) & 1, t = q & 3;
            const uint32_t a = hq ? v.z : v.x, b = hq ? v.w : v.y;
            uint2 o2;
            o2.x = __byte_perm(a, b, 0x5410);
            o2.y = __byte_perm(a, b, 0x7632);
            *reinterpret_cast<uint2 *>(xq6 + base + 16 * ((h * 4 + s) * 4 + t) + 8 * i) = o2;
        }
    }
    if (xfp4) {
        const int u = ((lane >> 4) * 4 + (lane & 3)) * 4 + ((lane >> 2) & 3);
        *reinterpret_cast<uint4 *>(xfp4 + base + 16 * u) = v;
    }
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
    return cudaLaunchKernelEx(&cfg, stage_x_kernel, x, N, K, nb, tok_stride, xq4, xq6, xfp4);
}

}  // namespace qg
