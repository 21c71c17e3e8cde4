// Reference GPU kernels: a per-element decoder, the dequantize entry and a
// plain warp-per-row product (fp32 FMAs, fixed lane-stride order, butterfly
// reduction).  Correct but slow; used when the fast path is forced off, as
// the retry after a non-sticky launch failure of the fast path (reflex-llm
// "docs/kernels.md": any cudaError falls through to the typed byte-load
// kernel), and for qgemv_dequantize.
#include "qg_kernels.cuh"

namespace qg {

struct RefMat {
    const uint8_t *w;
    const uint8_t *sc;
    int64_t row_bytes;
    int64_t sc_row_bytes;
    int M, K, type;
    float gscale;
};

__device__ __forceinline__ float f16_at(const uint8_t *p)
{
    return __half2float(__ushort_as_half((unsigned short)(p[0] | (p[1] << 8))));
}

__device__ __forceinline__ void scale_min_k4(const uint8_t *s12, int s, int &sc, int &mn)
{
    if (s < 4) {
        sc = s12[s] & 63;
        mn = s12[s + 4] & 63;
    } else {
        sc = (s12[s + 4] & 15) | ((s12[s - 4] >> 6) << 4);
        mn = (s12[s + 4] >> 4) | ((s12[s] >> 6) << 4);
    }
}

// Exact weight w[row][k] rounded once to fp32.
__device__ float ref_weight(const RefMat &m, int row, int k)
{
    const uint8_t *r = m.w + (int64_t)row * m.row_bytes;
    if (m.type == T_FP8) {
        const uint32_t e = e4m3x2_to_h2(r[k]);  // low byte -> low half
        const float fe = __half2float(__ushort_as_half((unsigned short)(e & 0xffffu)));
        const uint8_t *sp = m.sc + (int64_t)(row >> 7) * m.sc_row_bytes + 2 * (k >> 7);
        const uint32_t sb = (uint32_t)sp[0] | ((uint32_t)sp[1] << 8);
        return __fmul_rn(fe, __uint_as_float(sb << 16));
    }
    if (m.type == T_FP4) {
        const uint32_t byte = r[k >> 1];
        const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
        const uint32_t e = e2m1x2_to_h2(code);  // low nibble -> low half
        const uint32_t s = e4m3x2_to_h2(m.sc[(int64_t)row * m.sc_row_bytes + (k >> 4)]);
        const float fe = __half2float(__ushort_as_half((unsigned short)(e & 0xffffu)));
        const float fs = __half2float(__ushort_as_half((unsigned short)(s & 0xffffu)));
        return __fmul_rn(__fmul_rn(fe, fs), m.gscale);
    }
    const int b = k >> 8, j = k & 255;
    if (m.type == T_Q6K) {
        const uint8_t *blk = r + (int64_t)b * 210;
        const int h = j >> 7, s = (j >> 5) & 3, l = j & 31;
        const int low = blk[64 * h + 32 * (s & 1) + l];
        const int low4 = (s < 2) ? (low & 15) : (low >> 4);
        const int high2 = (blk[128 + 32 * h + l] >> (2 * s)) & 3;
        const int q = (low4 | (high2 << 4)) - 32;
        const int sc = (int8_t)blk[192 + 8 * h + l / 16 + 2 * s];
        return __fmul_rn(__fmul_rn(f16_at(blk + 208), (float)sc), (float)q);
    }
    const int bb = (m.type == T_Q4K) ? 144 : 176;
    const uint8_t *blk = r + (int64_t)b * bb;
    const int c = j >> 6, hi = (j >> 5) & 1, l = j & 31;
    const int qsoff = (m.type == T_Q4K) ? 16 : 48;
    const int byte = blk[qsoff + 32 * c + l];
    int q = hi ? (byte >> 4) : (byte & 15);
    if (m.type == T_Q5K) q += 16 * ((blk[16 + l] >> (2 * c + hi)) & 1);
    int sc, mn;
    scale_min_k4(blk + 4, 2 * c + hi, sc, mn);
    const float d = f16_at(blk), dmin = f16_at(blk + 2);
    return __fmaf_rn(__fmul_rn(d, (float)sc), (float)q, -__fmul_rn(dmin, (float)mn));
}

__global__ void qg_ref_dequant_kernel(RefMat m, float *out)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)m.M * m.K) return;
    const int row = (int)(i / m.K), k = (int)(i - (int64_t)row * m.K);
    out[i] = ref_weight(m, row, k);
}

__global__ void qg_ref_kernel(RefMat m, const __half *x, int N, const __half *res, void *y,
                                int out_f32)
{
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int tok = blockIdx.y;
    const int lane = threadIdx.x & 31;
    if (row >= m.M || tok >= N) return;
    float acc = 0.0f;
    for (int k = lane; k < m.K; k += 32)
        acc = __fmaf_rn(ref_weight(m, row, k), __half2float(x[(int64_t)tok * m.K + k]), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    if (lane == 0) {
        const int64_t o = (int64_t)tok * m.M + row;
        float v = acc;
        if (res) v = __fadd_rn(__half2float(res[o]), v);
        if (out_f32)
            reinterpret_cast<float *>(y)[o] = v;
        else
            reinterpret_cast<__half *>(y)[o] = __float2half_rn(v);
    }
}

// Reference SwiGLU pair: one warp per (row, token) computes both products
// as qg_ref_kernel does and stores h = silu(g) * u.
__global__ void qg_ref_swiglu_kernel(RefMat mg, RefMat mu, const __half *x, int N, void *y,
                                     int out_f32)
{
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int tok = blockIdx.y;
    const int lane = threadIdx.x & 31;
    if (row >= mg.M || tok >= N) return;
    float ag = 0.0f, au = 0.0f;
    for (int k = lane; k < mg.K; k += 32) {
        const float xv = __half2float(x[(int64_t)tok * mg.K + k]);
        ag = __fmaf_rn(ref_weight(mg, row, k), xv, ag);
        au = __fmaf_rn(ref_weight(mu, row, k), xv, au);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ag = __fadd_rn(ag, __shfl_xor_sync(0xffffffffu, ag, o));
        au = __fadd_rn(au, __shfl_xor_sync(0xffffffffu, au, o));
    }
    if (lane == 0) {
        const int64_t o = (int64_t)tok * mg.M + row;
        const float h = __fmul_rn(qg_silu(ag), au);
        if (out_f32)
            reinterpret_cast<float *>(y)[o] = h;
        else
            reinterpret_cast<__half *>(y)[o] = __float2half_rn(h);
    }
}

static RefMat make_ref(const Mat &mm, int K)
{
    RefMat r;
    r.w = mm.w;
    r.sc = mm.sc;
    r.row_bytes = mm.row_bytes;
    r.sc_row_bytes = mm.sc_row_bytes;
    r.M = mm.M;
    r.K = K;
    r.type = mm.type;
    r.gscale = mm.gscale;
    return r;
}

cudaError_t launch_dequant(const Mat &mm, int K, float *out, cudaStream_t stream)
{
    const RefMat r = make_ref(mm, K);
    const int64_t total = (int64_t)r.M * K;
    const unsigned blocks = (unsigned)((total + 255) / 256);
    qg_ref_dequant_kernel<<<blocks, 256, 0, stream>>>(r, out);
    return cudaGetLastError();
}

cudaError_t launch_ref_gemv(const Mat &mm, int K, const __half *x, int N, int out_f32,
                            cudaStream_t stream)
{
    const RefMat r = make_ref(mm, K);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((r.M + 3) / 4), (unsigned)N);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qg_ref_kernel, r, x, N, mm.res, mm.y, out_f32);
}

}  // namespace qg

namespace qg {
cudaError_t launch_ref_swiglu(const Mat &gate, const Mat &up, int K, const __half *x, int N,
                              int out_f32, cudaStream_t stream)
{
    const RefMat rg = make_ref(gate, K), ru = make_ref(up, K);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rg.M + 3) / 4), (unsigned)N);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qg_ref_swiglu_kernel, rg, ru, x, N, gate.y, out_f32);
}
}  // namespace qg
