// Inline-PTX helpers for the qgemv kernels (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace qg {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global->shared copy that bypasses L1.  src_bytes < 16
// reads only that many bytes and zero-fills the rest (src_bytes == 0 reads
// nothing).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr)
{
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
    return v;
}

// fp16x2 multiply, round to nearest, subnormals kept (no .ftz).
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Tensor-core MMA m16n8k16, fp16 inputs, fp32 accumulate (D = A.B + C).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with C = 0.
__device__ __forceinline__ void mma16816_zc(float (&d)[4], uint32_t a0, uint32_t a1,
                                            uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1)
{
    float z = 0.0f;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// Two packed e2m1 codes (low nibble first) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte_in_low8)
{
    uint32_t d;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n"
        : "=r"(d)
        : "r"(byte_in_low8));
    return d;
}

// Four code bytes of w (eight e2m1 values) -> four fp16x2, byte i in h[i],
// each byte's low nibble in the low half, exact.
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t &h0, uint32_t &h1, uint32_t &h2,
                                               uint32_t &h3)
{
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

// Two packed e4m3 codes (low byte first) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t pair_in_low16)
{
    uint32_t d;
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n"
        " cvt.rn.f16x2.e4m3x2 %0, lo;\n}\n"
        : "=r"(d)
        : "r"(pair_in_low16));
    return d;
}

// Four packed e4m3 codes -> (e0, e1) and (e2, e3) as fp16x2, exact: both
// conversions read their 16-bit halves of w directly.
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t w, uint32_t &lo2, uint32_t &hi2)
{
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
        " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}\n"
        : "=r"(lo2), "=r"(hi2)
        : "r"(w));
}

// Programmatic dependent launch controls (no-ops without a PDL predecessor).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Thread-block cluster helpers.
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::
                     : "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
// Split cluster barrier without memory ordering: arrive (relaxed) once this
// thread's reads of other CTAs' shared memory have returned, wait before
// the CTA may exit.  Unlike cluster_sync() it does not wait for this
// thread's earlier global stores to complete.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, float a, float b, float c, float d)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

}  // namespace qg

namespace qg {

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy (TMA, 1-D) helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(addr), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t addr)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(addr) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(addr),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `limit` polls and returns false (the caller
// records the timeout and carries on, so a logic error never hangs the GPU).
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity,
                                          uint32_t limit = (1u << 22))
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(addr, parity)) return true;
    return false;
}

// Non-blocking probe of a phase (no suspend): cheaper than try_wait for a
// single thread that must get back to issuing work as soon as the phase is
// complete.
__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded spin on mbar_test (the same contract as mbar_wait).
__device__ __forceinline__ bool mbar_wait_spin(uint32_t addr, uint32_t parity,
                                               uint32_t limit = (1u << 26))
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_test(addr, parity)) return true;
    return false;
}

// Bulk global->shared copy completing on an mbarrier (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];\n" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void bar_sync_named(int id, int threads)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace qg

namespace qg {

// 2-D tiled tensor copy global->shared, completing on an mbarrier.  tmap is
// the generic address of a CUtensorMap held in kernel-parameter space.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y,
                                            uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(tmap) : "memory");
}

// Arrive on an mbarrier once all prior cp.async of this thread have landed
// (the arrival is counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t mbar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(mbar) : "memory");
}

}  // namespace qg

namespace qg {

// 3-D tiled tensor copy global->shared, completing on an mbarrier.
// L2 policy for data read once (streamed weights): evicted first, so that
// activations and other reused data stay in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_3d_ef(uint32_t dst, const void *tmap, int x, int y, int z,
                                               uint32_t mbar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;\n" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(mbar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_ef(uint32_t dst, const void *src, uint32_t bytes,
                                            uint32_t mbar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;\n" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(mbar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            uint32_t mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

}  // namespace qg

namespace qg {

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, tensor memory) helpers.
// TMEM addresses: bits 31..16 lane, 15..0 column (32-bit cells).
// ---------------------------------------------------------------------------
// Allocate `ncols` columns (power of two >= 32) for this CTA; the base address
// is written to shared memory at dst.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the tensor core.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Store 8 / 32 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31, %32};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
// Load 8 consecutive columns of this thread's lane (call tc_wait_ld before use).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}

// Load 32 consecutive columns of this thread's lane (call tc_wait_ld before use).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor, no swizzle, K-major: core matrices of 8
// rows x 16 bytes; the two byte strides (between core matrices adjacent in K
// and in the other dimension) are both `stride`.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t stride)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((stride >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((stride >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// The same with separate strides: lbo between core matrices adjacent in K,
// sbo between 8-row groups of the other dimension.
__device__ __forceinline__ uint64_t smem_desc2(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: fp32 D, fp16 A and B, both K-major,
// M = 128, N = n.
__host__ __device__ constexpr uint32_t tc_idesc_f16(uint32_t n)
{
    return (1u << 4) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}
// D[tmem] (+)= A[tmem] . B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_t, uint32_t a_t, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_t),
        "r"(a_t), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[smem] . B[smem]^T (both operands by shared-memory descriptor).
__device__ __forceinline__ void tc_mma_ss(uint32_t d_t, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_t),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Eight MMAs of consecutive k-steps, D[d] (+)= A[a0 + 8 s] . B[b0 + s * 256 B]
// (s = 0..7; the first accumulates iff acc0), issued back to back while two
// mbarrier phases are probed (test_wait, no suspend): returns 1 iff both
// (bar1, par1) and (bar2, par2) were complete.  The probes' latency hides
// behind the MMAs, whose issue is close to synchronous with the tensor core.
__device__ __forceinline__ uint32_t tc_mma8_probe(uint32_t d, uint32_t a0, uint64_t b0,
                                                  uint32_t idesc, uint32_t acc0, uint32_t bar1,
                                                  uint32_t par1, uint32_t bar2, uint32_t par2)
{
    uint32_t ok;
    asm volatile(
        "{\n"
        " .reg .pred q1, q2, pa, pt;\n"
        " .reg .b64 bd;\n"
        " .reg .b32 aa;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 q1, [%6], %7;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 q2, [%8], %9;\n"
        " setp.ne.u32 pa, %5, 0;\n"
        " setp.eq.u32 pt, %5, %5;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %4, pa;\n"
        " add.u32 aa, %2, 8;\n add.u64 bd, %3, 16;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 16;\n add.u64 bd, %3, 32;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 24;\n add.u64 bd, %3, 48;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 32;\n add.u64 bd, %3, 64;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 40;\n add.u64 bd, %3, 80;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 48;\n add.u64 bd, %3, 96;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 56;\n add.u64 bd, %3, 112;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " and.pred q1, q1, q2;\n"
        " selp.u32 %0, 1, 0, q1;\n"
        "}\n"
        : "=r"(ok)
        : "r"(d), "r"(a0), "l"(b0), "r"(idesc), "r"(acc0), "r"(bar1), "r"(par1), "r"(bar2),
          "r"(par2)
        : "memory");
    return ok;
}
// The same with four MMAs (s = 0..3).
__device__ __forceinline__ uint32_t tc_mma4_probe(uint32_t d, uint32_t a0, uint64_t b0,
                                                  uint32_t idesc, uint32_t acc0, uint32_t bar1,
                                                  uint32_t par1, uint32_t bar2, uint32_t par2)
{
    uint32_t ok;
    asm volatile(
        "{\n"
        " .reg .pred q1, q2, pa, pt;\n"
        " .reg .b64 bd;\n"
        " .reg .b32 aa;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 q1, [%6], %7;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 q2, [%8], %9;\n"
        " setp.ne.u32 pa, %5, 0;\n"
        " setp.eq.u32 pt, %5, %5;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %4, pa;\n"
        " add.u32 aa, %2, 8;\n add.u64 bd, %3, 16;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 16;\n add.u64 bd, %3, 32;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " add.u32 aa, %2, 24;\n add.u64 bd, %3, 48;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [aa], bd, %4, pt;\n"
        " and.pred q1, q1, q2;\n"
        " selp.u32 %0, 1, 0, q1;\n"
        "}\n"
        : "=r"(ok)
        : "r"(d), "r"(a0), "l"(b0), "r"(idesc), "r"(acc0), "r"(bar1), "r"(par1), "r"(bar2),
          "r"(par2)
        : "memory");
    return ok;
}
// Arrive on a CTA mbarrier once all tcgen05.mma issued so far by this thread complete.
__device__ __forceinline__ void tc_commit(uint32_t mbar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
        : "memory");
}

}  // namespace qg
