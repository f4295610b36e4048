// Inline-PTX helpers for sm_103a: mbarriers with bounded waits, bulk (TMA) copies,
// cluster barriers and distributed shared memory, tcgen05 tensor-core plumbing.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "status.h"

namespace lora {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Record a device-side failure (first writer wins) in the context's status word.
__device__ __forceinline__ void raise_status(unsigned *status, unsigned code)
{
    if (status)
        atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster (its cluster address, from
// map_cluster), releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
                 : "memory");
}

// try_wait with acquire at cluster scope: pairs with arrivals made from other CTAs
// of the cluster (mbar_arrive_remote).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier for at most `limit_ns` nanoseconds.  On
// expiry the status word records `code` and false is returned; the caller keeps
// the barrier structure of its CTA/cluster intact and skips its stores.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned *status, unsigned code,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            raise_status(status, code);
            return false;
        }
    }
}

// mbar_wait_bounded with cluster-scope acquire.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          unsigned *status, unsigned code,
                                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            raise_status(status, code);
            return false;
        }
    }
}

// ---------------------------------------------------------------- bulk copies

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0),
// completion signalled as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync()
{
    cluster_arrive_release();
    cluster_wait_acquire();
}

__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_cluster(uint32_t local_smem, uint32_t rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_smem), "r"(rank));
    return ra;
}

// Asynchronous 16-byte store into a peer CTA's shared memory (cluster addresses of
// the destination and of the peer's mbarrier): the bytes complete a transaction on
// that mbarrier, which the peer waits on locally.
__device__ __forceinline__ void st_async_v4(uint32_t remote_dst, float4 v, uint32_t remote_bar)
{
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
        ::"r"(remote_dst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
        : "memory");
}

// Read a float from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_dsmem_f32(const float *local, uint32_t rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// ---------------------------------------------------------------- programmatic launch

// Wait until the preceding kernel in the stream has completed and its writes are
// visible (returns at once when the launch has no programmatic predecessor).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream to start launching its CTAs.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- bf16 vectors

__device__ __forceinline__ void unpack8(const uint4 &u, float f[8])
{
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float2 t = __bfloat1622float2(h[e]);
        f[2 * e] = t.x;
        f[2 * e + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float f[8])
{
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e)
        h[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
    return u;
}

// acc0 += sum over even e of a[e] b[e], acc1 += the odd ones, for 8 bf16 pairs:
// mixed-precision FMA (bf16 multiplicands, fp32 accumulator, one rounding: the
// same result as fmaf on the converted values), no conversion instructions.
__device__ __forceinline__ void dot8_bf16(const uint4 &a, const uint4 &b, float &acc0, float &acc1)
{
    asm("{\n\t.reg .b16 a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
        "mov.b32 {a0, a1}, %2;\n\tmov.b32 {a2, a3}, %3;\n\t"
        "mov.b32 {a4, a5}, %4;\n\tmov.b32 {a6, a7}, %5;\n\t"
        "mov.b32 {b0, b1}, %6;\n\tmov.b32 {b2, b3}, %7;\n\t"
        "mov.b32 {b4, b5}, %8;\n\tmov.b32 {b6, b7}, %9;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t"
        "fma.rn.f32.bf16 %0, a2, b2, %0;\n\tfma.rn.f32.bf16 %1, a3, b3, %1;\n\t"
        "fma.rn.f32.bf16 %0, a4, b4, %0;\n\tfma.rn.f32.bf16 %1, a5, b5, %1;\n\t"
        "fma.rn.f32.bf16 %0, a6, b6, %0;\n\tfma.rn.f32.bf16 %1, a7, b7, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace lora
