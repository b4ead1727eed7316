// ptx.cuh -- inline-PTX wrappers for sm_100-family features used by the sampler:
// thread-block clusters and distributed shared memory, mbarriers, and the bulk
// (TMA-engine) global->shared copy.
#pragma once

#include <cstdint>

namespace dst {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Full cluster barrier: release our shared-memory writes, acquire everybody's.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t dsmem_ld_u64(uint32_t a)
{
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t a)
{
    return __uint_as_float(dsmem_ld_u32(a));
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t a, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_u64(uint32_t a, uint64_t v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

// Generic helpers: read / write a trivially-copyable object of a remote CTA,
// 4 bytes at a time (the object must be 4-byte aligned and sized).
template <typename T>
__device__ __forceinline__ void dsmem_read(T& dst, const T& local_obj, uint32_t rank)
{
    static_assert(sizeof(T) % 4 == 0, "4-byte granularity");
    uint32_t a = dsmem_map(smem_addr(&local_obj), rank);
    uint32_t* d = reinterpret_cast<uint32_t*>(&dst);
#pragma unroll
    for (int i = 0; i < int(sizeof(T) / 4); ++i) d[i] = dsmem_ld_u32(a + 4 * i);
}

template <typename T>
__device__ __forceinline__ void dsmem_write(const T& src, T& local_obj, uint32_t rank)
{
    static_assert(sizeof(T) % 4 == 0, "4-byte granularity");
    uint32_t a = dsmem_map(smem_addr(&local_obj), rank);
    const uint32_t* s = reinterpret_cast<const uint32_t*>(&src);
#pragma unroll
    for (int i = 0; i < int(sizeof(T) / 4); ++i) dsmem_st_u32(a + 4 * i, s[i]);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `max_polls` unsuccessful polls; returns success.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t max_polls)
{
    for (uint32_t i = 0; i < max_polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---------------------------------------------------------------- bulk copy
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`
// (complete_tx). dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only), tracked per thread.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
                 : "memory");
}

}  // namespace dst
