// cluster.cuh -- inline-PTX wrappers for thread-block clusters (sm_103a):
// the CTA's place in its cluster, addresses in a peer CTA's shared memory,
// asynchronous stores and barrier arrivals across the cluster, the bounded
// cluster-scope barrier wait, and the cluster-wide barrier.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace dep {

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// The address of this CTA's shared-memory location `a` in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// Asynchronous store into another CTA of the cluster; its 16 bytes count
// towards the transaction total of that CTA's barrier `bar` (a peer address).
__device__ __forceinline__ void st_async_peer_v4(uint32_t a, float x, float y, float z, float w, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(a),
                 "f"(x), "f"(y), "f"(z), "f"(w), "r"(bar)
                 : "memory");
}
// Arrive on a barrier of another CTA of the cluster, releasing this thread's
// earlier writes to the cluster's shared memory.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t a)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(a) : "memory");
}
// Bounded wait that also acquires what other CTAs of the cluster released.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    auto test = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        return ok != 0;
    };
    if (test())
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (test())
            return true;
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

}  // namespace dep
