// Building blocks of the producer/consumer kernels (staged two-pass rows,
// staged columns): a ring cursor without divisions, distributed shared memory
// stores, remote mbarrier arrivals and a cluster-scope bounded wait, and
// barriers over part of a CTA or a whole cluster (inline PTX, sm_90+ forms).
#pragma once

#include "common.cuh"

namespace rwsm {

// Position in a ring of stages walked in order: the stage and the parity of
// the number of completed trips around the ring (the mbarrier phase parity
// of that stage's next use), advanced without divisions.
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int stages)
    {
        if (++slot == stages) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// ------------------------------------ distributed shared memory, barriers
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float a, float b)
{
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" :: "r"(addr), "f"(a), "f"(b)
                 : "memory");
}

// Arrive on an mbarrier of any CTA of the cluster, releasing this thread's
// earlier writes (distributed shared memory included) at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

// Bounded wait (as mbar_wait_bounded) with acquire at cluster scope: writes
// released by peers' mbar_arrive_cluster are visible after it returns true.
// Polls without a suspend-time hint.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
        if (ok)
            return true;
        if ((it & 255u) == 255u && global_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return false;
}

// Barrier over the first `count` threads of the CTA (a multiple of 32) on
// hardware barrier `id` (1..15; __syncthreads uses 0).
__device__ __forceinline__ void named_barrier(int id, int count)
{
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// Cluster-wide barrier for every thread of every CTA (release / acquire);
// the non-.aligned form, so it may follow divergent code.
__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

}  // namespace rwsm
