// cluster.cuh -- thread-block-cluster helpers: rank, barriers and
// distributed-shared-memory (DSMEM) access to the other CTAs of a cluster.
#pragma once

#include "common.cuh"

namespace dflv {

DFLV_DEVINL uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// Full cluster barrier: every thread of every CTA arrives (release) and waits
// (acquire), so shared-memory writes into any CTA before it are visible to
// every thread after it.
DFLV_DEVINL void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                     : "memory");
}
// Split form: arrive early (no ordering), wait later.  Arriving at kernel
// start and waiting before the first DSMEM access guarantees that every CTA
// of the cluster has started.
DFLV_DEVINL void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory"); }
DFLV_DEVINL void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory"); }

DFLV_DEVINL uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
// Loads from a peer CTA's shared memory.  They keep a memory clobber so they
// stay after the cluster barrier that publishes the data; callers issue all
// of their loads before using any result.
DFLV_DEVINL float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
DFLV_DEVINL int ld_dsmem_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
DFLV_DEVINL float2 ld_dsmem_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0,%1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
DFLV_DEVINL float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}
// Store into a peer CTA's shared memory (made visible by a later
// cluster_sync_all).
DFLV_DEVINL void st_dsmem_f2(uint32_t addr, float x, float y) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1,%2};\n" ::"r"(addr), "f"(x), "f"(y) : "memory");
}
DFLV_DEVINL void st_dsmem_u4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
DFLV_DEVINL void st_dsmem_f4(uint32_t addr, float x, float y, float z, float w) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "f"(x), "f"(y), "f"(z), "f"(w)
                 : "memory");
}

}  // namespace dflv
