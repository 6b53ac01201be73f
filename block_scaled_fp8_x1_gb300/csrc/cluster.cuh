// cluster.cuh -- thread-block-cluster queries and distributed shared-memory loads shared by
// the decode-shaped GEMMs (decode.cu, nvfp4.cu), whose split-K slices are reduced across
// the CTAs of a cluster.
#pragma once

#include <stdint.h>

namespace fp8rl {

// CTAs in this cluster, this cluster's index in the grid, and the grid's cluster count.
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_idx() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// 16-byte load from another CTA's shared memory (a shared::cluster address).
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

}  // namespace fp8rl
