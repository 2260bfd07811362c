// Thread-block cluster helpers: the CTA's rank in its cluster, the cluster
// barrier split into arrive (release) and wait (acquire), loads from another
// CTA's shared memory (DSMEM), and a launcher that sets the cluster size.
// Every thread of every CTA of a cluster must execute each arrive and each
// wait, in the same order and with its warp converged (the .aligned forms).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mgs {

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared-memory address p of this CTA, mapped to the cluster's CTA `rank`.
__device__ __forceinline__ unsigned dsmem_addr(const void *p, unsigned rank) {
    const unsigned local = static_cast<unsigned>(__cvta_generic_to_shared(p));
    unsigned remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}
__device__ __forceinline__ float ld_dsmem(const float *p, unsigned rank) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(dsmem_addr(p, rank)) : "memory");
    return v;
}
// 16 bytes (p 16-byte aligned)
__device__ __forceinline__ float4 ld_dsmem4(const float *p, unsigned rank) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(dsmem_addr(p, rank))
                 : "memory");
    return v;
}

// Launches kern on `blocks` CTAs (a multiple of S) in clusters of S along x
// (past the portable size of 8, up to 16, with the kernel's permission set
// here first).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kern)(KArgs...), int64_t blocks, int threads, size_t smem, int S, cudaStream_t s,
                           Args... args) {
    if (S > 8) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = unsigned(S);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, KArgs(args)...);
}

}  // namespace mgs
