// Device helpers shared by the scan kernels: mbarrier-tracked 1-D bulk copies
// (the Hopper/Blackwell TMA bulk path, no tensor map needed), bounded waits
// that record an error instead of hanging, and warp-level utilities.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (the descriptor type only; no driver calls here)
#include <cuda_runtime.h>

namespace mgs {

// Bits of the per-device error word.
enum : unsigned {
    ERR_MBAR_TIMEOUT = 1u,     // a bulk-copy barrier wait gave up
    ERR_FLAG_TIMEOUT = 2u,     // a look-back / flag wait gave up
    ERR_DRAIN_TIMEOUT = 4u,    // waiting for in-flight copies after an error gave up
};

// Launch-wide parameters every kernel receives.
struct DevCtl {
    unsigned *err;        // per-device error word (device address)
    uint64_t timeout_ns;  // bounded-wait limit
};

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(const DevCtl &c, unsigned bits) {
    atomicOr(c.err, bits);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// Waits for phase `parity` of `bar` to complete; gives up after the launch's
// timeout and returns false (the caller records the error and drains).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > timeout_ns) return false;
    }
}

// Flag publication for cross-warp carries: data stores, then a gpu-scope
// fence by every writer lane, then one release store of the flag; readers
// acquire the flag (each reading lane on its own) before touching the data.
__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until *flag is nonzero; returns the value, or 0 after the timeout.
__device__ __forceinline__ unsigned wait_flag_bounded(const unsigned *flag, uint64_t timeout_ns) {
    unsigned v = ld_acquire_gpu(flag);
    if (v != 0) return v;
    const uint64_t t0 = global_ns();
    while (true) {
        __nanosleep(64);
        v = ld_acquire_gpu(flag);
        if (v != 0) return v;
        if (global_ns() - t0 > timeout_ns) return 0;
    }
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before the previous kernel in the stream ends;
// pdl_wait() blocks until that kernel has completed and its writes are
// visible (it returns at once for a normal launch).  pdl_trigger() lets the
// next such kernel be scheduled once every block of this one has called it
// or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// L2 eviction hint for data streamed once.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// L2 eviction hint for data read again shortly (by a later launch).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared, completion signalled on `bar` as tx bytes.
// Both addresses must be 16-byte aligned and `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Tiled TMA loads through a tensor map (cp.async.bulk.tensor), completion on
// `bar` as tx bytes.  The map lives in kernel parameter space
// (__grid_constant__).  Coordinates are element indices, innermost first; the
// innermost one must be a multiple of 16 bytes, the others may be negative or
// past the end (those box elements are zero-filled).
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const CUtensorMap *map, int x, int y,
                                           uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst_smem, const CUtensorMap *map, int x, int y,
                                           int z, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// Tiled TMA store shared -> global through a tensor map (2-D), tracked as a
// bulk async-group of the issuing thread; the coordinates must not be
// negative.  bulk_commit() closes the group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, const void *src_smem) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_addr(src_smem))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed group of this thread has finished reading its
// shared-memory source (the source may then be reused or released; the
// global writes complete on their own).
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Hardware base-2 exponential and logarithm (MUFU; relative error of a few
// ulp for ex2, absolute error about 2^-22 for lg2; subnormal results flush).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Streaming (evict-first) vector stores for outputs written once.
__device__ __forceinline__ void st_cs(float *p, float v) { __stcs(p, v); }
__device__ __forceinline__ void st_cs4(float *p, float4 v) { __stcs(reinterpret_cast<float4 *>(p), v); }

// After a failed wait: waits (bounded) for every stage that still has copies in
// flight, so the warp never exits with TMA writes pending into its shared memory.
static __device__ __noinline__ void drain_ring(uint64_t *bar, int ns, uint32_t inflight, uint32_t phase,
                                        DevCtl c, int lane) {
    bool ok = true;
    for (int s = 0; s < ns; ++s)
        if (inflight & (1u << s))
            if (!mbar_wait_bounded(&bar[s], (phase >> s) & 1u, c.timeout_ns)) ok = false;
    if (!ok && lane == 0) record_error(c, ERR_DRAIN_TIMEOUT);
    __syncwarp();
}

// Per-warp ring of NS stages with one full-barrier each.  Lane 0 produces (bulk
// copies), the whole warp consumes.  After a failed wait, drain() waits (again
// bounded) for every stage that still has copies in flight so the warp never
// exits with TMA writes pending into its shared memory.
template <int NS>
struct WarpRing {
    uint64_t *bar;         // NS barriers in shared memory
    uint32_t inflight;     // bit s set: stage s has an armed, unconsumed phase
    uint32_t phase;        // bit s: parity expected next on stage s

    __device__ __forceinline__ void init(uint64_t *bars, int lane) {
        bar = bars;
        inflight = 0;
        phase = 0;
        if (lane == 0) {
            for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
            fence_barrier_init();
        }
        __syncwarp();
    }
    // Marks stage s armed (called by all lanes, uniformly, after lane 0 issued).
    __device__ __forceinline__ void armed(int s) { inflight |= (1u << s); }

    // All lanes wait for stage s; returns false on timeout.
    __device__ __forceinline__ bool wait(int s, const DevCtl &c) {
        bool ok = mbar_wait_bounded(&bar[s], (phase >> s) & 1u, c.timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            phase ^= (1u << s);
            inflight &= ~(1u << s);
        }
        return ok;
    }

    __device__ __forceinline__ void drain(const DevCtl &c, int lane) {
        drain_ring(bar, NS, inflight, phase, c, lane);
    }
};

}  // namespace mgs
