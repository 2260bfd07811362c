// Shared machinery of the time-chunked kernels (matrix_scan and
// matrix_affine_scan): a shape-only chunk plan, the workspace layout, flag
// publication and the bounded look-back wait, and small k x k helpers.
#pragma once

#include "mgs_tiles.cuh"

namespace mgs {

// y = M x for a k x k row-major M in shared memory (broadcast reads).
template <int K>
__device__ __forceinline__ void smem_matvec(const float *M, const float (&x)[K], float (&y)[K]) {
#pragma unroll
    for (int i = 0; i < K; ++i) {
        float r[K];
        if constexpr (K >= 4) {
#pragma unroll
            for (int c = 0; c < K / 4; ++c) {
                float4 q = reinterpret_cast<const float4 *>(M + i * K)[c];
                r[4 * c] = q.x; r[4 * c + 1] = q.y; r[4 * c + 2] = q.z; r[4 * c + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < K; ++c) r[c] = M[i * K + c];
        }
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int m = 0; m < K; ++m) {
            if (m & 1) s1 = fmaf(r[m], x[m], s1);
            else s0 = fmaf(r[m], x[m], s0);
        }
        y[i] = s0 + s1;
    }
}

// y = M^T x for a k x k row-major M in shared memory: y[m] = sum_i M[i][m] x[i].
template <int K>
__device__ __forceinline__ void smem_matvec_t(const float *M, const float (&x)[K], float (&y)[K]) {
#pragma unroll
    for (int m = 0; m < K; ++m) y[m] = 0.f;
#pragma unroll
    for (int i = 0; i < K; ++i) {
        float r[K];
        if constexpr (K >= 4) {
#pragma unroll
            for (int c = 0; c < K / 4; ++c) {
                float4 q = reinterpret_cast<const float4 *>(M + i * K)[c];
                r[4 * c] = q.x; r[4 * c + 1] = q.y; r[4 * c + 2] = q.z; r[4 * c + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < K; ++c) r[c] = M[i * K + c];
        }
#pragma unroll
        for (int m = 0; m < K; ++m) y[m] = fmaf(r[m], x[i], y[m]);
    }
}

struct ChunkPlan {
    int64_t G;  // lane groups (warps per chunk index)
    int64_t C;  // chunks per lane group (1: no chunking, no workspace)
    int64_t L;  // chunk length in steps (multiple of 4)
};

// Shape-only plan (the workspace size must not depend on the device): chunk
// only when there are fewer than 256 lane groups and T >= 64, aiming at about
// 1024 (group, chunk) items, with chunks of 32 to 64 steps so that the second
// pass over a chunk, a few microseconds after the first, still finds its
// inputs in L2 (about a thousand resident items x 64 KB stays well inside L2).
#ifndef MGS_CHUNK_ITEMS
#define MGS_CHUNK_ITEMS 1024
#endif
#ifndef MGS_CHUNK_LMIN
#define MGS_CHUNK_LMIN 32
#endif
#ifndef MGS_CHUNK_LMAX
#define MGS_CHUNK_LMAX 64
#endif
__host__ __device__ inline ChunkPlan plan_chunks(int64_t B, int64_t T, int64_t H, int K) {
    const int64_t lpw = 32 / K;
    ChunkPlan p;
    p.G = B * ((H + lpw - 1) / lpw);
    p.C = 1;
    p.L = T;
    if (p.G >= 256 || T < 64) return p;
    const int64_t c0 = (MGS_CHUNK_ITEMS + p.G - 1) / p.G;
    int64_t L = (T + c0 - 1) / c0;
    L = L < MGS_CHUNK_LMIN ? MGS_CHUNK_LMIN : (L > MGS_CHUNK_LMAX ? MGS_CHUNK_LMAX : L);
    L = (L + 3) / 4 * 4;
    p.L = L;
    p.C = (T + L - 1) / L;
    if (p.C < 2) {
        p.C = 1;
        p.L = T;
    }
    return p;
}

// Workspace: [ticket | one flag per item | nmat slots of LPW*K*K floats per item]
struct ChunkWs {
    unsigned *ticket, *flags;
    float *slots;
    int64_t items;
    int mf;  // floats per slot
    __host__ __device__ static size_t header_bytes(const ChunkPlan &p) {
        return align_up(256 + size_t(p.G * p.C) * 4, 256);
    }
    static size_t bytes(const ChunkPlan &p, int K, int nmat) {
        return header_bytes(p) + size_t(nmat) * size_t(p.G * p.C) * (32 / K) * K * K * 4;
    }
    __device__ ChunkWs(unsigned char *ws, const ChunkPlan &p, int mf_)
        : ticket(reinterpret_cast<unsigned *>(ws)), flags(reinterpret_cast<unsigned *>(ws + 256)),
          slots(reinterpret_cast<float *>(ws + header_bytes(p))), items(p.G * p.C), mf(mf_) {}
    // slot m of item
    __device__ float *slot(int m, int64_t item) const { return slots + (m * items + item) * mf; }
};

enum : unsigned { FLAG_AGG = 1u, FLAG_INCL = 2u };

// Column `col` of a k x k row-major matrix in the workspace (bypassing L1).
template <int K>
__device__ __forceinline__ void ld_ws_col(const float *mat, int col, float (&x)[K]) {
#pragma unroll
    for (int i = 0; i < K; ++i) x[i] = __ldcg(mat + i * K + col);
}
template <int K>
__device__ __forceinline__ void st_ws_col(float *mat, int col, const float (&x)[K]) {
#pragma unroll
    for (int i = 0; i < K; ++i) __stcg(mat + i * K + col, x[i]);
}

// y = X x, where X is held one column per thread of the k-group (this thread
// holds column `col` in xc): X goes through the warp's exchange buffer.
template <int K>
__device__ __forceinline__ void group_matvec(float *xw, int col, const float (&xc)[K], const float (&x)[K],
                                             float (&y)[K]) {
#pragma unroll
    for (int i = 0; i < K; ++i) xw[i * K + col] = xc[i];
    __syncwarp();
    smem_matvec<K>(xw, x, y);
    __syncwarp();
}

// Publishes `value` for this item once the whole warp has stored its data.
// The warp barrier orders every lane's data stores before lane 0's fence and
// release store (one fence per warp rather than one per lane).
__device__ __forceinline__ void publish(unsigned *flag, unsigned value, int lane) {
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        st_release_gpu(flag, value);
    }
    __syncwarp();
}

// Lane 0 waits (bounded) for a nonzero flag and broadcasts the value it saw;
// that broadcast value alone drives control flow, so the warp never diverges
// even if the flag advances (1 -> 2) meanwhile.  Each lane then acquires the
// flag itself until it reads a value at least that new (flags only grow), so
// its own later loads see the data published before that value.  Returns 0,
// uniformly, on timeout.
__device__ __forceinline__ unsigned lookback_flag(const unsigned *flag, int lane, const DevCtl &ctl) {
    unsigned f = 0;
    if (lane == 0) f = wait_flag_bounded(flag, ctl.timeout_ns);
    f = __shfl_sync(0xffffffffu, f, 0);
    if (f == 0) return 0;
    bool ok = true;
    unsigned v = ld_acquire_gpu(flag);
    if (v < f) {
        const uint64_t t0 = global_ns();
        while (v < f) {
            __nanosleep(32);
            v = ld_acquire_gpu(flag);
            if (v < f && global_ns() - t0 > ctl.timeout_ns) {
                ok = false;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok) ? f : 0u;
}

// Windowed look-back.  Scans the items of one lane group before (dir = -1) or
// after (dir = +1) chunk c, 32 at a time (lane j reads the flag of chunk
// c + dir*(1 + j)), for the nearest one whose inclusive value is published,
// waiting (bounded) until every chunk between it and c has published at least
// its aggregate.  Returns that chunk index, or -1 after the timeout; the result
// is uniform across the warp.  Each lane acquires the flag it reads and the
// closing __syncwarp (which orders memory among the warp's lanes) lets every
// lane read the data of all the chunks in the window.
__device__ __forceinline__ int64_t find_inclusive(const unsigned *flags, int64_t c, int dir, int64_t C, int lane,
                                                  const DevCtl &ctl) {
    const uint64_t t0 = global_ns();
    for (int64_t base = c + dir; base >= 0 && base < C; base += int64_t(dir) * 32) {
        const int64_t p = base + int64_t(dir) * lane;
        const bool valid = p >= 0 && p < C;
        unsigned f = valid ? ld_acquire_gpu(flags + p) : 0u;
        while (true) {
            const unsigned incl = __ballot_sync(0xffffffffu, valid && f == FLAG_INCL);
            const int first = incl ? __ffs(int(incl)) - 1 : 32;
            const bool need = valid && lane < first;
            const unsigned missing = __ballot_sync(0xffffffffu, need && f == 0u);
            if (missing == 0u) {
                if (first < 32) {
                    __syncwarp();
                    return base + int64_t(dir) * first;
                }
                break;  // 32 aggregates: look further
            }
            const bool late = (lane == 0) && (global_ns() - t0 > ctl.timeout_ns);
            if (__any_sync(0xffffffffu, late)) return -1;
            __nanosleep(64);
            if (need && f == 0u) f = ld_acquire_gpu(flags + p);
        }
    }
    return -1;
}

// K consecutive floats from global memory through L2 (16-byte loads when K >= 4).
template <int K>
__device__ __forceinline__ void lds_row_global(const float *p, float (&r)[K]) {
    if constexpr (K >= 4) {
#pragma unroll
        for (int c = 0; c < K / 4; ++c) {
            const float4 q = __ldcg(reinterpret_cast<const float4 *>(p) + c);
            r[4 * c] = q.x; r[4 * c + 1] = q.y; r[4 * c + 2] = q.z; r[4 * c + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < K; ++c) r[c] = __ldcg(p + c);
    }
}

// K consecutive floats from shared memory (16-byte loads when K >= 4).
template <int K>
__device__ __forceinline__ void lds_row_smem(const float *p, float (&r)[K]) {
    if constexpr (K >= 4) {
#pragma unroll
        for (int c = 0; c < K / 4; ++c) {
            const float4 q = reinterpret_cast<const float4 *>(p)[c];
            r[4 * c] = q.x; r[4 * c + 1] = q.y; r[4 * c + 2] = q.z; r[4 * c + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < K; ++c) r[c] = p[c];
    }
}

// k x k row-major matrix from the workspace into registers (L2, 16-byte loads).
template <int K>
__device__ __forceinline__ void ld_ws_mat(const float *m, float (&r)[K][K]) {
    if constexpr (K >= 4) {
#pragma unroll
        for (int i = 0; i < K; ++i)
#pragma unroll
            for (int c = 0; c < K / 4; ++c) {
                const float4 q = __ldcg(reinterpret_cast<const float4 *>(m + i * K) + c);
                r[i][4 * c] = q.x; r[i][4 * c + 1] = q.y; r[i][4 * c + 2] = q.z; r[i][4 * c + 3] = q.w;
            }
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i)
#pragma unroll
            for (int j = 0; j < K; ++j) r[i][j] = __ldcg(m + i * K + j);
    }
}

}  // namespace mgs
