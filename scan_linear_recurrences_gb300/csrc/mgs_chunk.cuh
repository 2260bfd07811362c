// Shared machinery of the time-chunked path of matrix_scan and
// matrix_affine_scan (few lanes, long sequences): a shape-only chunk plan, the
// workspace layout, the carry-chain kernel and small k x k helpers.
//
// The path is a reduce-then-scan in three launches on the caller's stream:
//   1. every chunk but the last in carry order (the first for the backward)
//      computes its aggregate - the chunk's map from its incoming carry to its
//      outgoing one - from the identity;
//   2. one block per lane group bulk-copies that group's aggregates into
//      shared memory and composes them in carry order, writing the incoming
//      carry of every chunk;
//   3. every chunk reruns its recurrence from its carry and writes outputs.
// Stream order is the only synchronisation: no flags, no waits on other
// blocks, no zeroing of the workspace, and every run adds in the same order,
// so results are reproducible bit for bit.
#pragma once

#include <utility>

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

// Workspace of the chunked path: three arrays of G*C items (lane group g,
// chunk c at item g*C + c) - the aggregates' matrices, their offsets, and the
// incoming carries - of mM, mC and mE floats per item, each array starting
// on a 256-byte boundary.
struct ScanWs {
    float *M, *Cv, *E;
    __host__ __device__ static size_t arr(const ChunkPlan &p, int mf) {
        return align_up(size_t(p.G * p.C) * size_t(mf) * 4, 256);
    }
    __host__ __device__ static size_t bytes(const ChunkPlan &p, int mM, int mC, int mE) {
        return arr(p, mM) + arr(p, mC) + arr(p, mE);
    }
    __host__ __device__ ScanWs(unsigned char *ws, const ChunkPlan &p, int mM, int mC)
        : M(reinterpret_cast<float *>(ws)), Cv(reinterpret_cast<float *>(ws + arr(p, mM))),
          E(reinterpret_cast<float *>(ws + arr(p, mM) + arr(p, mC))) {}
};

// Item -> (lane group, chunk) of the chunked path and the lane group's place
// in the batch (nper items per lane group, chunks from cfirst).
struct ChunkItem {
    int64_t g, c, bi;
    int head0;
    __device__ ChunkItem(int64_t item, int64_t nper, int64_t cfirst, int64_t gpb, int lpw) {
        const unsigned q = unsigned(item) / unsigned(nper);  // 32-bit: items, nper and gpb are below 2^32
        g = q;
        c = cfirst + (item - int64_t(q) * nper);
        const unsigned b32 = q / unsigned(gpb);
        bi = b32;
        head0 = int(q - b32 * unsigned(gpb)) * lpw;
    }
};

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


// ---------------------------------------------------------------- carry chain
// Launch 2 of the chunked path: one block (one warp) per lane group g, over
// the group's aggregates in carry order.  DIR = +1 (forward scans):
//     E_0 = initial state,   E_{p+1} = M_p E_p (+ C_p),   p = 0 .. C-2;
// DIR = -1 (backward scans):
//     E_{C-1} = 0,           E_{p-1} = M_p E_p + C_p,     p = C-1 .. 1.
// MAT: the carries are k x k matrices (matrix_scan), thread (lane, col) of a
// lane's k-group holding column col; otherwise k-vectors (matrix_affine_scan),
// every thread of the group holding the whole vector (k^2 FMAs, no shuffles)
// and storing its own element.  The aggregates come into shared memory by 1-D
// bulk copies, `nb` per batch in two alternating buffers, so their loads are
// all in flight at once instead of one memory latency per step.
// Per item floats: mM = LPW k^2; mC (and mE) = LPW k^2 (MAT) or LPW k.
template <int K, bool MAT, bool HASC, int DIR>
__global__ void __launch_bounds__(32)
    chain_kernel(const float *__restrict__ Ms, const float *__restrict__ Cs, float *__restrict__ Es,
                 const float *__restrict__ init, int64_t C, int64_t gpb, int64_t H, int nb, DevCtl ctl) {
    constexpr int LPW = 32 / K;
    constexpr int mM = LPW * K * K, mC = MAT ? LPW * K * K : LPW * K, mE = mC;
    constexpr int STEPF = mM + (HASC ? mC : 0);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *buf = reinterpret_cast<float *>(smem_raw);  // 2 buffers of nb * STEPF floats
    uint64_t *bars = reinterpret_cast<uint64_t *>(buf + 2 * size_t(nb) * STEPF);

    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    const int64_t bi = g / gpb;
    const int head0 = int(g - bi * gpb) * LPW;
    const int sub = lane / K, col = lane % K;
    const bool active = head0 + sub < H;
    const int64_t nsteps = C - 1;
    const int64_t nbat = (nsteps + nb - 1) / nb;
    if (lane == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // launched as a programmatic dependent of launch 1: wait for its
    // aggregates, then let launch 3 be scheduled
    pdl_wait();
    pdl_trigger();
    const uint64_t pol = policy_evict_first();
    // batch bt: steps [bt*nb, bt*nb + n); their aggregates are the contiguous
    // items g*C + plo .. g*C + plo + n - 1
    auto batch_n = [&](int64_t bt) { return int(min64(nb, nsteps - bt * nb)); };
    auto batch_plo = [&](int64_t bt) { return DIR > 0 ? bt * nb : C - bt * nb - batch_n(bt); };
    auto issue = [&](int64_t bt) {  // lane 0 only
        const int n = batch_n(bt), b = int(bt & 1);
        const int64_t it0 = g * C + batch_plo(bt);
        float *dst = buf + size_t(b) * nb * STEPF;
        mbar_arrive_expect_tx(&bars[b], uint32_t(n) * STEPF * 4u);
        bulk_g2s(dst, Ms + it0 * mM, uint32_t(n) * mM * 4u, &bars[b], pol);
        if constexpr (HASC) bulk_g2s(dst + size_t(n) * mM, Cs + it0 * mC, uint32_t(n) * mC * 4u, &bars[b], pol);
    };
    if (lane == 0) {
        if (nbat > 0) issue(0);
        if (nbat > 1) issue(1);
    }

    // the carry of the first chunk in carry order
    float x[K];
#pragma unroll
    for (int i = 0; i < K; ++i) x[i] = 0.f;
    if constexpr (MAT) {
        if (DIR > 0) {  // P_0 = I
#pragma unroll
            for (int i = 0; i < K; ++i) x[i] = (i == col) ? 1.f : 0.f;
        }
    } else {
        if (DIR > 0 && init != nullptr && active) lds_row_global<K>(init + (bi * H + head0 + sub) * K, x);
    }
    auto store = [&](int64_t chunk) {
        if (!active) return;
        float *e = Es + (g * C + chunk) * mE;
        if constexpr (MAT) {
            st_ws_col<K>(e + sub * K * K, col, x);
        } else {
            float v = x[0];
#pragma unroll
            for (int i = 1; i < K; ++i) v = (i == col) ? x[i] : v;
            __stcg(e + sub * K + col, v);
        }
    };
    store(DIR > 0 ? 0 : C - 1);

    uint32_t phase = 0;
    for (int64_t bt = 0; bt < nbat; ++bt) {
        const int b = int(bt & 1);
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[b], (phase >> b) & 1u, ctl.timeout_ns));
        if (!ok) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            // the other buffer may still have a copy in flight
            if (bt + 1 < nbat && !mbar_wait_bounded(&bars[b ^ 1], (phase >> (b ^ 1)) & 1u, ctl.timeout_ns) &&
                lane == 0)
                record_error(ctl, ERR_DRAIN_TIMEOUT);
            __syncwarp();
            return;
        }
        phase ^= 1u << b;
        const int n = batch_n(bt);
        const float *sm = buf + size_t(b) * nb * STEPF;
        const float *sc = sm + size_t(n) * mM;
        for (int q = 0; q < n; ++q) {
            const int idx = DIR > 0 ? q : n - 1 - q;  // position of this step's aggregate in the batch
            const float *Mp = sm + idx * mM + sub * K * K;
            float y[K];
#pragma unroll
            for (int i = 0; i < K; ++i) {
                float r[K];
                lds_row_smem<K>(Mp + i * K, r);
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int m = 0; m < K; ++m) {
                    if (m & 1) s1 = fmaf(r[m], x[m], s1);
                    else s0 = fmaf(r[m], x[m], s0);
                }
                y[i] = s0 + s1;
            }
            if constexpr (HASC) {
#pragma unroll
                for (int i = 0; i < K; ++i)
                    y[i] += MAT ? sc[idx * mC + sub * K * K + i * K + col] : sc[idx * mC + sub * K + i];
            }
#pragma unroll
            for (int i = 0; i < K; ++i) x[i] = y[i];
            const int64_t k = bt * nb + q;
            store(DIR > 0 ? k + 1 : C - 2 - k);
        }
        __syncwarp();
        if (bt + 2 < nbat && lane == 0) {
            fence_proxy_async_smem();
            issue(bt + 2);
        }
    }
}

// Launches a one-warp-per-block kernel as a programmatic dependent of the
// previous kernel in the stream (the kernel calls pdl_wait() before reading
// what that kernel wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, int smem, cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Aggregates per batch of the chain kernel: about 48 KB of shared memory per
// buffer, at most the whole chain.
inline int chain_batch(int64_t C, int step_floats) {
    const int64_t nb = (48 * 1024) / (int64_t(step_floats) * 4);
    return int(nb < 1 ? 1 : (nb > C - 1 ? C - 1 : nb));
}
inline size_t chain_smem(int nb, int step_floats) { return size_t(2) * nb * step_floats * 4 + 2 * sizeof(uint64_t); }

// Launches the chain kernel for lane-group count G.
template <int K, bool MAT, bool HASC, int DIR>
cudaError_t launch_chain(const float *Ms, const float *Cs, float *Es, const float *init, int64_t G, int64_t C,
                         int64_t gpb, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    constexpr int LPW = 32 / K;
    constexpr int stepf = LPW * K * K + (HASC ? (MAT ? LPW * K * K : LPW * K) : 0);
    const int nb = chain_batch(C, stepf);
    const int smem = int(chain_smem(nb, stepf));
    cudaError_t e = ensure_smem_attr((const void *)chain_kernel<K, MAT, HASC, DIR>, smem);
    if (e != cudaSuccess) return e;
    if (G > 0x7fffffff) return cudaErrorInvalidConfiguration;
    return launch_pdl(chain_kernel<K, MAT, HASC, DIR>, dim3(unsigned(G)), smem, s, Ms, Cs, Es, init, C, gpb, H, nb, ctl);
}

}  // namespace mgs
