// matrix_scan forward and backward ("mingru-scans" home page, scan-op table,
// matrix_scan row): prefix products P_t = A_t P_{t-1}, P_0 = I, and the
// adjoint Lambda_t = G_t + A_{t+1}^T Lambda_{t+1}, dA_t = Lambda_t P_{t-1}^T.
//
// Layout of the work: a warp owns 32/k adjacent heads of one batch row; inside
// a head's k-thread group, thread j owns COLUMN j of P (forward) and of Lambda
// (backward), so the k x k product per step is a broadcast read of A_t from
// shared memory and k^2 register FMAs with no shuffles.  Inputs stream through
// the same per-warp TMA bulk-copy ring as matrix_affine_scan.
#include <mutex>

#include "../../include/mgscan.h"
#include "mgs_chunk.cuh"

namespace mgs {
namespace {

template <int K>
struct MsShape {
    static constexpr int LPW = 32 / K;
    static constexpr int MF = LPW * K * K;  // floats of one k x k tensor per time step
    static constexpr int TS = K >= 16 ? 2 : (K >= 8 ? 4 : 8);
    static constexpr int NS = 4;
    using TM = MatTile<K, false>;
};

constexpr int kWarpsPerBlock = 1;

// Per-warp shared memory: the ring (stages of 1 or 3 swizzled k x k boxes,
// each a multiple of 1024 bytes for k >= 8), an exchange buffer, the barriers,
// and ALIGN bytes of slack so the kernel can align the base at run time.
template <int STEPF, int TS, int NS, int EXTRAF, size_t ALIGN>
struct MsLayout {
    static constexpr size_t ring_bytes = size_t(NS) * TS * STEPF * sizeof(float);
    static constexpr size_t extra_bytes = size_t(EXTRAF) * sizeof(float);
    static constexpr size_t warp_bytes = align_up(ring_bytes + extra_bytes + NS * sizeof(uint64_t), 128) + ALIGN;
};

// ---------------------------------------------------------------- forward
template <int K>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    ms_fwd_kernel(const __grid_constant__ CUtensorMap tmA, float *__restrict__ P, int64_t B,
                  int64_t T, int64_t H, int64_t groups_per_b, DevCtl ctl) {
    using S = MsShape<K>;
    constexpr int STEPF = S::MF;
    using L = MsLayout<STEPF, S::TS, S::NS, 0, S::TM::kAlign>;
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = int64_t(blockIdx.x) * kWarpsPerBlock + warp;
    if (g >= B * groups_per_b) return;
    unsigned char *base = align_smem(smem_raw + size_t(warp) * L::warp_bytes, S::TM::kAlign);
    float *ring = reinterpret_cast<float *>(base);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + L::ring_bytes + L::extra_bytes);

    const int64_t bi = g / groups_per_b;
    const int64_t head0 = (g % groups_per_b) * S::LPW;
    const int nl = int(min64(S::LPW, H - head0));
    const int sub = lane / K, col = lane % K;
    const bool active = sub < nl;
    const int64_t nblk = (T + S::TS - 1) / S::TS;

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) prefetch_tmap(&tmA);
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        mbar_arrive_expect_tx(&bars[s], uint32_t(S::TS * STEPF * 4));
        S::TM::load(ring + size_t(s) * S::TS * STEPF, &tmA, int(head0), int(bi * T + j * S::TS), &bars[s], pol);
    };
    const int npro = int(min64(S::NS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float pc[K];
#pragma unroll
    for (int i = 0; i < K; ++i) pc[i] = (i == col) ? 1.f : 0.f;
    float *pout = P + (bi * T * H + head0 + sub) * K * K + col;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t t0 = j * S::TS;
        const int n = int(min64(S::TS, T - t0));
        const float *st = ring + size_t(s) * S::TS * STEPF;
#pragma unroll
        for (int u = 0; u < S::TS; ++u) {
            if (u < n) {
                float nc[K];
                tile_matvec(TileRef<K, false>{st, u, sub}, pc, nc);
#pragma unroll
                for (int i = 0; i < K; ++i) pc[i] = nc[i];
                if (active) {
                    float *dst = pout + (t0 + u) * H * K * K;
#pragma unroll
                    for (int i = 0; i < K; ++i) st_cs(dst + i * K, pc[i]);
                }
            }
        }
        __syncwarp();
        if (j + S::NS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + S::NS);
            }
            rg.armed(s);
        }
    }
}

// ---------------------------------------------------------------- backward
template <int K>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    ms_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                  const __grid_constant__ CUtensorMap tmP, float *__restrict__ dA, int64_t B,
                  int64_t T, int64_t H, int64_t groups_per_b, DevCtl ctl) {
    using S = MsShape<K>;
    constexpr int STEPF = 3 * S::MF;  // A_t, G_t, P_{t-1}
    constexpr int XF = S::MF;         // Lambda exchange buffer, [lane][row][col]
    using L = MsLayout<STEPF, S::TS, S::NS, XF, S::TM::kAlign>;
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = int64_t(blockIdx.x) * kWarpsPerBlock + warp;
    if (g >= B * groups_per_b) return;
    unsigned char *base = align_smem(smem_raw + size_t(warp) * L::warp_bytes, S::TM::kAlign);
    float *ring = reinterpret_cast<float *>(base);
    float *xch = reinterpret_cast<float *>(base + L::ring_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + L::ring_bytes + L::extra_bytes);

    const int64_t bi = g / groups_per_b;
    const int64_t head0 = (g % groups_per_b) * S::LPW;
    const int nl = int(min64(S::LPW, H - head0));
    const int sub = lane / K, col = lane % K;
    const bool active = sub < nl;
    const int64_t nblk = (T + S::TS - 1) / S::TS;

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmP);
    }
    // Block j covers t = T-1-j*TS down to max(0, T-(j+1)*TS); box row of step u
    // is TS-1-u; the P box starts one row earlier and holds P_{t-1}.
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * S::TS * STEPF;
        const int r0 = int(bi * T + T - (j + 1) * S::TS);
        mbar_arrive_expect_tx(&bars[s], uint32_t(S::TS * STEPF * 4));
        S::TM::load(st, &tmA, int(head0), r0, &bars[s], pol);
        S::TM::load(st + S::TS * S::MF, &tmG, int(head0), r0, &bars[s], pol);
        S::TM::load(st + 2 * S::TS * S::MF, &tmP, int(head0), r0 - 1, &bars[s], pol);
    };
    const int npro = int(min64(S::NS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mu[K];  // column `col` of A_{t+1}^T Lambda_{t+1}
#pragma unroll
    for (int i = 0; i < K; ++i) mu[i] = 0.f;
    float *xw = xch + sub * K * K;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tt = T - 1 - j * S::TS;
        const int n = int(min64(S::TS, tt + 1));
        const float *st = ring + size_t(s) * S::TS * STEPF;
#pragma unroll
        for (int u = 0; u < S::TS; ++u) {
            if (u < n) {
                const int64_t t = tt - u;
                const int q = S::TS - 1 - u;  // box row of step u
                const TileRef<K, false> At{st, q, sub}, Gt{st + S::TS * S::MF, q, sub}, Pp{st + 2 * S::TS * S::MF, q, sub};
                float lc[K];  // column `col` of Lambda_t
#pragma unroll
                for (int i = 0; i < K; ++i) lc[i] = Gt.at(i, col) + mu[i];
                // exchange Lambda_t so this thread can form row `col` of dA_t
#pragma unroll
                for (int i = 0; i < K; ++i) xw[i * K + col] = lc[i];
                __syncwarp();
                float lrow[K];  // row `col` of Lambda_t
#pragma unroll
                for (int jj = 0; jj < K; ++jj) lrow[jj] = xw[col * K + jj];
                float darow[K];
                if (t >= 1) {
                    tile_matvec(Pp, lrow, darow);  // dA[row][m] = sum_j L[row][j] P[m][j]
                } else {
#pragma unroll
                    for (int m = 0; m < K; ++m) darow[m] = lrow[m];  // P_0 = I
                }
                tile_matvec_t(At, lc, mu);
                __syncwarp();
                if (active) {
                    float *dst = dA + ((bi * T + t) * H + head0 + sub) * K * K + col * K;
                    if constexpr (K >= 4) {
#pragma unroll
                        for (int c = 0; c < K / 4; ++c)
                            st_cs4(dst + 4 * c, make_float4(darow[4 * c], darow[4 * c + 1], darow[4 * c + 2], darow[4 * c + 3]));
                    } else {
#pragma unroll
                        for (int c = 0; c < K; ++c) st_cs(dst + c, darow[c]);
                    }
                }
            }
        }
        __syncwarp();
        if (j + S::NS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + S::NS);
            }
            rg.armed(s);
        }
    }
}

template <int K>
cudaError_t ms_fwd_t(const float *A, float *P, int64_t B, int64_t T, int64_t H, const DevCtl &ctl,
                     cudaStream_t s) {
    using S = MsShape<K>;
    using L = MsLayout<S::MF, S::TS, S::NS, 0, S::TM::kAlign>;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const int smem = int(L::warp_bytes * kWarpsPerBlock);
    CUtensorMap tA;
    cudaError_t e = S::TM::make(&tA, A, B * T, H, S::TS);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr((const void *)ms_fwd_kernel<K>, smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (B * gpb + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    ms_fwd_kernel<K><<<dim3(unsigned(blocks)), kWarpsPerBlock * 32, smem, s>>>(tA, P, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

template <int K>
cudaError_t ms_bwd_t(const float *A, const float *P, const float *G, float *dA, int64_t B,
                     int64_t T, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    using S = MsShape<K>;
    using L = MsLayout<3 * S::MF, S::TS, S::NS, S::MF, S::TM::kAlign>;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const int smem = int(L::warp_bytes * kWarpsPerBlock);
    CUtensorMap tA, tG, tP;
    cudaError_t e;
    if ((e = S::TM::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TM::make(&tG, G, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TM::make(&tP, P, B * T, H, S::TS)) != cudaSuccess) return e;
    e = ensure_smem_attr((const void *)ms_bwd_kernel<K>, smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (B * gpb + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    ms_bwd_kernel<K><<<dim3(unsigned(blocks)), kWarpsPerBlock * 32, smem, s>>>(tA, tG, tP, dA, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

// ================================================================ time-chunked path
// With few lanes (B*H/(32/k) warps well below the SM count) the sequential
// per-lane loop leaves the GPU idle.  T is then split into C chunks of L
// steps and the scan runs as a reduce-then-scan in three launches (see
// mgs_chunk.cuh): one warp per (lane group, chunk) item computes the chunk's
// aggregate, one block per lane group chains the aggregates into every
// chunk's incoming carry, and one warp per item reruns its chunk from the
// carry, writing outputs.  The inputs of the rerun are still in L2.
//   forward:  aggregate M = A_e ... A_s, carry E_{c+1} = M_c E_c (E_0 = I);
//   backward: aggregate (M, C) with mu_out = M mu_in + C, M = A_s^T ... A_e^T,
//             carry mu_in(c-1) = M_c mu_in(c) + C_c (mu_in(C-1) = 0).

template <int K>
struct MsChunkShape {
    static constexpr int LPW = 32 / K;
    static constexpr int MF = LPW * K * K;
    static constexpr int FTS = K >= 16 ? 2 : 4;  // steps per stage, forward
    static constexpr int BTS = 2;                // steps per stage, backward
    static constexpr int NS = 4;
    using TM = MatTile<K>;
};


// Launch 1, forward: the product of the chunk's A_t (chunks 0 .. C-2).
template <int K>
__global__ void __launch_bounds__(32)
    ms_fwd_agg_kernel(const __grid_constant__ CUtensorMap tmA, float *__restrict__ Ms, int64_t T, int64_t gpb,
                      int64_t C, int64_t Lc, DevCtl ctl) {
    using S = MsChunkShape<K>;
    constexpr int TS = S::FTS, NS = S::NS, BOXF = TS * S::MF;
    using Lay = MsLayout<S::MF, TS, NS, 0, S::TM::kAlign>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TM::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + Lay::ring_bytes + Lay::extra_bytes);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C - 1, 0, gpb, S::LPW);
    const int sub = lane / K, col = lane % K;
    const QuadOffsets<K> qo(sub, col);  // this thread's offsets in a staged box
    const int64_t tb = it.c * Lc, len = min64(Lc, T - tb);
    const int64_t nb = (len + TS - 1) / TS;

    WarpRing<NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();  // launch 3 reads the chunk again
    if (lane == 0) prefetch_tmap(&tmA);
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        mbar_arrive_expect_tx(&bars[s], uint32_t(BOXF * 4));
        S::TM::load(ring + size_t(s) * BOXF, &tmA, it.head0, int(it.bi * T + tb + j * TS), &bars[s], pol);
    };
    const int npro = int(min64(NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float m[K];  // column `col` of the chunk product
#pragma unroll
    for (int i = 0; i < K; ++i) m[i] = (i == col) ? 1.f : 0.f;
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(TS, len - j * TS));
        const float *st = ring + size_t(s) * BOXF;
        if constexpr (K <= 8) {
            // A of step u + 1 is loaded while step u computes (rows past n are
            // staged box rows too, loaded and not used)
            float a[K][K];
            tile_load(TileRefQ<K>{st, qo}, a);
#pragma unroll
            for (int u = 0; u < TS; ++u) {
                float an[K][K];
                if (u + 1 < TS) tile_load(TileRefQ<K>{st + (u + 1) * S::MF, qo}, an);
                if (u < n) {
                    float nm[K];
                    reg_matvec(a, m, nm);
#pragma unroll
                    for (int i = 0; i < K; ++i) m[i] = nm[i];
                }
                if (u + 1 < TS) {
#pragma unroll
                    for (int i = 0; i < K; ++i)
#pragma unroll
                        for (int c = 0; c < K; ++c) a[i][c] = an[i][c];
                }
            }
        } else {  // k = 16: the block does not fit in registers twice
#pragma unroll
            for (int u = 0; u < TS; ++u) {
                if (u < n) {
                    float nm[K];
                    tile_matvec(TileRefQ<K>{st + u * S::MF, qo}, m, nm);
#pragma unroll
                    for (int i = 0; i < K; ++i) m[i] = nm[i];
                }
            }
        }
        __syncwarp();
        if (j + NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + NS);
            }
            rg.armed(s);
        }
    }
    st_ws_col<K>(Ms + (it.g * C + it.c) * S::MF + sub * K * K, col, m);
}

// Launch 3, forward: P_t from the chunk's carry (all chunks).
template <int K>
__global__ void __launch_bounds__(32)
    ms_fwd_out_kernel(const __grid_constant__ CUtensorMap tmA, float *__restrict__ P, const float *__restrict__ Es,
                      int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc, DevCtl ctl) {
    using S = MsChunkShape<K>;
    constexpr int TS = S::FTS, NS = S::NS, BOXF = TS * S::MF;
    using Lay = MsLayout<S::MF, TS, NS, 0, S::TM::kAlign>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TM::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + Lay::ring_bytes + Lay::extra_bytes);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C, 0, gpb, S::LPW);
    const int sub = lane / K, col = lane % K;
    const QuadOffsets<K> qo(sub, col);  // this thread's offsets in a staged box
    const bool active = it.head0 + sub < H;
    const int64_t tb = it.c * Lc, len = min64(Lc, T - tb);
    const int64_t nb = (len + TS - 1) / TS;

    WarpRing<NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) prefetch_tmap(&tmA);
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        mbar_arrive_expect_tx(&bars[s], uint32_t(BOXF * 4));
        S::TM::load(ring + size_t(s) * BOXF, &tmA, it.head0, int(it.bi * T + tb + j * TS), &bars[s], pol);
    };
    const int npro = int(min64(NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float m[K];  // column `col` of P_t, from the carry (P at the end of chunk c-1)
    pdl_wait();   // the carries of launch 2
    ld_ws_col<K>(Es + (it.g * C + it.c) * S::MF + sub * K * K, col, m);
    float *pout = P + (it.bi * T * H + it.head0 + sub) * K * K + col;
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t t0 = tb + j * TS;
        const int n = int(min64(TS, len - j * TS));
        const float *st = ring + size_t(s) * BOXF;
        auto put = [&](int u) {
            if (active) {
                float *dst = pout + (t0 + u) * H * K * K;
#pragma unroll
                for (int i = 0; i < K; ++i) st_cs(dst + i * K, m[i]);
            }
        };
        if constexpr (K <= 8) {
            float a[K][K];  // A of step u; step u + 1's is loaded while u computes
            tile_load(TileRefQ<K>{st, qo}, a);
#pragma unroll
            for (int u = 0; u < TS; ++u) {
                float an[K][K];
                if (u + 1 < TS) tile_load(TileRefQ<K>{st + (u + 1) * S::MF, qo}, an);
                if (u < n) {
                    float nm[K];
                    reg_matvec(a, m, nm);
#pragma unroll
                    for (int i = 0; i < K; ++i) m[i] = nm[i];
                    put(u);
                }
                if (u + 1 < TS) {
#pragma unroll
                    for (int i = 0; i < K; ++i)
#pragma unroll
                        for (int c = 0; c < K; ++c) a[i][c] = an[i][c];
                }
            }
        } else {  // k = 16: the block does not fit in registers twice
#pragma unroll
            for (int u = 0; u < TS; ++u) {
                if (u < n) {
                    float nm[K];
                    tile_matvec(TileRefQ<K>{st + u * S::MF, qo}, m, nm);
#pragma unroll
                    for (int i = 0; i < K; ++i) m[i] = nm[i];
                    put(u);
                }
            }
        }
        __syncwarp();
        if (j + NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + NS);
            }
            rg.armed(s);
        }
    }
}

// Launch 1, backward: (M, C) of chunks 1 .. C-1, t walking down the chunk.
template <int K>
__global__ void __launch_bounds__(32)
    ms_bwd_agg_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                      float *__restrict__ Ms, float *__restrict__ Cs, int64_t T, int64_t gpb, int64_t C, int64_t Lc,
                      DevCtl ctl) {
    using S = MsChunkShape<K>;
    constexpr int TS = S::BTS, NS = S::NS, BOXF = TS * S::MF;
    using Lay = MsLayout<2 * S::MF, TS, NS, 0, S::TM::kAlign>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TM::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + Lay::ring_bytes + Lay::extra_bytes);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C - 1, 1, gpb, S::LPW);
    const int sub = lane / K, col = lane % K;
    const QuadOffsets<K> qo(sub, col);  // this thread's offsets in a staged box
    const int64_t tb = it.c * Lc, te = min64(T, tb + Lc), len = te - tb;
    const int64_t nb = (len + TS - 1) / TS;

    WarpRing<NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmG);
    }
    // block j covers t = te-1-j*TS down to max(tb, te-(j+1)*TS); boxes start
    // at row te-(j+1)*TS, step u at box row TS-1-u
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        const int r0 = int(it.bi * T + te - (j + 1) * TS);
        float *st = ring + size_t(s) * 2 * BOXF;
        mbar_arrive_expect_tx(&bars[s], uint32_t(2 * BOXF * 4));
        S::TM::load(st, &tmA, it.head0, r0, &bars[s], pol);
        S::TM::load(st + BOXF, &tmG, it.head0, r0, &bars[s], pol);
    };
    const int npro = int(min64(NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mu[K], mm[K];  // columns of the chunk map's offset C and matrix M
#pragma unroll
    for (int i = 0; i < K; ++i) {
        mu[i] = 0.f;
        mm[i] = (i == col) ? 1.f : 0.f;
    }
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tt = te - 1 - j * TS;
        const int n = int(min64(TS, tt - tb + 1));
        const float *st = ring + size_t(s) * 2 * BOXF;
        if constexpr (K <= 8) {
            // A and the G column of step u + 1 are loaded while step u computes
            float a[K][K], gc[K];
            tile_load(TileRefQ<K>{st + (TS - 1) * S::MF, qo}, a);
    #pragma unroll
            for (int i = 0; i < K; ++i) gc[i] = TileRefQ<K>{st + BOXF + (TS - 1) * S::MF, qo}.at_col(i);
    #pragma unroll
            for (int u = 0; u < TS; ++u) {
                float an[K][K], gn[K];
                if (u + 1 < TS) {
                    const int q1 = TS - 2 - u;
                    tile_load(TileRefQ<K>{st + q1 * S::MF, qo}, an);
    #pragma unroll
                    for (int i = 0; i < K; ++i) gn[i] = TileRefQ<K>{st + BOXF + q1 * S::MF, qo}.at_col(i);
                }
                if (u < n) {
                    float lc[K], nm[K];
    #pragma unroll
                    for (int i = 0; i < K; ++i) lc[i] = gc[i] + mu[i];
                    reg_matvec_t2(a, lc, mm, mu, nm);
    #pragma unroll
                    for (int i = 0; i < K; ++i) mm[i] = nm[i];
                }
                if (u + 1 < TS) {
    #pragma unroll
                    for (int i = 0; i < K; ++i) {
                        gc[i] = gn[i];
    #pragma unroll
                        for (int c = 0; c < K; ++c) a[i][c] = an[i][c];
                    }
                }
            }
        } else {  // k = 16: the block does not fit in registers twice
#pragma unroll
            for (int u = 0; u < TS; ++u) {
                if (u < n) {
                    const int q = TS - 1 - u;
                    const TileRefQ<K> At{st + q * S::MF, qo}, Gt{st + BOXF + q * S::MF, qo};
                    float lc[K], nm[K];
#pragma unroll
                    for (int i = 0; i < K; ++i) lc[i] = Gt.at_col(i) + mu[i];
                    tile_matvec_t2(At, lc, mm, mu, nm);
#pragma unroll
                    for (int i = 0; i < K; ++i) mm[i] = nm[i];
                }
            }
        }
        __syncwarp();
        if (j + NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + NS);
            }
            rg.armed(s);
        }
    }
    const int64_t slot = (it.g * C + it.c) * S::MF + sub * K * K;
    st_ws_col<K>(Ms + slot, col, mm);
    st_ws_col<K>(Cs + slot, col, mu);
}

// Launch 3, backward: dA_t from the chunk's carry mu_in (all chunks).
template <int K>
__global__ void __launch_bounds__(32)
    ms_bwd_out_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ CUtensorMap tmP, float *__restrict__ dA, const float *__restrict__ Es,
                      int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc, DevCtl ctl) {
    using S = MsChunkShape<K>;
    constexpr int TS = S::BTS, NS = S::NS, BOXF = TS * S::MF;
    using Lay = MsLayout<3 * S::MF, TS, NS, S::MF, S::TM::kAlign>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TM::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    float *xch = reinterpret_cast<float *>(sbase + Lay::ring_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + Lay::ring_bytes + Lay::extra_bytes);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C, 0, gpb, S::LPW);
    const int sub = lane / K, col = lane % K;
    const QuadOffsets<K> qo(sub, col);  // this thread's offsets in a staged box
    const bool active = it.head0 + sub < H;
    const int64_t tb = it.c * Lc, te = min64(T, tb + Lc), len = te - tb;
    const int64_t nb = (len + TS - 1) / TS;
    float *xw = xch + sub * K * K;

    WarpRing<NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmP);
    }
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        const int r0 = int(it.bi * T + te - (j + 1) * TS);
        float *st = ring + size_t(s) * 3 * BOXF;
        mbar_arrive_expect_tx(&bars[s], uint32_t(3 * BOXF * 4));
        S::TM::load(st, &tmA, it.head0, r0, &bars[s], pol);
        S::TM::load(st + BOXF, &tmG, it.head0, r0, &bars[s], pol);
        S::TM::load(st + 2 * BOXF, &tmP, it.head0, r0 - 1, &bars[s], pol);
    };
    const int npro = int(min64(NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mu[K];  // column `col` of A_{t+1}^T Lambda_{t+1}, from the carry
    pdl_wait();    // the carries of launch 2
    ld_ws_col<K>(Es + (it.g * C + it.c) * S::MF + sub * K * K, col, mu);
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tt = te - 1 - j * TS;
        const int n = int(min64(TS, tt - tb + 1));
        const float *st = ring + size_t(s) * 3 * BOXF;
#pragma unroll
        for (int u = 0; u < TS; ++u) {
            if (u < n) {
                const int64_t t = tt - u;
                const int q = TS - 1 - u;
                const TileRefQ<K> At{st + q * S::MF, qo}, Gt{st + BOXF + q * S::MF, qo},
                    Pp{st + 2 * BOXF + q * S::MF, qo};
                float lc[K], lrow[K], darow[K];
                if constexpr (K <= 8) {
                    // both blocks of the step into registers, every load issued
                    // before any use (the P box row of t = 0 is loaded, not used)
                    float a[K][K], pp[K][K];
                    tile_load(At, a);
                    tile_load(Pp, pp);
#pragma unroll
                    for (int i = 0; i < K; ++i) lc[i] = Gt.at_col(i) + mu[i];
#pragma unroll
                    for (int i = 0; i < K; ++i) xw[i * K + col] = lc[i];
                    __syncwarp();
#pragma unroll
                    for (int x = 0; x < K; ++x) lrow[x] = xw[col * K + x];
                    if (t >= 1) {
                        reg_matvec(pp, lrow, darow);  // dA[row][m] = sum_j L[row][j] P_{t-1}[m][j]
                    } else {
#pragma unroll
                        for (int x = 0; x < K; ++x) darow[x] = lrow[x];  // P_0 = I
                    }
                    reg_matvec_t(a, lc, mu);
                } else {
#pragma unroll
                    for (int i = 0; i < K; ++i) lc[i] = Gt.at_col(i) + mu[i];
#pragma unroll
                    for (int i = 0; i < K; ++i) xw[i * K + col] = lc[i];
                    __syncwarp();
#pragma unroll
                    for (int x = 0; x < K; ++x) lrow[x] = xw[col * K + x];
                    if (t >= 1) {
                        tile_matvec(Pp, lrow, darow);
                    } else {
#pragma unroll
                        for (int x = 0; x < K; ++x) darow[x] = lrow[x];
                    }
                    tile_matvec_t(At, lc, mu);
                }
                __syncwarp();
                if (active) {
                    float *dst = dA + ((it.bi * T + t) * H + it.head0 + sub) * K * K + col * K;
                    if constexpr (K >= 4) {
#pragma unroll
                        for (int x = 0; x < K / 4; ++x)
                            st_cs4(dst + 4 * x, make_float4(darow[4 * x], darow[4 * x + 1], darow[4 * x + 2], darow[4 * x + 3]));
                    } else {
#pragma unroll
                        for (int x = 0; x < K; ++x) st_cs(dst + x, darow[x]);
                    }
                }
            }
        }
        __syncwarp();
        if (j + NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + NS);
            }
            rg.armed(s);
        }
    }
}

template <int K>
cudaError_t ms_fwd_chunk_t(const float *A, float *P, int64_t B, int64_t T, int64_t H, const ChunkPlan &pl,
                           unsigned char *ws, const DevCtl &ctl, cudaStream_t s) {
    using S = MsChunkShape<K>;
    using Lay = MsLayout<S::MF, S::FTS, S::NS, 0, S::TM::kAlign>;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const ScanWs w(ws, pl, S::MF, 0);
    if (pl.G * pl.C > 0x7fffffff) return cudaErrorInvalidConfiguration;
    CUtensorMap tA;
    cudaError_t e;
    if ((e = S::TM::make(&tA, A, B * T, H, S::FTS)) != cudaSuccess) return e;
    const int smem = int(Lay::warp_bytes);
    if ((e = ensure_smem_attr((const void *)ms_fwd_agg_kernel<K>, smem)) != cudaSuccess) return e;
    if ((e = ensure_smem_attr((const void *)ms_fwd_out_kernel<K>, smem)) != cudaSuccess) return e;
    ms_fwd_agg_kernel<K><<<dim3(unsigned(pl.G * (pl.C - 1))), 32, smem, s>>>(tA, w.M, T, gpb, pl.C, pl.L, ctl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_chain<K, true, false, +1>(w.M, nullptr, w.E, nullptr, pl.G, pl.C, gpb, H, ctl, s)) != cudaSuccess)
        return e;
    return launch_pdl(ms_fwd_out_kernel<K>, dim3(unsigned(pl.G * pl.C)), smem, s, tA, P, w.E, T, H, gpb, pl.C, pl.L,
                      ctl);
}

template <int K>
cudaError_t ms_bwd_chunk_t(const float *A, const float *P, const float *G, float *dA, int64_t B, int64_t T,
                           int64_t H, const ChunkPlan &pl, unsigned char *ws, const DevCtl &ctl, cudaStream_t s) {
    using S = MsChunkShape<K>;
    using LayA = MsLayout<2 * S::MF, S::BTS, S::NS, 0, S::TM::kAlign>;
    using LayO = MsLayout<3 * S::MF, S::BTS, S::NS, S::MF, S::TM::kAlign>;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const ScanWs w(ws, pl, S::MF, S::MF);
    if (pl.G * pl.C > 0x7fffffff) return cudaErrorInvalidConfiguration;
    CUtensorMap tA, tG, tP;
    cudaError_t e;
    if ((e = S::TM::make(&tA, A, B * T, H, S::BTS)) != cudaSuccess) return e;
    if ((e = S::TM::make(&tG, G, B * T, H, S::BTS)) != cudaSuccess) return e;
    if ((e = S::TM::make(&tP, P, B * T, H, S::BTS)) != cudaSuccess) return e;
    const int sa = int(LayA::warp_bytes), so = int(LayO::warp_bytes);
    if ((e = ensure_smem_attr((const void *)ms_bwd_agg_kernel<K>, sa)) != cudaSuccess) return e;
    if ((e = ensure_smem_attr((const void *)ms_bwd_out_kernel<K>, so)) != cudaSuccess) return e;
    ms_bwd_agg_kernel<K><<<dim3(unsigned(pl.G * (pl.C - 1))), 32, sa, s>>>(tA, tG, w.M, w.Cv, T, gpb, pl.C, pl.L,
                                                                           ctl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_chain<K, true, true, -1>(w.M, w.Cv, w.E, nullptr, pl.G, pl.C, gpb, H, ctl, s)) != cudaSuccess)
        return e;
    return launch_pdl(ms_bwd_out_kernel<K>, dim3(unsigned(pl.G * pl.C)), so, s, tA, tG, tP, dA, w.E, T, H, gpb, pl.C,
                      pl.L, ctl);
}

}  // namespace

size_t ms_workspace_bytes(int64_t B, int64_t T, int64_t H, int K, bool bwd) {
    const ChunkPlan p = plan_chunks(B, T, H, K);
    if (p.C <= 1) return 0;
    const int mf = 32 * K;  // floats of one k x k matrix per lane group
    return ScanWs::bytes(p, mf, bwd ? mf : 0, mf);
}

#define MS_DISPATCH(K_, CALL)            \
    switch (K_) {                        \
        case 1: return CALL(1);          \
        case 2: return CALL(2);          \
        case 4: return CALL(4);          \
        case 8: return CALL(8);          \
        case 16: return CALL(16);        \
        default: return cudaErrorInvalidValue; \
    }

cudaError_t launch_ms_fwd(int K, const float *A, float *P, int64_t B, int64_t T, int64_t H,
                          void *ws, size_t, const DevCtl &ctl, cudaStream_t s) {
    const ChunkPlan pl = plan_chunks(B, T, H, K);
    unsigned char *w = static_cast<unsigned char *>(ws);
    if (pl.C > 1) {
#define CALL_FC(k) ms_fwd_chunk_t<k>(A, P, B, T, H, pl, w, ctl, s)
        MS_DISPATCH(K, CALL_FC)
#undef CALL_FC
    }
#define CALL_F(k) ms_fwd_t<k>(A, P, B, T, H, ctl, s)
    MS_DISPATCH(K, CALL_F)
#undef CALL_F
}

cudaError_t launch_ms_bwd(int K, const float *A, const float *P, const float *G, float *dA,
                          int64_t B, int64_t T, int64_t H, void *ws, size_t, const DevCtl &ctl,
                          cudaStream_t s) {
    const ChunkPlan pl = plan_chunks(B, T, H, K);
    unsigned char *w = static_cast<unsigned char *>(ws);
    if (pl.C > 1) {
#define CALL_BC(k) ms_bwd_chunk_t<k>(A, P, G, dA, B, T, H, pl, w, ctl, s)
        MS_DISPATCH(K, CALL_BC)
#undef CALL_BC
    }
#define CALL_B(k) ms_bwd_t<k>(A, P, G, dA, B, T, H, ctl, s)
    MS_DISPATCH(K, CALL_B)
#undef CALL_B
}

}  // namespace mgs

// ================================================================ no-allocation scratch
// Scratch for mgs_matrix_scan_fwd_noalloc: one file-scope array per device
// context that loads the library.  Host code never uses the array's name as
// an address (in host code it is only a stand-in); the device address comes
// from cudaGetSymbolAddress, looked up once per device context with that
// device current (again if the context is torn down and re-created), and is
// passed to the kernel like any caller workspace.
namespace {
static __device__ __align__(256) unsigned char g_ms_noalloc_scratch[MGS_NOALLOC_SCRATCH_BYTES];

mgs::SymbolAddressCache g_scratch_cache;

cudaError_t noalloc_scratch_address(unsigned char **out) {
    void *p = nullptr;
    cudaError_t e = mgs::cached_symbol_address(g_scratch_cache, (const void *)&g_ms_noalloc_scratch, &p);
    *out = static_cast<unsigned char *>(p);
    return e;
}
}  // namespace

namespace mgs {

size_t ms_static_scratch_bytes() { return MGS_NOALLOC_SCRATCH_BYTES; }

cudaError_t launch_ms_fwd_static_scratch(int K, const float *A, float *P, int64_t B, int64_t T,
                                         int64_t H, const DevCtl &ctl, cudaStream_t s) {
    const size_t need = ms_workspace_bytes(B, T, H, K, false);
    if (need == 0) return launch_ms_fwd(K, A, P, B, T, H, nullptr, 0, ctl, s);
    if (need > MGS_NOALLOC_SCRATCH_BYTES) return cudaErrorInvalidValue;
    unsigned char *scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    return launch_ms_fwd(K, A, P, B, T, H, scratch, MGS_NOALLOC_SCRATCH_BYTES, ctl, s);
}

}  // namespace mgs
