// matrix_scan forward and backward ("mingru-scans" home page, scan-op table,
// matrix_scan row): prefix products P_t = A_t P_{t-1}, P_0 = I, and the
// adjoint Lambda_t = G_t + A_{t+1}^T Lambda_{t+1}, dA_t = Lambda_t P_{t-1}^T.
//
// Layout of the work: a warp owns 32/k adjacent heads of one batch row; inside
// a head's k-thread group, thread j owns COLUMN j of P (forward) and of Lambda
// (backward), so the k x k product per step is a broadcast read of A_t from
// shared memory and k^2 register FMAs with no shuffles.  Inputs stream through
// the same per-warp TMA bulk-copy ring as matrix_affine_scan.
#include "mgs_tiles.cuh"

namespace mgs {
namespace {

template <int K>
struct MsShape {
    static constexpr int LPW = 32 / K;
    static constexpr int MF = LPW * K * K;  // floats of one k x k tensor per time step
    static constexpr int TS = K >= 16 ? 2 : (K >= 8 ? 4 : 8);
    static constexpr int NS = 4;
    using TM = HeadTile<K * K, LPW>;
};

constexpr int kWarpsPerBlock = 1;

template <int STEPF, int TS, int NS, int EXTRAF>
struct MsLayout {
    static constexpr size_t ring_bytes = size_t(NS) * TS * STEPF * sizeof(float);
    static constexpr size_t extra_bytes = size_t(EXTRAF) * sizeof(float);
    static constexpr size_t warp_bytes = align_up(ring_bytes + extra_bytes + NS * sizeof(uint64_t), 128);
};

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

// ---------------------------------------------------------------- forward
template <int K>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    ms_fwd_kernel(const __grid_constant__ CUtensorMap tmA, float *__restrict__ P, int64_t B,
                  int64_t T, int64_t H, int64_t groups_per_b, DevCtl ctl) {
    using S = MsShape<K>;
    constexpr int STEPF = S::MF;
    using L = MsLayout<STEPF, S::TS, S::NS, 0>;
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = int64_t(blockIdx.x) * kWarpsPerBlock + warp;
    if (g >= B * groups_per_b) return;
    unsigned char *base = smem_raw + size_t(warp) * L::warp_bytes;
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
                smem_matvec<K>(st + u * STEPF + sub * K * K, pc, nc);
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
    using L = MsLayout<STEPF, S::TS, S::NS, XF>;
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = int64_t(blockIdx.x) * kWarpsPerBlock + warp;
    if (g >= B * groups_per_b) return;
    unsigned char *base = smem_raw + size_t(warp) * L::warp_bytes;
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
                const float *At = st + q * S::MF + sub * K * K;
                const float *Gt = At + S::TS * S::MF;
                const float *Pp = At + 2 * S::TS * S::MF;
                float lc[K];  // column `col` of Lambda_t
#pragma unroll
                for (int i = 0; i < K; ++i) lc[i] = Gt[i * K + col] + mu[i];
                // exchange Lambda_t so this thread can form row `col` of dA_t
#pragma unroll
                for (int i = 0; i < K; ++i) xw[i * K + col] = lc[i];
                __syncwarp();
                float lrow[K];  // row `col` of Lambda_t
#pragma unroll
                for (int jj = 0; jj < K; ++jj) lrow[jj] = xw[col * K + jj];
                float darow[K];
                if (t >= 1) {
                    smem_matvec<K>(Pp, lrow, darow);  // dA[row][m] = sum_j L[row][j] P[m][j]
                } else {
#pragma unroll
                    for (int m = 0; m < K; ++m) darow[m] = lrow[m];  // P_0 = I
                }
                smem_matvec_t<K>(At, lc, mu);
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
    using L = MsLayout<S::MF, S::TS, S::NS, 0>;
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
    using L = MsLayout<3 * S::MF, S::TS, S::NS, S::MF>;
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

}  // namespace

size_t ms_workspace_bytes(int64_t, int64_t, int64_t, int, bool) { return 0; }

cudaError_t launch_ms_fwd(int K, const float *A, float *P, int64_t B, int64_t T, int64_t H,
                          void *, size_t, const DevCtl &ctl, cudaStream_t s) {
    switch (K) {
        case 1: return ms_fwd_t<1>(A, P, B, T, H, ctl, s);
        case 2: return ms_fwd_t<2>(A, P, B, T, H, ctl, s);
        case 4: return ms_fwd_t<4>(A, P, B, T, H, ctl, s);
        case 8: return ms_fwd_t<8>(A, P, B, T, H, ctl, s);
        case 16: return ms_fwd_t<16>(A, P, B, T, H, ctl, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_ms_bwd(int K, const float *A, const float *P, const float *G, float *dA,
                          int64_t B, int64_t T, int64_t H, void *, size_t, const DevCtl &ctl,
                          cudaStream_t s) {
    switch (K) {
        case 1: return ms_bwd_t<1>(A, P, G, dA, B, T, H, ctl, s);
        case 2: return ms_bwd_t<2>(A, P, G, dA, B, T, H, ctl, s);
        case 4: return ms_bwd_t<4>(A, P, G, dA, B, T, H, ctl, s);
        case 8: return ms_bwd_t<8>(A, P, G, dA, B, T, H, ctl, s);
        case 16: return ms_bwd_t<16>(A, P, G, dA, B, T, H, ctl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mgs
