// matrix_affine_scan forward and backward ("mingru-scans" home page, scan-op
// table, matrix_affine_scan row): h_t = A_t h_{t-1} + b_t over per-token k x k
// blocks, and its reverse-mode adjoint.
//
// Design (one GB300 SM runs several of these warps side by side):
//  * A warp owns 32/k consecutive heads of one batch row ("lanes"); k threads
//    per lane, thread i owning row i of every A_t and coordinate i of h.
//  * Inputs stream through a per-warp ring of NS stages in shared memory.  Each
//    stage holds TS time steps of every input; one tiled TMA load
//    (cp.async.bulk.tensor) per input fills it, tracked by one mbarrier.
//  * Forward: h_{t-1} is all-gathered inside the k-thread group with k
//    shuffles, then k FMAs give h_t[i]; the store is coalesced (128 B/warp).
//  * Backward walks t downwards: lambda_t = g_t + mu_{t+1}; db_t, the dA_t row
//    lambda_t[i] h_{t-1}^T and the next mu_t = A_t^T lambda_t (a butterfly
//    reduce-scatter over the group, k-1 shuffles) all come from registers, so
//    nothing beyond the outputs is written.
#include "mgs_tiles.cuh"

namespace mgs {
namespace {

template <int K>
struct MasShape {
    static constexpr int LPW = 32 / K;          // lanes (heads) per warp
    static constexpr int AF = LPW * K * K;      // floats of A per time step
    static constexpr int VF = LPW * K;          // floats of one per-lane vector per time step
    // time steps per stage: about 8-10 KB of A per stage
    static constexpr int TS = K >= 16 ? 4 : (K >= 8 ? 8 : 16);
    static constexpr int NS = 4;                // stages in flight
    using TA = HeadTile<K * K, LPW>;
    using TV = HeadTile<K, LPW>;
};

// Per-warp shared memory: NS stages of STAGEF floats, then NS barriers.
template <int STAGEF, int NS>
struct Ring {
    static constexpr size_t stage_bytes = size_t(STAGEF) * sizeof(float);
    static constexpr size_t ring_bytes = NS * stage_bytes;
    static constexpr size_t warp_bytes = align_up(ring_bytes + NS * sizeof(uint64_t), 128);
};

// Loads K consecutive floats from shared memory (16-byte aligned when K >= 4).
template <int K>
__device__ __forceinline__ void lds_row(const float *p, float (&r)[K]) {
    if constexpr (K >= 4) {
#pragma unroll
        for (int c = 0; c < K / 4; ++c) {
            float4 q = reinterpret_cast<const float4 *>(p)[c];
            r[4 * c + 0] = q.x;
            r[4 * c + 1] = q.y;
            r[4 * c + 2] = q.z;
            r[4 * c + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < K; ++c) r[c] = p[c];
    }
}

template <int K>
__device__ __forceinline__ void stg_row_cs(float *p, const float (&r)[K]) {
    if constexpr (K >= 4) {
#pragma unroll
        for (int c = 0; c < K / 4; ++c)
            st_cs4(p + 4 * c, make_float4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]));
    } else {
#pragma unroll
        for (int c = 0; c < K; ++c) st_cs(p + c, r[c]);
    }
}

// Sum over the K threads of an aligned group of p[c], delivered to the thread
// whose in-group index is c (butterfly reduce-scatter, K-1 shuffles).
template <int K>
__device__ __forceinline__ float group_reduce_scatter(const float (&p)[K], int row) {
    float v[K];
#pragma unroll
    for (int c = 0; c < K; ++c) v[c] = p[c];
#pragma unroll
    for (int o = K / 2; o >= 1; o >>= 1) {
        const bool up = (row & o) != 0;
#pragma unroll
        for (int c = 0; c < o; ++c) {
            const float send = up ? v[c] : v[c + o];
            const float keep = up ? v[c + o] : v[c];
            v[c] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// ---------------------------------------------------------------- forward
template <int K>
__global__ void __launch_bounds__(32)
    mas_fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const float *__restrict__ h0, float *__restrict__ h, int64_t B, int64_t T,
                   int64_t H, int64_t groups_per_b, DevCtl ctl) {
    using S = MasShape<K>;
    constexpr int A_STAGE = S::TS * S::AF, STAGEF = A_STAGE + S::TS * S::VF;
    using R = Ring<STAGEF, S::NS>;
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + R::ring_bytes);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * S::LPW;
    const int nl = int(min64(S::LPW, H - head0));
    const int sub = lane / K, row = lane % K, gbase = lane & ~(K - 1);
    const bool active = sub < nl;
    const int64_t nblk = (T + S::TS - 1) / S::TS;
    const int row0 = int(bi * T);

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * STAGEF;
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        S::TA::load(st, &tmA, head0, row0 + int(j * S::TS), &bars[s], pol);
        S::TV::load(st + A_STAGE, &tmB, head0, row0 + int(j * S::TS), &bars[s], pol);
    };

    const int npro = int(min64(S::NS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float hprev = (h0 != nullptr && active) ? h0[(bi * H + head0 + sub) * K + row] : 0.f;
    float *hout = h + (bi * T * H + head0 + sub) * K + row;  // + t*H*K per step
    const int64_t hstride = H * K;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(S::TS, T - j * S::TS));
        const float *sa = ring + size_t(s) * STAGEF + (sub * K + row) * K;
        const float *sb = ring + size_t(s) * STAGEF + A_STAGE + sub * K + row;
#pragma unroll
        for (int u = 0; u < S::TS; ++u) {
            if (u < n) {
                float a[K];
                lds_row<K>(sa + u * S::AF, a);
                float acc0 = sb[u * S::VF];
                float acc1 = 0.f;
#pragma unroll
                for (int c = 0; c < K; ++c) {
                    const float x = __shfl_sync(0xffffffffu, hprev, gbase + c);
                    if (c & 1)
                        acc1 = fmaf(a[c], x, acc1);
                    else
                        acc0 = fmaf(a[c], x, acc0);
                }
                hprev = acc0 + acc1;
                if (active) st_cs(hout, hprev);
                hout += hstride;
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
__global__ void __launch_bounds__(32)
    mas_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                   const __grid_constant__ CUtensorMap tmH, const float *__restrict__ h0,
                   float *__restrict__ dA, float *__restrict__ db, float *__restrict__ dh0, int64_t B,
                   int64_t T, int64_t H, int64_t groups_per_b, DevCtl ctl) {
    using S = MasShape<K>;
    constexpr int A_STAGE = S::TS * S::AF, V_STAGE = S::TS * S::VF;
    constexpr int STAGEF = A_STAGE + 2 * V_STAGE;  // A_t, g_t, h_{t-1}
    using R = Ring<STAGEF, S::NS>;
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + R::ring_bytes);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * S::LPW;
    const int nl = int(min64(S::LPW, H - head0));
    const int sub = lane / K, row = lane % K;
    const bool active = sub < nl;
    const int64_t nblk = (T + S::TS - 1) / S::TS;

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmH);
    }
    // Block j covers t = T-1-j*TS down to max(0, T-(j+1)*TS).  Its boxes start
    // at row bi*T + T-(j+1)*TS (possibly before this batch row: unused, and
    // zero-filled when negative) so step u (t = T-1-j*TS-u) sits at box row
    // TS-1-u.  The h box starts one row earlier and holds h_{t-1}.
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * STAGEF;
        const int r0 = int(bi * T + T - (j + 1) * S::TS);
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        S::TA::load(st, &tmA, head0, r0, &bars[s], pol);
        S::TV::load(st + A_STAGE, &tmG, head0, r0, &bars[s], pol);
        S::TV::load(st + A_STAGE + V_STAGE, &tmH, head0, r0 - 1, &bars[s], pol);
    };

    const int npro = int(min64(S::NS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mu = 0.f;  // (A_{t+1}^T lambda_{t+1})[row], zero past the end
    const int64_t hk = H * K;
    float *dbp = db + (bi * T * H + head0 + sub) * K + row;          // + t*H*K
    float *dAp = dA + (bi * T * H + head0 + sub) * K * K + row * K;  // + t*H*K*K

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tt = T - 1 - j * S::TS;
        const int n = int(min64(S::TS, tt + 1));
        const float *st = ring + size_t(s) * STAGEF;
#pragma unroll
        for (int u = 0; u < S::TS; ++u) {
            if (u < n) {
                const int64_t t = tt - u;
                const int q = S::TS - 1 - u;  // box row of step u
                const float lam = st[A_STAGE + q * S::VF + sub * K + row] + mu;
                float hp[K];
                if (t >= 1) {
                    lds_row<K>(st + A_STAGE + V_STAGE + q * S::VF + sub * K, hp);
                } else if (h0 != nullptr && active) {
#pragma unroll
                    for (int c = 0; c < K; ++c) hp[c] = h0[(bi * H + head0 + sub) * K + c];
                } else {
#pragma unroll
                    for (int c = 0; c < K; ++c) hp[c] = 0.f;
                }
                float a[K];
                lds_row<K>(st + q * S::AF + (sub * K + row) * K, a);
                float p[K], dar[K];
#pragma unroll
                for (int c = 0; c < K; ++c) {
                    p[c] = a[c] * lam;
                    dar[c] = lam * hp[c];
                }
                mu = group_reduce_scatter<K>(p, row);
                if (active) {
                    st_cs(dbp + t * hk, lam);
                    stg_row_cs<K>(dAp + t * hk * K, dar);
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
    if (dh0 != nullptr && active) dh0[(bi * H + head0 + sub) * K + row] = mu;
}

template <int K>
cudaError_t mas_fwd_t(const float *A, const float *b, const float *h0, float *h, int64_t B,
                      int64_t T, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    using S = MasShape<K>;
    using R = Ring<S::TS * (S::AF + S::VF), S::NS>;
    CUtensorMap tA, tB;
    cudaError_t e;
    if ((e = S::TA::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tB, b, B * T, H, S::TS)) != cudaSuccess) return e;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(R::warp_bytes);
    if ((e = ensure_smem_attr((const void *)mas_fwd_kernel<K>, smem)) != cudaSuccess) return e;
    mas_fwd_kernel<K><<<dim3(unsigned(blocks)), 32, smem, s>>>(tA, tB, h0, h, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

template <int K>
cudaError_t mas_bwd_t(const float *A, const float *h0, const float *h, const float *gh, float *dA,
                      float *db, float *dh0, int64_t B, int64_t T, int64_t H, const DevCtl &ctl,
                      cudaStream_t s) {
    using S = MasShape<K>;
    using R = Ring<S::TS * (S::AF + 2 * S::VF), S::NS>;
    CUtensorMap tA, tG, tH;
    cudaError_t e;
    if ((e = S::TA::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tG, gh, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tH, h, B * T, H, S::TS)) != cudaSuccess) return e;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(R::warp_bytes);
    if ((e = ensure_smem_attr((const void *)mas_bwd_kernel<K>, smem)) != cudaSuccess) return e;
    mas_bwd_kernel<K><<<dim3(unsigned(blocks)), 32, smem, s>>>(tA, tG, tH, h0, dA, db, dh0, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mas_fwd(int K, const float *A, const float *b, const float *h0, float *h,
                           int64_t B, int64_t T, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    switch (K) {
        case 1: return mas_fwd_t<1>(A, b, h0, h, B, T, H, ctl, s);
        case 2: return mas_fwd_t<2>(A, b, h0, h, B, T, H, ctl, s);
        case 4: return mas_fwd_t<4>(A, b, h0, h, B, T, H, ctl, s);
        case 8: return mas_fwd_t<8>(A, b, h0, h, B, T, H, ctl, s);
        case 16: return mas_fwd_t<16>(A, b, h0, h, B, T, H, ctl, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mas_bwd(int K, const float *A, const float *h0, const float *h,
                           const float *gh, float *dA, float *db, float *dh0, int64_t B,
                           int64_t T, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    switch (K) {
        case 1: return mas_bwd_t<1>(A, h0, h, gh, dA, db, dh0, B, T, H, ctl, s);
        case 2: return mas_bwd_t<2>(A, h0, h, gh, dA, db, dh0, B, T, H, ctl, s);
        case 4: return mas_bwd_t<4>(A, h0, h, gh, dA, db, dh0, B, T, H, ctl, s);
        case 8: return mas_bwd_t<8>(A, h0, h, gh, dA, db, dh0, B, T, H, ctl, s);
        case 16: return mas_bwd_t<16>(A, h0, h, gh, dA, db, dh0, B, T, H, ctl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mgs
