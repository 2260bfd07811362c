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
#include "mgs_chunk.cuh"

namespace mgs {
namespace {

#ifndef MGS_MAS_FWD_NS
#define MGS_MAS_FWD_NS 4
#endif
#ifndef MGS_MAS_FWD_TS8
#define MGS_MAS_FWD_TS8 8
#endif
// NSX: stages in flight when nonzero, else the tuned default.
template <int K, bool FWD = false, int NSX = 0>
struct MasShape {
    static constexpr int LPW = 32 / K;          // lanes (heads) per warp
    static constexpr int AF = LPW * K * K;      // floats of A per time step
    static constexpr int VF = LPW * K;          // floats of one per-lane vector per time step
    // time steps per stage: about 8-10 KB of A per stage
    static constexpr int TS = K >= 16 ? 4 : (K >= 8 ? (FWD ? MGS_MAS_FWD_TS8 : 8) : 16);
    static constexpr int NS = NSX ? NSX : (FWD ? MGS_MAS_FWD_NS : 4);  // stages in flight
    using TA = MatTile<K, false>;
    using TV = HeadTile<K, LPW>;
};

// Per-warp shared memory: NS stages of STAGEF floats (each starting on an
// ALIGN-byte boundary, the A box first), then NS barriers; ALIGN bytes of
// slack let the kernel align the dynamic base at run time.
template <int STAGEF, int NS, size_t ALIGN>
struct Ring {
    static constexpr size_t stage_bytes = size_t(STAGEF) * sizeof(float);   // transferred per stage
    static constexpr size_t stage_stride = align_up(stage_bytes, ALIGN);
    static constexpr size_t ring_bytes = NS * stage_stride;
    static constexpr size_t warp_bytes = align_up(ring_bytes + NS * sizeof(uint64_t), 128) + ALIGN;
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
template <int K, int NSX>
__global__ void __launch_bounds__(32)
    mas_fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const float *__restrict__ h0, float *__restrict__ h, int64_t B, int64_t T,
                   int64_t H, int64_t groups_per_b, DevCtl ctl) {
    using S = MasShape<K, true, NSX>;
    constexpr int A_STAGE = S::TS * S::AF, STAGEF = A_STAGE + S::TS * S::VF;
    using R = Ring<STAGEF, S::NS, S::TA::kAlign>;
    constexpr int SSTR = int(R::stage_stride / sizeof(float));
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    unsigned char *sbase = align_smem(smem_raw, S::TA::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + R::ring_bytes);

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
        float *st = ring + size_t(s) * SSTR;
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
        const float *st = ring + size_t(s) * SSTR;
        const float *sb = st + A_STAGE + sub * K + row;
#pragma unroll
        for (int u = 0; u < S::TS; ++u) {
            if (u < n) {
                float a[K];
                TileRef<K, false>{st, u, sub}.row(row, a);
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
template <int K, int NSX>
__global__ void __launch_bounds__(32)
    mas_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                   const __grid_constant__ CUtensorMap tmH, const float *__restrict__ h0,
                   float *__restrict__ dA, float *__restrict__ db, float *__restrict__ dh0, int64_t B,
                   int64_t T, int64_t H, int64_t groups_per_b, DevCtl ctl) {
    using S = MasShape<K, false, NSX>;
    constexpr int A_STAGE = S::TS * S::AF, V_STAGE = S::TS * S::VF;
    constexpr int STAGEF = A_STAGE + 2 * V_STAGE;  // A_t, g_t, h_{t-1}
    using R = Ring<STAGEF, S::NS, S::TA::kAlign>;
    constexpr int SSTR = int(R::stage_stride / sizeof(float));
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    unsigned char *sbase = align_smem(smem_raw, S::TA::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + R::ring_bytes);

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
        float *st = ring + size_t(s) * SSTR;
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
        const float *st = ring + size_t(s) * SSTR;
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
                TileRef<K, false>{st, q, sub}.row(row, a);
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

// ---------------------------------------------------------------- recompute-mode backward
// The backward without the saved forward output.  Phase A runs the forward
// over the warp's whole sequence (A and b streamed as in mas_fwd_kernel),
// keeping only h at the start of every chunk of RC = TS steps (one stage), in
// the workspace.  Phase B walks the chunks downwards, each chunk's stage of
// A, b and g resident in shared memory while the ring's other slots take the
// next chunks down: the chunk's h is recomputed forward from its checkpoint
// into shared memory, then the adjoint runs back over the chunk as in
// mas_bwd_kernel.  Per step A and b are read twice and g once, dA and db are
// written once; h is never stored.
template <int K>
struct MasRc {
    using S = MasShape<K>;
    static constexpr int RS = 1;           // stages per chunk
    static constexpr int RC = RS * S::TS;  // steps per chunk
    static constexpr int NS = 4;           // ring slots: chunk c in slot c % NS
    static constexpr int A_STAGE = S::TS * S::AF, V_STAGE = S::TS * S::VF;
    static constexpr int STAGEF = A_STAGE + 2 * V_STAGE;  // A_t, b_t, g_t
    using R = Ring<STAGEF, NS, S::TA::kAlign>;
    static constexpr size_t hs_off = align_up(R::ring_bytes + NS * sizeof(uint64_t), 128);
    // h of a chunk: row 0 the state before it, row u+1 the state after its step u
    static constexpr size_t warp_bytes = hs_off + size_t(RC + 1) * S::VF * sizeof(float) + S::TA::kAlign;
};

template <int K>
__global__ void __launch_bounds__(32)
    mas_bwd_rc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmG, const float *__restrict__ h0,
                      float *__restrict__ ck, float *__restrict__ dA, float *__restrict__ db,
                      float *__restrict__ dh0, int64_t B, int64_t T, int64_t H, int64_t groups_per_b,
                      DevCtl ctl) {
    using M = MasRc<K>;
    using S = typename M::S;
    using R = typename M::R;
    constexpr int NS = M::NS, TS = S::TS, RC = M::RC, VF = S::VF;
    constexpr int SSTR = int(R::stage_stride / sizeof(float));
    extern __shared__ __align__(128) unsigned char smem_raw[];

    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    unsigned char *sbase = align_smem(smem_raw, S::TA::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + R::ring_bytes);
    float *hs = reinterpret_cast<float *>(sbase + M::hs_off);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * S::LPW;
    const int nl = int(min64(S::LPW, H - head0));
    const int sub = lane / K, row = lane % K, gbase = lane & ~(K - 1);
    const bool active = sub < nl;
    const int row0 = int(bi * T);
    const int64_t nblk = (T + TS - 1) / TS;  // phase A stages
    const int64_t nck = (T + RC - 1) / RC;   // chunks
    float *ckp = ck + g * nck * VF + lane;   // the group's checkpoints; lane = sub * K + row

    WarpRing<NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmG);
    }

    // ---- phase A: the forward, checkpoints only
    auto issue_f = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * SSTR;
        mbar_arrive_expect_tx(&bars[s], uint32_t((M::A_STAGE + M::V_STAGE) * sizeof(float)));
        S::TA::load(st, &tmA, head0, row0 + int(j * TS), &bars[s], pol);
        S::TV::load(st + M::A_STAGE, &tmB, head0, row0 + int(j * TS), &bars[s], pol);
    };
    {
        const int npro = int(min64(NS, nblk));
        if (lane == 0)
            for (int s = 0; s < npro; ++s) issue_f(s, s);
        for (int s = 0; s < npro; ++s) rg.armed(s);
    }
    float hprev = (h0 != nullptr && active) ? h0[(bi * H + head0 + sub) * K + row] : 0.f;
    ckp[0] = hprev;
    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(TS, T - j * TS));
        const float *st = ring + size_t(s) * SSTR;
        const float *sb = st + M::A_STAGE + lane;
#pragma unroll
        for (int u = 0; u < TS; ++u) {
            if (u < n) {
                float a[K];
                TileRef<K, false>{st, u, sub}.row(row, a);
                float acc0 = sb[u * VF];
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
            }
        }
        // chunks end on stage boundaries: h after this stage starts the next chunk
        if ((j + 1) % M::RS == 0 && (j + 1) * TS < T) ckp[((j + 1) / M::RS) * VF] = hprev;
        __syncwarp();
        if (j + NS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue_f(s, j + NS);
            }
            rg.armed(s);
        }
    }

    // ---- phase B: chunks downwards; chunk c in slot c % NS
    auto issue_b = [&](int s, int64_t c) {  // lane 0 only
        float *st = ring + size_t(s) * SSTR;
        const int rr = row0 + int(c * RC);
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        S::TA::load(st, &tmA, head0, rr, &bars[s], pol);
        S::TV::load(st + M::A_STAGE, &tmB, head0, rr, &bars[s], pol);
        S::TV::load(st + M::A_STAGE + M::V_STAGE, &tmG, head0, rr, &bars[s], pol);
    };
    __syncwarp();
    for (int64_t c = nck - 1; c >= 0 && c >= nck - NS; --c) {
        if (lane == 0) {
            fence_proxy_async_smem();
            issue_b(int(c % NS), c);
        }
        rg.armed(int(c % NS));
    }
    float mu = 0.f;  // (A_{t+1}^T lambda_{t+1})[row], zero past the end
    const int64_t hk = H * K;
    float *dbp = db + (bi * T * H + head0 + sub) * K + row;          // + t*H*K
    float *dAp = dA + (bi * T * H + head0 + sub) * K * K + row * K;  // + t*H*K*K
    float hnext = ckp[(nck - 1) * VF];  // each chunk's checkpoint is read one chunk ahead
    for (int64_t c = nck - 1; c >= 0; --c) {
        const int s = int(c % NS);
        float hv = hnext;
        if (c >= 1) hnext = ckp[(c - 1) * VF];
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(RC, T - c * RC));
        const float *st = ring + size_t(s) * SSTR;
        // the chunk's h, forward from its checkpoint
        hs[lane] = hv;
        const float *sb = st + M::A_STAGE + lane;
#pragma unroll
        for (int u = 0; u < TS; ++u) {
            if (u < n) {
                float a[K];
                TileRef<K, false>{st, u, sub}.row(row, a);
                float acc0 = sb[u * VF];
                float acc1 = 0.f;
#pragma unroll
                for (int cc = 0; cc < K; ++cc) {
                    const float x = __shfl_sync(0xffffffffu, hv, gbase + cc);
                    if (cc & 1)
                        acc1 = fmaf(a[cc], x, acc1);
                    else
                        acc0 = fmaf(a[cc], x, acc0);
                }
                hv = acc0 + acc1;
                hs[(u + 1) * VF + lane] = hv;
            }
        }
        __syncwarp();
        // the adjoint back over the chunk
#pragma unroll
        for (int u = TS - 1; u >= 0; --u) {
            if (u < n) {
                const int64_t t = c * RC + u;
                const float lam = st[M::A_STAGE + M::V_STAGE + u * VF + lane] + mu;
                float hp[K];
                lds_row<K>(hs + u * VF + sub * K, hp);  // h_{t-1}
                float a[K];
                TileRef<K, false>{st, u, sub}.row(row, a);
                float p[K], dar[K];
#pragma unroll
                for (int cc = 0; cc < K; ++cc) {
                    p[cc] = a[cc] * lam;
                    dar[cc] = lam * hp[cc];
                }
                mu = group_reduce_scatter<K>(p, row);
                if (active) {
                    st_cs(dbp + t * hk, lam);
                    stg_row_cs<K>(dAp + t * hk * K, dar);
                }
            }
        }
        __syncwarp();  // every read of the chunk's slot and of hs is done
        if (c >= NS) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue_b(s, c - NS);
            }
            rg.armed(s);
        }
    }
    if (dh0 != nullptr && active) dh0[(bi * H + head0 + sub) * K + row] = mu;
}

template <int K>
size_t mas_rc_workspace_t(int64_t B, int64_t T, int64_t H) {
    using M = MasRc<K>;
    const int64_t gpb = (H + M::S::LPW - 1) / M::S::LPW;
    return size_t(B) * size_t(gpb) * size_t((T + M::RC - 1) / M::RC) * M::S::VF * sizeof(float);
}

template <int K>
cudaError_t mas_bwd_rc_t(const float *A, const float *b, const float *h0, const float *gh, float *dA, float *db,
                         float *dh0, int64_t B, int64_t T, int64_t H, void *ws, const DevCtl &ctl,
                         cudaStream_t s) {
    using M = MasRc<K>;
    using S = typename M::S;
    CUtensorMap tA, tB, tG;
    cudaError_t e;
    if ((e = S::TA::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tB, b, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tG, gh, B * T, H, S::TS)) != cudaSuccess) return e;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(M::warp_bytes);
    if ((e = ensure_smem_attr((const void *)mas_bwd_rc_kernel<K>, smem)) != cudaSuccess) return e;
    mas_bwd_rc_kernel<K><<<dim3(unsigned(blocks)), 32, smem, s>>>(tA, tB, tG, h0, static_cast<float *>(ws), dA, db,
                                                                  dh0, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

template <int K, int NSX>
cudaError_t mas_fwd_launch(const float *A, const float *b, const float *h0, float *h, int64_t B, int64_t T,
                           int64_t H, const DevCtl &ctl, cudaStream_t s) {
    using S = MasShape<K, true, NSX>;
    using R = Ring<S::TS * (S::AF + S::VF), S::NS, S::TA::kAlign>;
    CUtensorMap tA, tB;
    cudaError_t e;
    if ((e = S::TA::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tB, b, B * T, H, S::TS)) != cudaSuccess) return e;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(R::warp_bytes);
    const auto kern = mas_fwd_kernel<K, NSX>;
    if ((e = ensure_smem_attr((const void *)kern, smem)) != cudaSuccess) return e;
    kern<<<dim3(unsigned(blocks)), 32, smem, s>>>(tA, tB, h0, h, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

template <int K>
cudaError_t mas_fwd_t(const float *A, const float *b, const float *h0, float *h, int64_t B,
                      int64_t T, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    return mas_fwd_launch<K, 0>(A, b, h0, h, B, T, H, ctl, s);
}

template <int K, int NSX>
cudaError_t mas_bwd_launch(const float *A, const float *h0, const float *h, const float *gh, float *dA, float *db,
                           float *dh0, int64_t B, int64_t T, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    using S = MasShape<K, false, NSX>;
    using R = Ring<S::TS * (S::AF + 2 * S::VF), S::NS, S::TA::kAlign>;
    CUtensorMap tA, tG, tH;
    cudaError_t e;
    if ((e = S::TA::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tG, gh, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tH, h, B * T, H, S::TS)) != cudaSuccess) return e;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(R::warp_bytes);
    const auto kern = mas_bwd_kernel<K, NSX>;
    if ((e = ensure_smem_attr((const void *)kern, smem)) != cudaSuccess) return e;
    kern<<<dim3(unsigned(blocks)), 32, smem, s>>>(tA, tG, tH, h0, dA, db, dh0, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

template <int K>
cudaError_t mas_bwd_t(const float *A, const float *h0, const float *h, const float *gh, float *dA,
                      float *db, float *dh0, int64_t B, int64_t T, int64_t H, const DevCtl &ctl,
                      cudaStream_t s) {
    return mas_bwd_launch<K, 0>(A, h0, h, gh, dA, db, dh0, B, T, H, ctl, s);
}

// ================================================================ time-chunked path
// Few lanes and a long sequence: T is split into C chunks, one warp per
// (lane group, chunk) item, as for matrix_scan (the three launches of
// mgs_chunk.cuh).  The forward aggregate of a chunk is the affine map
// h_end = M h_in + c with M = A_e ... A_s (built one column per thread:
// M[:, j] <- A_t M[:, j], broadcast reads of A_t, no shuffles) and c the
// chunk's own recurrence from h = 0.  The backward aggregate is
// mu_out = M mu_in + C with M = A_s^T ... A_e^T.

template <int K>
struct MasChunkShape {
    static constexpr int LPW = 32 / K;
    static constexpr int AF = LPW * K * K, VF = LPW * K;
    static constexpr int TS = K >= 16 ? 4 : (K >= 8 ? 8 : 16);
    static constexpr int NS = 4;
    using TA = MatTile<K>;
    using TV = HeadTile<K, LPW>;
};

template <int STAGEF, int NS, size_t ALIGN>
struct ChunkRing {
    static constexpr size_t stage_bytes = size_t(STAGEF) * sizeof(float);  // transferred per full stage
    static constexpr size_t stage_stride = align_up(stage_bytes, ALIGN);
    static constexpr size_t ring_bytes = NS * stage_stride;
    static constexpr size_t bar_offset = ring_bytes;
    static constexpr size_t warp_bytes = align_up(bar_offset + NS * sizeof(uint64_t), 128) + ALIGN;
};


// The chunked path is the reduce-then-scan of mgs_chunk.cuh:
//   forward:  aggregate h_end = M h_in + c of chunks 0 .. C-2 (M = A_e ... A_s
//             built one column per thread, c the chunk's recurrence from zero),
//             carries E_0 = h0, E_{p+1} = M_p E_p + c_p, then every chunk's
//             recurrence from its carry;
//   backward: aggregate mu_out = M mu_in + C of chunks 1 .. C-1 (M = A_s^T ...
//             A_e^T), carries mu_in(C-1) = 0, mu_in(p-1) = M_p mu_in(p) + C_p,
//             then every chunk's adjoint from its carry.

// Launch 1, forward.
template <int K>
__global__ void __launch_bounds__(32)
    mas_fwd_agg_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       float *__restrict__ Ms, float *__restrict__ Cs, int64_t T, int64_t gpb, int64_t C, int64_t Lc,
                       DevCtl ctl) {
    using S = MasChunkShape<K>;
    constexpr int A_STAGE = S::TS * S::AF, STAGEF = A_STAGE + S::TS * S::VF;
    using R = ChunkRing<STAGEF, S::NS, S::TA::kAlign>;
    constexpr int SSTR = int(R::stage_stride / sizeof(float));
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TA::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + R::bar_offset);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C - 1, 0, gpb, S::LPW);
    const int sub = lane / K, r = lane % K, gbase = lane & ~(K - 1);
    const QuadOffsets<K> qo(sub, r);  // this thread's offsets in a staged box
    const int64_t tb = it.c * Lc, len = min64(Lc, T - tb);
    const int64_t nb = (len + S::TS - 1) / S::TS;

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();  // launch 3 reads the chunk again
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * SSTR;
        const int row = int(it.bi * T + tb + j * S::TS);
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        S::TA::load(st, &tmA, it.head0, row, &bars[s], pol);
        S::TV::load(st + A_STAGE, &tmB, it.head0, row, &bars[s], pol);
    };
    const int npro = int(min64(S::NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float cv = 0.f;  // row r of the chunk offset c
    float mcol[K];   // column r of the chunk matrix M
#pragma unroll
    for (int i = 0; i < K; ++i) mcol[i] = (i == r) ? 1.f : 0.f;
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(S::TS, len - j * S::TS));
        const float *st = ring + size_t(s) * SSTR;
        // one step: c <- A c + b (row r, from the group's shuffled c) and the
        // column of M <- A M from the step's block in registers
        auto step = [&](const float (&ablk)[K][K], int u) {
            float a[K];
            TileRef<K>{st, u, sub}.row(r, a);
            float acc0 = st[A_STAGE + u * S::VF + sub * K + r], acc1 = 0.f;
#pragma unroll
            for (int jj = 0; jj < K; ++jj) {
                const float x = __shfl_sync(0xffffffffu, cv, gbase + jj);
                if (jj & 1) acc1 = fmaf(a[jj], x, acc1);
                else acc0 = fmaf(a[jj], x, acc0);
            }
            cv = acc0 + acc1;
            float nm[K];
            reg_matvec(ablk, mcol, nm);
#pragma unroll
            for (int i = 0; i < K; ++i) mcol[i] = nm[i];
        };
        if constexpr (K >= 4 && K <= 8) {
            // step u + 1's block is loaded while step u computes (rows past n
            // are staged box rows too, loaded and not used)
            float ab[K][K];
            tile_load(TileRefQ<K>{st, qo}, ab);
#pragma unroll
            for (int u = 0; u < S::TS; ++u) {
                float an[K][K];
                if (u + 1 < S::TS) tile_load(TileRefQ<K>{st + (u + 1) * S::AF, qo}, an);
                if (u < n) step(ab, u);
                if (u + 1 < S::TS) {
#pragma unroll
                    for (int i = 0; i < K; ++i)
#pragma unroll
                        for (int c = 0; c < K; ++c) ab[i][c] = an[i][c];
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < S::TS; ++u) {
                if (u < n) {
                    const TileRef<K> Ablk{st, u, sub};
                    float a[K];
                    Ablk.row(r, a);
                    float acc0 = st[A_STAGE + u * S::VF + sub * K + r], acc1 = 0.f;
#pragma unroll
                    for (int jj = 0; jj < K; ++jj) {
                        const float x = __shfl_sync(0xffffffffu, cv, gbase + jj);
                        if (jj & 1) acc1 = fmaf(a[jj], x, acc1);
                        else acc0 = fmaf(a[jj], x, acc0);
                    }
                    cv = acc0 + acc1;
                    float nm[K];
                    tile_matvec(Ablk, mcol, nm);
#pragma unroll
                    for (int i = 0; i < K; ++i) mcol[i] = nm[i];
                }
            }
        }
        __syncwarp();
        if (j + S::NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + S::NS);
            }
            rg.armed(s);
        }
    }
    const int64_t item = it.g * C + it.c;
    st_ws_col<K>(Ms + item * S::AF + sub * K * K, r, mcol);
    __stcg(Cs + item * S::VF + sub * K + r, cv);
}

// Launch 3, forward: h_t from the chunk's carry (all chunks).
template <int K>
__global__ void __launch_bounds__(32)
    mas_fwd_out_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       float *__restrict__ h, const float *__restrict__ Es, int64_t T, int64_t H, int64_t gpb,
                       int64_t C, int64_t Lc, DevCtl ctl) {
    using S = MasChunkShape<K>;
    constexpr int A_STAGE = S::TS * S::AF, STAGEF = A_STAGE + S::TS * S::VF;
    using R = ChunkRing<STAGEF, S::NS, S::TA::kAlign>;
    constexpr int SSTR = int(R::stage_stride / sizeof(float));
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TA::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + R::bar_offset);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C, 0, gpb, S::LPW);
    const int sub = lane / K, r = lane % K, gbase = lane & ~(K - 1);
    const bool active = it.head0 + sub < H;
    const int64_t tb = it.c * Lc, len = min64(Lc, T - tb);
    const int64_t nb = (len + S::TS - 1) / S::TS;

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * SSTR;
        const int row = int(it.bi * T + tb + j * S::TS);
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        S::TA::load(st, &tmA, it.head0, row, &bars[s], pol);
        S::TV::load(st + A_STAGE, &tmB, it.head0, row, &bars[s], pol);
    };
    const int npro = int(min64(S::NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    pdl_wait();  // the carries of launch 2
    float hprev = __ldcg(Es + (it.g * C + it.c) * S::VF + sub * K + r);
    const int64_t hstride = H * K;
    float *hout = h + (it.bi * T * H + it.head0 + sub) * K + r + tb * hstride;
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(S::TS, len - j * S::TS));
        const float *st = ring + size_t(s) * SSTR;
#pragma unroll
        for (int u = 0; u < S::TS; ++u) {
            if (u < n) {
                float a[K];
                TileRef<K>{st, u, sub}.row(r, a);
                float acc0 = st[A_STAGE + u * S::VF + sub * K + r], acc1 = 0.f;
#pragma unroll
                for (int jj = 0; jj < K; ++jj) {
                    const float x = __shfl_sync(0xffffffffu, hprev, gbase + jj);
                    if (jj & 1) acc1 = fmaf(a[jj], x, acc1);
                    else acc0 = fmaf(a[jj], x, acc0);
                }
                hprev = acc0 + acc1;
                if (active) st_cs(hout, hprev);
                hout += hstride;
            }
        }
        __syncwarp();
        if (j + S::NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + S::NS);
            }
            rg.armed(s);
        }
    }
}

// Launch 1, backward: (M, C) of chunks 1 .. C-1, t walking down the chunk.
template <int K>
__global__ void __launch_bounds__(32)
    mas_bwd_agg_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                       float *__restrict__ Ms, float *__restrict__ Cs, int64_t T, int64_t gpb, int64_t C, int64_t Lc,
                       DevCtl ctl) {
    using S = MasChunkShape<K>;
    constexpr int A_STAGE = S::TS * S::AF, V_STAGE = S::TS * S::VF;
    constexpr int STAGEF = A_STAGE + V_STAGE;
    using R = ChunkRing<STAGEF, S::NS, S::TA::kAlign>;
    constexpr int SSTR = int(R::stage_stride / sizeof(float));
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TA::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + R::bar_offset);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C - 1, 1, gpb, S::LPW);
    const int sub = lane / K, r = lane % K;
    const QuadOffsets<K> qo(sub, r);  // this thread's offsets in a staged box
    const int64_t tb = it.c * Lc, te = min64(T, tb + Lc), len = te - tb;
    const int64_t nb = (len + S::TS - 1) / S::TS;

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmG);
    }
    // block j covers t = te-1-j*TS down to max(tb, te-(j+1)*TS); boxes start at
    // row te-(j+1)*TS, step u at box row TS-1-u
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        const int r0 = int(it.bi * T + te - (j + 1) * S::TS);
        float *st = ring + size_t(s) * SSTR;
        mbar_arrive_expect_tx(&bars[s], uint32_t(STAGEF * 4));
        S::TA::load(st, &tmA, it.head0, r0, &bars[s], pol);
        S::TV::load(st + A_STAGE, &tmG, it.head0, r0, &bars[s], pol);
    };
    const int npro = int(min64(S::NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mu = 0.f;  // row r of the chunk offset C
    float mcol[K];   // column r of M = A_s^T ... A_e^T
#pragma unroll
    for (int i = 0; i < K; ++i) mcol[i] = (i == r) ? 1.f : 0.f;
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tt = te - 1 - j * S::TS;
        const int n = int(min64(S::TS, tt - tb + 1));
        const float *st = ring + size_t(s) * SSTR;
        // one step (box row q): mu <- A^T (g + mu) by the group's reduce-scatter,
        // and the column of M <- A^T M from the step's block in registers
        auto bstep = [&](const float (&ablk)[K][K], int q) {
            const float lam = st[A_STAGE + q * S::VF + sub * K + r] + mu;
            float a[K], p[K], nm[K];
            TileRef<K>{st, q, sub}.row(r, a);
#pragma unroll
            for (int x = 0; x < K; ++x) p[x] = a[x] * lam;
            mu = group_reduce_scatter<K>(p, r);
            reg_matvec_t(ablk, mcol, nm);
#pragma unroll
            for (int i = 0; i < K; ++i) mcol[i] = nm[i];
        };
        if constexpr (K >= 4 && K <= 8) {
            float ab[K][K];
            tile_load(TileRefQ<K>{st + (S::TS - 1) * S::AF, qo}, ab);
#pragma unroll
            for (int u = 0; u < S::TS; ++u) {
                float an[K][K];
                if (u + 1 < S::TS) tile_load(TileRefQ<K>{st + (S::TS - 2 - u) * S::AF, qo}, an);
                if (u < n) bstep(ab, S::TS - 1 - u);
                if (u + 1 < S::TS) {
#pragma unroll
                    for (int i = 0; i < K; ++i)
#pragma unroll
                        for (int c = 0; c < K; ++c) ab[i][c] = an[i][c];
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < S::TS; ++u) {
                if (u < n) {
                    const int q = S::TS - 1 - u;
                    const TileRef<K> Ablk{st, q, sub};
                    const float lam = st[A_STAGE + q * S::VF + sub * K + r] + mu;
                    float a[K], p[K], nm[K];
                    Ablk.row(r, a);
#pragma unroll
                    for (int x = 0; x < K; ++x) p[x] = a[x] * lam;
                    mu = group_reduce_scatter<K>(p, r);
                    tile_matvec_t(Ablk, mcol, nm);
#pragma unroll
                    for (int i = 0; i < K; ++i) mcol[i] = nm[i];
                }
            }
        }
        __syncwarp();
        if (j + S::NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + S::NS);
            }
            rg.armed(s);
        }
    }
    const int64_t item = it.g * C + it.c;
    st_ws_col<K>(Ms + item * S::AF + sub * K * K, r, mcol);
    __stcg(Cs + item * S::VF + sub * K + r, mu);
}

// Launch 3, backward: db, dA (and dh0 from chunk 0) from the chunk's carry.
template <int K>
__global__ void __launch_bounds__(32)
    mas_bwd_out_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                       const __grid_constant__ CUtensorMap tmH, const float *__restrict__ h0, float *__restrict__ dA,
                       float *__restrict__ db, float *__restrict__ dh0, const float *__restrict__ Es, int64_t T,
                       int64_t H, int64_t gpb, int64_t C, int64_t Lc, DevCtl ctl) {
    using S = MasChunkShape<K>;
    constexpr int A_STAGE = S::TS * S::AF, V_STAGE = S::TS * S::VF;
    constexpr int STAGEF = A_STAGE + 2 * V_STAGE;
    using R = ChunkRing<STAGEF, S::NS, S::TA::kAlign>;
    constexpr int SSTR = int(R::stage_stride / sizeof(float));
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sbase = align_smem(smem_raw, S::TA::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + R::bar_offset);

    const int lane = threadIdx.x;
    const ChunkItem it(blockIdx.x, C, 0, gpb, S::LPW);
    const int sub = lane / K, r = lane % K;
    const bool active = it.head0 + sub < H;
    const int64_t bi = it.bi;
    const int head0 = it.head0;
    const int64_t tb = it.c * Lc, te = min64(T, tb + Lc), len = te - tb;
    const int64_t nb = (len + S::TS - 1) / S::TS;

    WarpRing<S::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmH);
    }
    // as in launch 1; the h box starts one row earlier and holds h_{t-1}
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        const int r0 = int(bi * T + te - (j + 1) * S::TS);
        float *st = ring + size_t(s) * SSTR;
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        S::TA::load(st, &tmA, head0, r0, &bars[s], pol);
        S::TV::load(st + A_STAGE, &tmG, head0, r0, &bars[s], pol);
        S::TV::load(st + A_STAGE + V_STAGE, &tmH, head0, r0 - 1, &bars[s], pol);
    };
    const int npro = int(min64(S::NS, nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    pdl_wait();  // the carries of launch 2
    float mu = __ldcg(Es + (it.g * C + it.c) * S::VF + sub * K + r);  // (A_{t+1}^T lambda_{t+1})[r] past the chunk
    const int64_t hk = H * K;
    float *dbp = db + (bi * T * H + head0 + sub) * K + r;
    float *dAp = dA + (bi * T * H + head0 + sub) * K * K + r * K;
    for (int64_t j = 0; j < nb; ++j) {
        const int s = int(j % S::NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tt = te - 1 - j * S::TS;
        const int n = int(min64(S::TS, tt - tb + 1));
        const float *st = ring + size_t(s) * SSTR;
#pragma unroll
        for (int u = 0; u < S::TS; ++u) {
            if (u < n) {
                const int64_t t = tt - u;
                const int q = S::TS - 1 - u;
                const TileRef<K> Ablk{st, q, sub};
                const float lam = st[A_STAGE + q * S::VF + sub * K + r] + mu;
                float a[K], p[K], hp[K], dar[K];
                Ablk.row(r, a);
#pragma unroll
                for (int x = 0; x < K; ++x) p[x] = a[x] * lam;
                mu = group_reduce_scatter<K>(p, r);
                if (t >= 1) {
                    lds_row<K>(st + A_STAGE + V_STAGE + q * S::VF + sub * K, hp);
                } else if (h0 != nullptr && active) {
#pragma unroll
                    for (int x = 0; x < K; ++x) hp[x] = h0[(bi * H + head0 + sub) * K + x];
                } else {
#pragma unroll
                    for (int x = 0; x < K; ++x) hp[x] = 0.f;
                }
#pragma unroll
                for (int x = 0; x < K; ++x) dar[x] = lam * hp[x];
                if (active) {
                    st_cs(dbp + t * hk, lam);
                    stg_row_cs<K>(dAp + t * hk * K, dar);
                }
            }
        }
        __syncwarp();
        if (j + S::NS < nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + S::NS);
            }
            rg.armed(s);
        }
    }
    if (it.c == 0 && dh0 != nullptr && active) dh0[(bi * H + head0 + sub) * K + r] = mu;
}

template <int K>
cudaError_t mas_fwd_chunk_t(const float *A, const float *b, const float *h0, float *h, int64_t B, int64_t T,
                            int64_t H, const ChunkPlan &pl, unsigned char *ws, const DevCtl &ctl, cudaStream_t s) {
    using S = MasChunkShape<K>;
    using R = ChunkRing<S::TS * (S::AF + S::VF), S::NS, S::TA::kAlign>;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const ScanWs w(ws, pl, S::AF, S::VF);
    if (pl.G * pl.C > 0x7fffffff) return cudaErrorInvalidConfiguration;
    CUtensorMap tA, tB;
    cudaError_t e;
    if ((e = S::TA::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tB, b, B * T, H, S::TS)) != cudaSuccess) return e;
    const int smem = int(R::warp_bytes);
    if ((e = ensure_smem_attr((const void *)mas_fwd_agg_kernel<K>, smem)) != cudaSuccess) return e;
    if ((e = ensure_smem_attr((const void *)mas_fwd_out_kernel<K>, smem)) != cudaSuccess) return e;
    mas_fwd_agg_kernel<K><<<dim3(unsigned(pl.G * (pl.C - 1))), 32, smem, s>>>(tA, tB, w.M, w.Cv, T, gpb, pl.C, pl.L,
                                                                              ctl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_chain<K, false, true, +1>(w.M, w.Cv, w.E, h0, pl.G, pl.C, gpb, H, ctl, s)) != cudaSuccess) return e;
    return launch_pdl(mas_fwd_out_kernel<K>, dim3(unsigned(pl.G * pl.C)), smem, s, tA, tB, h, w.E, T, H, gpb, pl.C,
                      pl.L, ctl);
}

template <int K>
cudaError_t mas_bwd_chunk_t(const float *A, const float *h0, const float *h, const float *gh, float *dA,
                            float *db, float *dh0, int64_t B, int64_t T, int64_t H, const ChunkPlan &pl,
                            unsigned char *ws, const DevCtl &ctl, cudaStream_t s) {
    using S = MasChunkShape<K>;
    using RA = ChunkRing<S::TS * (S::AF + S::VF), S::NS, S::TA::kAlign>;
    using RO = ChunkRing<S::TS * (S::AF + 2 * S::VF), S::NS, S::TA::kAlign>;
    const int64_t gpb = (H + S::LPW - 1) / S::LPW;
    const ScanWs w(ws, pl, S::AF, S::VF);
    if (pl.G * pl.C > 0x7fffffff) return cudaErrorInvalidConfiguration;
    CUtensorMap tA, tG, tH;
    cudaError_t e;
    if ((e = S::TA::make(&tA, A, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tG, gh, B * T, H, S::TS)) != cudaSuccess) return e;
    if ((e = S::TV::make(&tH, h, B * T, H, S::TS)) != cudaSuccess) return e;
    const int sa = int(RA::warp_bytes), so = int(RO::warp_bytes);
    if ((e = ensure_smem_attr((const void *)mas_bwd_agg_kernel<K>, sa)) != cudaSuccess) return e;
    if ((e = ensure_smem_attr((const void *)mas_bwd_out_kernel<K>, so)) != cudaSuccess) return e;
    mas_bwd_agg_kernel<K><<<dim3(unsigned(pl.G * (pl.C - 1))), 32, sa, s>>>(tA, tG, w.M, w.Cv, T, gpb, pl.C, pl.L,
                                                                            ctl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_chain<K, false, true, -1>(w.M, w.Cv, w.E, nullptr, pl.G, pl.C, gpb, H, ctl, s)) != cudaSuccess)
        return e;
    return launch_pdl(mas_bwd_out_kernel<K>, dim3(unsigned(pl.G * pl.C)), so, s, tA, tG, tH, h0, dA, db, dh0, w.E, T,
                      H, gpb, pl.C, pl.L, ctl);
}

}  // namespace

size_t mas_workspace_bytes(int64_t B, int64_t T, int64_t H, int K) {
    const ChunkPlan p = plan_chunks(B, T, H, K);
    if (p.C <= 1) return 0;
    return ScanWs::bytes(p, 32 * K, 32, 32);  // per lane group: M (32/k blocks of k x k), c and E (32 floats)
}

#define MAS_DISPATCH(K_, CALL)                 \
    switch (K_) {                              \
        case 1: return CALL(1);                \
        case 2: return CALL(2);                \
        case 4: return CALL(4);                \
        case 8: return CALL(8);                \
        case 16: return CALL(16);              \
        default: return cudaErrorInvalidValue; \
    }

cudaError_t launch_mas_fwd(int K, const float *A, const float *b, const float *h0, float *h,
                           int64_t B, int64_t T, int64_t H, void *ws, size_t, const DevCtl &ctl,
                           cudaStream_t s) {
    const ChunkPlan pl = plan_chunks(B, T, H, K);
    if (pl.C > 1) {
        unsigned char *w = static_cast<unsigned char *>(ws);
#define CALL_FC(k) mas_fwd_chunk_t<k>(A, b, h0, h, B, T, H, pl, w, ctl, s)
        MAS_DISPATCH(K, CALL_FC)
#undef CALL_FC
    }
#define CALL_F(k) mas_fwd_t<k>(A, b, h0, h, B, T, H, ctl, s)
    MAS_DISPATCH(K, CALL_F)
#undef CALL_F
}

cudaError_t launch_mas_bwd(int K, const float *A, const float *h0, const float *h,
                           const float *gh, float *dA, float *db, float *dh0, int64_t B,
                           int64_t T, int64_t H, void *ws, size_t, const DevCtl &ctl, cudaStream_t s) {
    const ChunkPlan pl = plan_chunks(B, T, H, K);
    if (pl.C > 1) {
        unsigned char *w = static_cast<unsigned char *>(ws);
#define CALL_BC(k) mas_bwd_chunk_t<k>(A, h0, h, gh, dA, db, dh0, B, T, H, pl, w, ctl, s)
        MAS_DISPATCH(K, CALL_BC)
#undef CALL_BC
    }
#define CALL_B(k) mas_bwd_t<k>(A, h0, h, gh, dA, db, dh0, B, T, H, ctl, s)
    MAS_DISPATCH(K, CALL_B)
#undef CALL_B
}

// Few lane groups and a long sequence (where the saved-h path splits T into
// chunks): the recompute mode runs the time-chunked forward into the
// workspace and the time-chunked saved-h backward on it; the workspace holds
// h (256-byte aligned) followed by the chunked kernels' own workspace.  h is
// still not kept between the forward and the backward call.
static size_t rc_h_bytes(int64_t B, int64_t T, int64_t H, int K) {
    return align_up(size_t(B) * size_t(T) * size_t(H) * size_t(K) * sizeof(float), 256);
}

size_t mas_rc_workspace_bytes(int64_t B, int64_t T, int64_t H, int K) {
    if (plan_chunks(B, T, H, K).C > 1) return rc_h_bytes(B, T, H, K) + mas_workspace_bytes(B, T, H, K);
    switch (K) {
        case 1: return mas_rc_workspace_t<1>(B, T, H);
        case 2: return mas_rc_workspace_t<2>(B, T, H);
        case 4: return mas_rc_workspace_t<4>(B, T, H);
        case 8: return mas_rc_workspace_t<8>(B, T, H);
        case 16: return mas_rc_workspace_t<16>(B, T, H);
        default: return 0;
    }
}

cudaError_t launch_mas_bwd_recompute(int K, const float *A, const float *b, const float *h0, const float *gh,
                                     float *dA, float *db, float *dh0, int64_t B, int64_t T, int64_t H, void *ws,
                                     const DevCtl &ctl, cudaStream_t s) {
    if (plan_chunks(B, T, H, K).C > 1) {
        float *h = static_cast<float *>(ws);
        const size_t hb = rc_h_bytes(B, T, H, K), cb = mas_workspace_bytes(B, T, H, K);
        void *cw = static_cast<unsigned char *>(ws) + hb;
        cudaError_t e = launch_mas_fwd(K, A, b, h0, h, B, T, H, cw, cb, ctl, s);
        if (e != cudaSuccess) return e;
        return launch_mas_bwd(K, A, h0, h, gh, dA, db, dh0, B, T, H, cw, cb, ctl, s);
    }
#define CALL_RC(k) mas_bwd_rc_t<k>(A, b, h0, gh, dA, db, dh0, B, T, H, ws, ctl, s)
    MAS_DISPATCH(K, CALL_RC)
#undef CALL_RC
}

}  // namespace mgs
