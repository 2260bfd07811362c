// parallel_scan_log forward and backward ("mingru-scans" home page, scan-op
// table, parallel_scan_log row; Heinsen 2023, arXiv:2311.06281, cited in the
// home page's lineage paragraph).
//
// Forward, per (batch, channel) lane:
//     log h_t = logaddexp(log_coeffs_t + log h_{t-1}, log_values_t),
//     h_t = exp(log h_t),
// which equals Heinsen's exp(a*_t + logcumsumexp(log_values - a*)) without
// ever forming the cumulative sum a*_t (whose fp32 cancellation at T = 4096
// would cost about three decimal digits).  logaddexp is max-shifted:
// max(x, y) + log(1 + exp(-|x - y|)).  The state is carried in base 2
// (L = log2 h), so each step is two multiplies by log2(e), the hardware
// ex2/lg2 pair and a final ex2 for h_t.
//
// Error budget of the base-2 form: converting an input x to base 2 rounds
// x*log2(e) (relative error 2^-24), i.e. an absolute error of about
// 6e-8*|x| in the exponent; ex2 and lg2 add a few 1e-7.  For |log_values|,
// |log_coeffs|, |log h| up to 50 every step's relative error in h stays
// below about 4e-6, and the recurrence contracts it (the weight of the
// carried term is below 1).
// Backward walks t downwards in linear space (a_t = exp(log_coeffs_t) in (0, 1]
// for gates), lambda_t = g_t + a_{t+1} lambda_{t+1}.
//
// A warp owns 128 adjacent channels of one batch row (4 per thread, float4);
// each stage of TS time steps arrives by one tiled TMA load per input tensor.
#include <math_constants.h>

#include "mgs_tiles.cuh"

namespace mgs {
namespace {

constexpr int kChan = 128;  // channels per warp
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int NT, int TS, int NS>  // NT row tensors per stage
struct PslRing {
    static constexpr int BOXF = TS * kChan;  // floats per tensor box
    static constexpr int STAGEF = NT * BOXF;
    static constexpr size_t stage_bytes = size_t(STAGEF) * sizeof(float);
    static constexpr size_t ring_bytes = NS * stage_bytes;
    static constexpr size_t warp_bytes = align_up(ring_bytes + NS * sizeof(uint64_t), 128);
};

// Stage depth, measured on the minGRU shape (B=64 T=4096 D=1024): forward
// 12 steps x 4 stages (2 tensors x 512 B x 12 = 12 KB per stage) beat 8 x 4
// by 11 %; backward 8 steps x 2 stages (4 tensors: 16 KB per stage) beat 4 x 4
// by 4 %.  Both keep 48 KB or less per warp, so every warp of that shape is
// resident at once (4 per SM).
#ifndef MGS_PSL_FWD_TS
#define MGS_PSL_FWD_TS 12
#endif
#ifndef MGS_PSL_FWD_NS
#define MGS_PSL_FWD_NS 4
#endif
#ifndef MGS_PSL_BWD_TS
#define MGS_PSL_BWD_TS 8
#endif
#ifndef MGS_PSL_BWD_NS
#define MGS_PSL_BWD_NS 2
#endif
constexpr int kFwdTS = MGS_PSL_FWD_TS, kFwdNS = MGS_PSL_FWD_NS;
constexpr int kBwdTS = MGS_PSL_BWD_TS, kBwdNS = MGS_PSL_BWD_NS;

// log2(2^x + 2^y); both -inf gives -inf (avoids inf - inf).
__device__ __forceinline__ float logaddexp2_f(float x, float y) {
    const float m = fmaxf(x, y);
    const float r = m + lg2_approx(1.f + ex2_approx(-fabsf(x - y)));
    return (m == -CUDART_INF_F) ? m : r;
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

cudaError_t make_rows_map(CUtensorMap *m, const float *base, int64_t rows, int64_t D, int TS) {
    const uint64_t dims[2] = {uint64_t(D), uint64_t(rows)};
    const uint64_t str[1] = {uint64_t(D) * 4u};
    const uint32_t box[2] = {uint32_t(kChan), uint32_t(TS)};
    return make_tmap(m, base, 2, dims, str, box);
}

// ---------------------------------------------------------------- forward
__global__ void __launch_bounds__(32)
    psl_fwd_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmV,
                   const float *__restrict__ lh0, float *__restrict__ h, float *__restrict__ logh,
                   int64_t B, int64_t T, int64_t D, int64_t groups_per_b, DevCtl ctl) {
    using R = PslRing<2, kFwdTS, kFwdNS>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + R::ring_bytes);

    const int64_t bi = g / groups_per_b;
    const int c0 = int(g % groups_per_b) * kChan;
    const bool active = c0 + 4 * lane < D;
    const int64_t nblk = (T + kFwdTS - 1) / kFwdTS;
    const int row0 = int(bi * T);

    WarpRing<kFwdNS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmV);
    }
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * R::STAGEF;
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        tma_load_2d(st, &tmC, c0, row0 + int(j * kFwdTS), &bars[s], pol);
        tma_load_2d(st + R::BOXF, &tmV, c0, row0 + int(j * kFwdTS), &bars[s], pol);
    };
    const int npro = int(min64(kFwdNS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float4 L;  // log2 h_{t-1} for the thread's four channels
    if (lh0 != nullptr && active) {
        const float4 l = ld4(lh0 + bi * D + c0 + 4 * lane);
        L = make_float4(l.x * kLog2e, l.y * kLog2e, l.z * kLog2e, l.w * kLog2e);
    } else {
        L = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
    }
    float *hp = h + bi * T * D + c0 + 4 * lane;
    float *lp = (logh != nullptr) ? logh + bi * T * D + c0 + 4 * lane : nullptr;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % kFwdNS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(kFwdTS, T - j * kFwdTS));
        const float *sc = ring + size_t(s) * R::STAGEF + 4 * lane;
        const float *sv = sc + R::BOXF;
#pragma unroll
        for (int u = 0; u < kFwdTS; ++u) {
            if (u < n) {
                const float4 a = ld4(sc + u * kChan);
                const float4 v = ld4(sv + u * kChan);
                L.x = logaddexp2_f(fmaf(a.x, kLog2e, L.x), v.x * kLog2e);
                L.y = logaddexp2_f(fmaf(a.y, kLog2e, L.y), v.y * kLog2e);
                L.z = logaddexp2_f(fmaf(a.z, kLog2e, L.z), v.z * kLog2e);
                L.w = logaddexp2_f(fmaf(a.w, kLog2e, L.w), v.w * kLog2e);
                if (active) {
                    st_cs4(hp, make_float4(ex2_approx(L.x), ex2_approx(L.y), ex2_approx(L.z), ex2_approx(L.w)));
                    if (lp != nullptr) {
                        st_cs4(lp, make_float4(L.x * kLn2, L.y * kLn2, L.z * kLn2, L.w * kLn2));
                        lp += D;
                    }
                }
                hp += D;
            }
        }
        __syncwarp();
        if (j + kFwdNS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + kFwdNS);
            }
            rg.armed(s);
        }
    }
}

// ---------------------------------------------------------------- backward
__global__ void __launch_bounds__(32)
    psl_bwd_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmH,
                   const float *__restrict__ lh0, float *__restrict__ dlc, float *__restrict__ dlv,
                   float *__restrict__ dlh0, int64_t B, int64_t T, int64_t D, int64_t groups_per_b,
                   DevCtl ctl) {
    using R = PslRing<4, kBwdTS, kBwdNS>;  // log_coeffs_t, log_values_t, g_t, h_{t-1}
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + R::ring_bytes);

    const int64_t bi = g / groups_per_b;
    const int c0 = int(g % groups_per_b) * kChan;
    const bool active = c0 + 4 * lane < D;
    const int64_t nblk = (T + kBwdTS - 1) / kBwdTS;

    WarpRing<kBwdNS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmH);
    }
    // Block j covers t = T-1-j*TS down to max(0, T-(j+1)*TS); box row of step
    // u is TS-1-u; the h box starts one row earlier and holds h_{t-1}.
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * R::STAGEF;
        const int r0 = int(bi * T + T - (j + 1) * kBwdTS);
        mbar_arrive_expect_tx(&bars[s], uint32_t(R::stage_bytes));
        tma_load_2d(st, &tmC, c0, r0, &bars[s], pol);
        tma_load_2d(st + R::BOXF, &tmV, c0, r0, &bars[s], pol);
        tma_load_2d(st + 2 * R::BOXF, &tmG, c0, r0, &bars[s], pol);
        tma_load_2d(st + 3 * R::BOXF, &tmH, c0, r0 - 1, &bars[s], pol);
    };
    const int npro = int(min64(kBwdNS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float4 h0v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lh0 != nullptr && active) {
        const float4 l = ld4(lh0 + bi * D + c0 + 4 * lane);
        h0v = make_float4(ex2_approx(l.x * kLog2e), ex2_approx(l.y * kLog2e), ex2_approx(l.z * kLog2e),
                          ex2_approx(l.w * kLog2e));
    }
    float4 nx = make_float4(0.f, 0.f, 0.f, 0.f);  // a_{t+1} lambda_{t+1}
    const int64_t out0 = bi * T * D + c0 + 4 * lane;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % kBwdNS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tt = T - 1 - j * kBwdTS;
        const int n = int(min64(kBwdTS, tt + 1));
        const float *st = ring + size_t(s) * R::STAGEF + 4 * lane;
#pragma unroll
        for (int u = 0; u < kBwdTS; ++u) {
            if (u < n) {
                const int64_t t = tt - u;
                const int q = (kBwdTS - 1 - u) * kChan;
                const float4 c = ld4(st + q), v = ld4(st + R::BOXF + q), gg = ld4(st + 2 * R::BOXF + q);
                const float4 hp = (t >= 1) ? ld4(st + 3 * R::BOXF + q) : h0v;
                const float4 a = make_float4(ex2_approx(c.x * kLog2e), ex2_approx(c.y * kLog2e),
                                             ex2_approx(c.z * kLog2e), ex2_approx(c.w * kLog2e));
                const float4 lam = make_float4(gg.x + nx.x, gg.y + nx.y, gg.z + nx.z, gg.w + nx.w);
                nx = make_float4(a.x * lam.x, a.y * lam.y, a.z * lam.z, a.w * lam.w);
                if (active) {
                    const int64_t o = out0 + t * D;
                    st_cs4(dlv + o, make_float4(lam.x * ex2_approx(v.x * kLog2e), lam.y * ex2_approx(v.y * kLog2e),
                                                lam.z * ex2_approx(v.z * kLog2e), lam.w * ex2_approx(v.w * kLog2e)));
                    st_cs4(dlc + o, make_float4(nx.x * hp.x, nx.y * hp.y, nx.z * hp.z, nx.w * hp.w));
                }
            }
        }
        __syncwarp();
        if (j + kBwdNS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + kBwdNS);
            }
            rg.armed(s);
        }
    }
    if (dlh0 != nullptr && active) {
        *reinterpret_cast<float4 *>(dlh0 + bi * D + c0 + 4 * lane) =
            make_float4(nx.x * h0v.x, nx.y * h0v.y, nx.z * h0v.z, nx.w * h0v.w);
    }
}


// ---------------------------------------------------------------- backward, recomputing h
// Backward without the saved forward output (the pages' log-space op
// recomputes its forward).  Phase A runs the forward recurrence once over the
// whole sequence and writes log2 h at the start of every kRcS-step segment to
// the workspace.  Phase B walks the segments from the last to the first: each
// segment's log_coeffs, log_values and grad_h arrive by TMA into one of two
// buffers (the next segment's loads are in flight while this one is used), h
// over the segment is recomputed from its checkpoint into registers, and the
// reverse sweep of the saved-h kernel runs over it.  DRAM traffic is 28
// bytes per element (log_coeffs and log_values are read twice) against 24 with
// the saved h; what it saves is keeping h.
constexpr int kRcS = 16;   // steps per segment (checkpoint spacing)
constexpr int kRcNA = 3;   // phase-A stages

struct RcLayout {
    static constexpr int BOXF = kRcS * kChan;                        // floats per tensor box
    static constexpr size_t a_bytes = size_t(kRcNA) * 2 * BOXF * 4;  // phase A: lc, lv per stage
    static constexpr size_t b_bytes = size_t(2) * 3 * BOXF * 4;      // phase B: 2 x (lc, lv, g)
    static constexpr size_t ring_bytes = a_bytes > b_bytes ? a_bytes : b_bytes;
    static constexpr size_t warp_bytes = align_up(ring_bytes + (kRcNA + 2) * sizeof(uint64_t), 128);
};

__global__ void __launch_bounds__(32)
    psl_bwd_recompute_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmV,
                             const __grid_constant__ CUtensorMap tmG, const float *__restrict__ lh0,
                             float *__restrict__ dlc, float *__restrict__ dlv, float *__restrict__ dlh0,
                             float *__restrict__ ckpt, int64_t B, int64_t T, int64_t D, int64_t groups_per_b,
                             DevCtl ctl) {
    using L = RcLayout;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    uint64_t *barsA = reinterpret_cast<uint64_t *>(smem_raw + L::ring_bytes);
    uint64_t *barsB = barsA + kRcNA;

    const int64_t bi = g / groups_per_b;
    const int c0 = int(g % groups_per_b) * kChan;
    const bool active = c0 + 4 * lane < D;
    const int64_t nseg = (T + kRcS - 1) / kRcS;
    const int row0 = int(bi * T);
    float *ck = ckpt + bi * nseg * D + c0 + 4 * lane;  // checkpoint of segment j at ck + j*D
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmG);
    }

    // ---- phase A: forward, checkpoints
    float4 Lg;
    if (lh0 != nullptr && active) {
        const float4 l = ld4(lh0 + bi * D + c0 + 4 * lane);
        Lg = make_float4(l.x * kLog2e, l.y * kLog2e, l.z * kLog2e, l.w * kLog2e);
    } else {
        Lg = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
    }
    const float4 L0 = Lg;
    if (active) *reinterpret_cast<float4 *>(ck) = Lg;
    {
        WarpRing<kRcNA> ra;
        ra.init(barsA, lane);
        auto issueA = [&](int s, int64_t j) {  // lane 0 only
            float *st = ring + size_t(s) * 2 * L::BOXF;
            mbar_arrive_expect_tx(&barsA[s], uint32_t(2 * L::BOXF * 4));
            tma_load_2d(st, &tmC, c0, row0 + int(j * kRcS), &barsA[s], pol);
            tma_load_2d(st + L::BOXF, &tmV, c0, row0 + int(j * kRcS), &barsA[s], pol);
        };
        const int npro = int(min64(kRcNA, nseg));
        if (lane == 0)
            for (int s = 0; s < npro; ++s) issueA(s, s);
        for (int s = 0; s < npro; ++s) ra.armed(s);
        for (int64_t j = 0; j < nseg; ++j) {
            const int s = int(j % kRcNA);
            if (!ra.wait(s, ctl)) {
                if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
                ra.drain(ctl, lane);
                return;
            }
            const int n = int(min64(kRcS, T - j * kRcS));
            const float *sc = ring + size_t(s) * 2 * L::BOXF + 4 * lane;
            const float *sv = sc + L::BOXF;
#pragma unroll
            for (int u = 0; u < kRcS; ++u) {
                if (u < n) {
                    const float4 a = ld4(sc + u * kChan), v = ld4(sv + u * kChan);
                    Lg.x = logaddexp2_f(fmaf(a.x, kLog2e, Lg.x), v.x * kLog2e);
                    Lg.y = logaddexp2_f(fmaf(a.y, kLog2e, Lg.y), v.y * kLog2e);
                    Lg.z = logaddexp2_f(fmaf(a.z, kLog2e, Lg.z), v.z * kLog2e);
                    Lg.w = logaddexp2_f(fmaf(a.w, kLog2e, Lg.w), v.w * kLog2e);
                }
            }
            __syncwarp();
            if (j + kRcNA < nseg) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issueA(s, j + kRcNA);
                }
                ra.armed(s);
            }
            if (j + 1 < nseg && active) *reinterpret_cast<float4 *>(ck + (j + 1) * D) = Lg;
        }
    }

    // ---- phase B: segments from the last to the first
    __syncwarp();
    if (lane == 0) fence_proxy_async_smem();  // phase-A reads of the ring precede phase-B copies into it
    WarpRing<2> rb;
    rb.init(barsB, lane);
    auto issueB = [&](int buf, int64_t j) {  // lane 0 only
        float *st = ring + size_t(buf) * 3 * L::BOXF;
        mbar_arrive_expect_tx(&barsB[buf], uint32_t(3 * L::BOXF * 4));
        tma_load_2d(st, &tmC, c0, row0 + int(j * kRcS), &barsB[buf], pol);
        tma_load_2d(st + L::BOXF, &tmV, c0, row0 + int(j * kRcS), &barsB[buf], pol);
        tma_load_2d(st + 2 * L::BOXF, &tmG, c0, row0 + int(j * kRcS), &barsB[buf], pol);
    };
    const int nprob = int(min64(2, nseg));
    if (lane == 0)
        for (int b2 = 0; b2 < nprob; ++b2) issueB(b2, nseg - 1 - b2);
    for (int b2 = 0; b2 < nprob; ++b2) rb.armed(b2);

    float4 nx = make_float4(0.f, 0.f, 0.f, 0.f);  // a_{t+1} lambda_{t+1}
    // each segment's checkpoint is read one segment ahead (a global read at the
    // top of a segment would sit on its critical path)
    float4 Lnext = active ? ld4(ck + (nseg - 1) * D) : L0;
    for (int64_t jj = 0; jj < nseg; ++jj) {
        const int64_t j = nseg - 1 - jj;
        const int buf = int(jj & 1);
        const float4 Ls = Lnext;
        if (j >= 1 && active) Lnext = ld4(ck + (j - 1) * D);
        if (!rb.wait(buf, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rb.drain(ctl, lane);
            return;
        }
        const int n = int(min64(kRcS, T - j * kRcS));
        const float *sc = ring + size_t(buf) * 3 * L::BOXF + 4 * lane;
        const float *sv = sc + L::BOXF;
        const float *sg = sc + 2 * L::BOXF;
        // h over the segment, from its checkpoint
        float4 hreg[kRcS];
        float4 Lr = Ls;
#pragma unroll
        for (int u = 0; u < kRcS; ++u) {
            if (u < n) {
                const float4 a = ld4(sc + u * kChan), v = ld4(sv + u * kChan);
                Lr.x = logaddexp2_f(fmaf(a.x, kLog2e, Lr.x), v.x * kLog2e);
                Lr.y = logaddexp2_f(fmaf(a.y, kLog2e, Lr.y), v.y * kLog2e);
                Lr.z = logaddexp2_f(fmaf(a.z, kLog2e, Lr.z), v.z * kLog2e);
                Lr.w = logaddexp2_f(fmaf(a.w, kLog2e, Lr.w), v.w * kLog2e);
                hreg[u] = make_float4(ex2_approx(Lr.x), ex2_approx(Lr.y), ex2_approx(Lr.z), ex2_approx(Lr.w));
            }
        }
        const float4 hstart = make_float4(ex2_approx(Ls.x), ex2_approx(Ls.y), ex2_approx(Ls.z), ex2_approx(Ls.w));
        // reverse sweep over the segment
#pragma unroll
        for (int u = kRcS - 1; u >= 0; --u) {
            if (u < n) {
                const float4 c = ld4(sc + u * kChan), v = ld4(sv + u * kChan), gg = ld4(sg + u * kChan);
                const float4 hp = (u >= 1) ? hreg[u >= 1 ? u - 1 : 0] : hstart;
                const float4 a = make_float4(ex2_approx(c.x * kLog2e), ex2_approx(c.y * kLog2e),
                                             ex2_approx(c.z * kLog2e), ex2_approx(c.w * kLog2e));
                const float4 lam = make_float4(gg.x + nx.x, gg.y + nx.y, gg.z + nx.z, gg.w + nx.w);
                nx = make_float4(a.x * lam.x, a.y * lam.y, a.z * lam.z, a.w * lam.w);
                if (active) {
                    const int64_t o = (bi * T + j * kRcS + u) * D + c0 + 4 * lane;
                    st_cs4(dlv + o, make_float4(lam.x * ex2_approx(v.x * kLog2e), lam.y * ex2_approx(v.y * kLog2e),
                                                lam.z * ex2_approx(v.z * kLog2e), lam.w * ex2_approx(v.w * kLog2e)));
                    st_cs4(dlc + o, make_float4(nx.x * hp.x, nx.y * hp.y, nx.z * hp.z, nx.w * hp.w));
                }
            }
        }
        __syncwarp();
        if (jj + 2 < nseg) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issueB(buf, j - 2);
            }
            rb.armed(buf);
        }
    }
    if (dlh0 != nullptr && active) {
        const float4 h0v = make_float4(ex2_approx(L0.x), ex2_approx(L0.y), ex2_approx(L0.z), ex2_approx(L0.w));
        *reinterpret_cast<float4 *>(dlh0 + bi * D + c0 + 4 * lane) =
            make_float4(nx.x * h0v.x, nx.y * h0v.y, nx.z * h0v.z, nx.w * h0v.w);
    }
}

}  // namespace

cudaError_t launch_psl_fwd(const float *lc, const float *lv, const float *lh0, float *h,
                           float *logh, int64_t B, int64_t T, int64_t D, const DevCtl &ctl,
                           cudaStream_t s) {
    using R = PslRing<2, kFwdTS, kFwdNS>;
    CUtensorMap tC, tV;
    cudaError_t e;
    if ((e = make_rows_map(&tC, lc, B * T, D, kFwdTS)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tV, lv, B * T, D, kFwdTS)) != cudaSuccess) return e;
    const int64_t gpb = (D + kChan - 1) / kChan;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(R::warp_bytes);
    if ((e = ensure_smem_attr((const void *)psl_fwd_kernel, smem)) != cudaSuccess) return e;
    psl_fwd_kernel<<<dim3(unsigned(blocks)), 32, smem, s>>>(tC, tV, lh0, h, logh, B, T, D, gpb, ctl);
    return cudaGetLastError();
}

cudaError_t launch_psl_bwd(const float *lc, const float *lv, const float *lh0, const float *h,
                           const float *gh, float *dlc, float *dlv, float *dlh0, int64_t B,
                           int64_t T, int64_t D, const DevCtl &ctl, cudaStream_t s) {
    using R = PslRing<4, kBwdTS, kBwdNS>;
    CUtensorMap tC, tV, tG, tH;
    cudaError_t e;
    if ((e = make_rows_map(&tC, lc, B * T, D, kBwdTS)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tV, lv, B * T, D, kBwdTS)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tG, gh, B * T, D, kBwdTS)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tH, h, B * T, D, kBwdTS)) != cudaSuccess) return e;
    const int64_t gpb = (D + kChan - 1) / kChan;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(R::warp_bytes);
    if ((e = ensure_smem_attr((const void *)psl_bwd_kernel, smem)) != cudaSuccess) return e;
    psl_bwd_kernel<<<dim3(unsigned(blocks)), 32, smem, s>>>(tC, tV, tG, tH, lh0, dlc, dlv, dlh0, B, T, D, gpb, ctl);
    return cudaGetLastError();
}

size_t psl_recompute_workspace_bytes(int64_t B, int64_t T, int64_t D) {
    const int64_t nseg = (T + kRcS - 1) / kRcS;
    return size_t(B) * size_t(nseg) * size_t(D) * sizeof(float);
}

cudaError_t launch_psl_bwd_recompute(const float *lc, const float *lv, const float *lh0, const float *gh,
                                     float *dlc, float *dlv, float *dlh0, void *ws, int64_t B, int64_t T,
                                     int64_t D, const DevCtl &ctl, cudaStream_t s) {
    CUtensorMap tC, tV, tG;
    cudaError_t e;
    if ((e = make_rows_map(&tC, lc, B * T, D, kRcS)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tV, lv, B * T, D, kRcS)) != cudaSuccess) return e;
    if ((e = make_rows_map(&tG, gh, B * T, D, kRcS)) != cudaSuccess) return e;
    const int64_t gpb = (D + kChan - 1) / kChan;
    const int64_t blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(RcLayout::warp_bytes);
    if ((e = ensure_smem_attr((const void *)psl_bwd_recompute_kernel, smem)) != cudaSuccess) return e;
    psl_bwd_recompute_kernel<<<dim3(unsigned(blocks)), 32, smem, s>>>(tC, tV, tG, lh0, dlc, dlv, dlh0,
                                                                     static_cast<float *>(ws), B, T, D, gpb, ctl);
    return cudaGetLastError();
}

}  // namespace mgs
