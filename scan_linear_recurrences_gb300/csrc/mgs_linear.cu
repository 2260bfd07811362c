// The diagonal linear recurrence (matrix_affine_scan with k = 1, which
// linear_scan is; "mingru-scans" home page, scan-op table, linear_scan row)
// scanned in parallel over time in one launch:
//   h_t = a_t h_{t-1} + b_t                     (forward)
//   lambda_t = g_t + a_{t+1} lambda_{t+1}       (backward; db_t = lambda_t,
//   da_t = lambda_t h_{t-1}, dh0 = a_0 lambda_0)
// One thread-block cluster of S CTAs owns 32 channels of one batch row
// (thread = channel, so every load and store of a warp is 128 contiguous
// bytes); CTA r holds the r-th segment of W*L steps and each of its W warps L
// consecutive steps, with their inputs in registers (read once).  A warp
// composes its steps into one affine map (x_end = m x_start + c), warp 0
// composes the warps' maps into each warp's offset within the CTA and the
// CTA's total, and after a cluster barrier every CTA applies the totals of
// the CTAs before it (read from their shared memory) to h0 to get the state
// entering its segment.  Each warp then walks its steps from its own entry
// state.  No workspace; T <= S W L = 1024.
//
// parallel_scan_log with few lanes runs on the same skeleton (the
// "mingru-scans" home page, scan-op table, parallel_scan_log row, at its lab
// and long-T shapes).  In base 2 (a = log_coeffs log2 e, v = log_values
// log2 e) a step is L_t = logaddexp2(a_t + L_{t-1}, v_t), and steps s..e
// act on the state entering them as x -> logaddexp2(A + x, V) with
// A = a_s + ... + a_e and V the steps run from L = -inf; two such maps, p
// then q, compose to A = A_p + A_q, V = logaddexp2(A_q + V_p, V_q).  Every
// step's own arithmetic is that of the one-warp-per-128-channels kernel.
// Its backward is the linear recurrence lambda_t = g_t + a_{t+1} lambda_{t+1}
// (a = exp(log_coeffs)), as above, with d_log_values = lambda_t exp(lv_t),
// d_log_coeffs = a_t lambda_t h_{t-1}, d_log_h0 = a_0 lambda_0 h_0.  It
// runs up to T = 32768 with the *_mb_ kernels at the end of this file: the
// same scheme with each warp holding R blocks of L = 8 steps; the first walk
// composes all of them, the second reads each block again (from L2) as it
// reruns it, both loading the next block(s) while one (the forward: two side
// by side) is worked on.  The backward without the saved h always runs
// there, whatever T.
#include <math_constants.h>

#include "mgs_launch.h"
#include "mgs_device.cuh"
#include "mgs_cluster.cuh"

namespace mgs {
namespace {

constexpr int kLinWarps = 8;   // W
constexpr int kLinMaxCta = 8;  // S at most: the portable cluster size limit
constexpr int kLinMaxCtaWide = 16;  // S at most with few lane groups (non-portable cluster size)
constexpr int64_t kLinMaxT = int64_t(16) * kLinWarps * kLinMaxCta;  // one block a warp
constexpr int64_t kLinMaxTBlocks = 32768;  // several blocks a warp: R <= 64 blocks of 8 steps

struct LinSmem {
    float m[kLinWarps][32], c[kLinWarps][32];    // each warp's map
    float pm[kLinWarps][32], pc[kLinWarps][32];  // each warp's offset within the CTA
    float tm[32], tc[32];                        // the CTA's total map
};

// Warp 0: the warps' offsets within the CTA (in scan order: forward from warp
// 0, backward from warp W-1) and the CTA's total.
template <bool kRev>
__device__ __forceinline__ void lin_cta_offsets(LinSmem &s, int lane) {
    float pm = 1.f, pc = 0.f;
    for (int i = 0; i < kLinWarps; ++i) {
        const int k = kRev ? kLinWarps - 1 - i : i;
        s.pm[k][lane] = pm;
        s.pc[k][lane] = pc;
        pc = fmaf(s.m[k][lane], pc, s.c[k][lane]);
        pm *= s.m[k][lane];
    }
    s.tm[lane] = pm;
    s.tc[lane] = pc;
}

// The two synchronisations of the kernels.  With one CTA (no cluster) the
// first is a block barrier and the second is not needed.  Otherwise the first
// is a full cluster barrier (release: warp 0's totals become visible to the
// other CTAs), and the second is split: arrive (relaxed: the DSMEM loads have
// completed, their values are used before it) once this CTA has read the
// others' totals, wait just before exit.
template <bool kCl>
__device__ __forceinline__ void lin_sync1() {
    if constexpr (kCl) {
        cluster_arrive();
        cluster_wait();
    } else {
        __syncthreads();
    }
}
template <bool kCl>
__device__ __forceinline__ void lin_arrive2() {
    if constexpr (kCl) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
template <bool kCl>
__device__ __forceinline__ void lin_wait2() {
    if constexpr (kCl) cluster_wait();
}

// Steps of this warp inside [0, T) (none for a channel past D).
__device__ __forceinline__ int lin_steps_here(bool act, int L, int64_t t0, int64_t T) {
    return (!act || t0 >= T) ? 0 : int(min64(L, T - t0));
}

template <int L, bool kCl>
__global__ void __launch_bounds__(32 * kLinWarps)
    lin_fwd_kernel(const float *__restrict__ a, const float *__restrict__ b, const float *__restrict__ h0,
                   float *__restrict__ h, int64_t T, int64_t D, int64_t groups, int S) {
    __shared__ LinSmem sm;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned r = kCl ? cluster_rank() : 0u;
    const int64_t lg = blockIdx.x / S, bi = lg / groups;
    const int64_t ch = (lg - bi * groups) * 32 + lane;
    const bool act = ch < D;
    const int64_t t0 = (int64_t(r) * kLinWarps + w) * L;
    const int n = lin_steps_here(act, L, t0, T);
    const int64_t base = (bi * T + t0) * D + ch;
    const int ds = int(D);  // steps apart: 32-bit offsets
    const float hinit = (h0 != nullptr && act) ? h0[bi * D + ch] : 0.f;  // loaded with the inputs
    float av[L], bv[L];
#pragma unroll
    for (int u = 0; u < L; ++u) {
        av[u] = u < n ? a[base + u * ds] : 1.f;
        bv[u] = u < n ? b[base + u * ds] : 0.f;
    }
    float m = 1.f, c = 0.f;
#pragma unroll
    for (int u = 0; u < L; ++u) {
        c = fmaf(av[u], c, bv[u]);
        m *= av[u];
    }
    sm.m[w][lane] = m;
    sm.c[w][lane] = c;
    __syncthreads();
    if (w == 0) lin_cta_offsets<false>(sm, lane);
    lin_sync1<kCl>();
    // the state entering this CTA's segment: h0 through the CTAs before it
    float x = hinit;
    if constexpr (kCl)
        for (unsigned q = 0; q < r; ++q) x = fmaf(ld_dsmem(&sm.tm[lane], q), x, ld_dsmem(&sm.tc[lane], q));
    lin_arrive2<kCl>();  // done reading the other CTAs' shared memory
    x = fmaf(sm.pm[w][lane], x, sm.pc[w][lane]);
#pragma unroll
    for (int u = 0; u < L; ++u) {
        x = fmaf(av[u], x, bv[u]);
        if (u < n) __stcs(h + base + u * ds, x);
    }
    lin_wait2<kCl>();  // no CTA leaves while another may still read its shared memory
}

template <int L, bool kCl>
__global__ void __launch_bounds__(32 * kLinWarps)
    lin_bwd_kernel(const float *__restrict__ a, const float *__restrict__ h0, const float *__restrict__ h,
                   const float *__restrict__ g, float *__restrict__ da, float *__restrict__ db,
                   float *__restrict__ dh0, int64_t T, int64_t D, int64_t groups, int S) {
    __shared__ LinSmem sm;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned r = kCl ? cluster_rank() : 0u;
    const int64_t lg = blockIdx.x / S, bi = lg / groups;
    const int64_t ch = (lg - bi * groups) * 32 + lane;
    const bool act = ch < D;
    const int64_t t0 = (int64_t(r) * kLinWarps + w) * L;
    const int n = lin_steps_here(act, L, t0, T);
    const int64_t base = (bi * T + t0) * D + ch;
    const int ds = int(D);  // steps apart: 32-bit offsets
    const float hinit = (h0 != nullptr && act) ? h0[bi * D + ch] : 0.f;
    // step t's coefficient is a_{t+1} (none past the end: lambda_T = 0), and
    // da_t needs h_{t-1} (h0, or zero, before the first step); steps past n
    // are the identity
    float an[L], gv[L], hp[L];
#pragma unroll
    for (int u = 0; u < L; ++u) {
        an[u] = u < n ? (t0 + u + 1 < T ? a[base + (u + 1) * ds] : 0.f) : 1.f;
        gv[u] = u < n ? g[base + u * ds] : 0.f;
        hp[u] = u < n ? (t0 + u >= 1 ? h[base + (u - 1) * ds] : hinit) : 0.f;
    }
    float m = 1.f, c = 0.f;
#pragma unroll
    for (int u = L - 1; u >= 0; --u) {
        c = fmaf(an[u], c, gv[u]);
        m *= an[u];
    }
    sm.m[w][lane] = m;
    sm.c[w][lane] = c;
    __syncthreads();
    if (w == 0) lin_cta_offsets<true>(sm, lane);
    lin_sync1<kCl>();
    // lambda leaving this CTA's segment: zero past the end through the CTAs after it
    float x = 0.f;
    if constexpr (kCl)
        for (int q = S - 1; q > int(r); --q)
            x = fmaf(ld_dsmem(&sm.tm[lane], unsigned(q)), x, ld_dsmem(&sm.tc[lane], unsigned(q)));
    lin_arrive2<kCl>();
    float lam = fmaf(sm.pm[w][lane], x, sm.pc[w][lane]);
#pragma unroll
    for (int u = L - 1; u >= 0; --u) {
        lam = fmaf(an[u], lam, gv[u]);
        if (u < n) {
            __stcs(db + base + u * ds, lam);
            __stcs(da + base + u * ds, lam * hp[u]);
        }
    }
    // lam is lambda_0 in the first warp of the first CTA
    if (r == 0 && w == 0 && act && dh0 != nullptr) dh0[bi * D + ch] = a[bi * T * D + ch] * lam;
    lin_wait2<kCl>();
}

// ---------------------------------------------------------------- parallel_scan_log
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// log2(2^x + 2^y), max-shifted; both -inf gives -inf.
__device__ __forceinline__ float lae2(float x, float y) {
    const float m = fmaxf(x, y);
    const float r = m + lg2_approx(1.f + ex2_approx(-fabsf(x - y)));
    return (m == -CUDART_INF_F) ? m : r;
}

// Warp 0: the log-space maps' offsets within the CTA (forward order) and the total.
__device__ __forceinline__ void psl_cta_offsets(LinSmem &s, int lane) {
    float pa = 0.f, pv = -CUDART_INF_F;
    for (int k = 0; k < kLinWarps; ++k) {
        s.pm[k][lane] = pa;
        s.pc[k][lane] = pv;
        pv = lae2(s.m[k][lane] + pv, s.c[k][lane]);
        pa += s.m[k][lane];
    }
    s.tm[lane] = pa;
    s.tc[lane] = pv;
}

template <int L, bool kCl>
__global__ void __launch_bounds__(32 * kLinWarps, 2)  // two CTAs per SM (clusters of 8 need them)
    psl_fwd_cl_kernel(const float *__restrict__ lc, const float *__restrict__ lv, const float *__restrict__ lh0,
                      float *__restrict__ h, float *__restrict__ logh, int64_t T, int64_t D, int64_t groups,
                      int S) {
    __shared__ LinSmem sm;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned r = kCl ? cluster_rank() : 0u;
    const int64_t lg = blockIdx.x / S, bi = lg / groups;
    const int64_t ch = (lg - bi * groups) * 32 + lane;
    const bool act = ch < D;
    const int64_t t0 = (int64_t(r) * kLinWarps + w) * L;
    const int n = lin_steps_here(act, L, t0, T);
    const int64_t base = (bi * T + t0) * D + ch;
    const float linit = (lh0 != nullptr && act) ? lh0[bi * D + ch] * kLog2e : -CUDART_INF_F;
    // steps past n are the identity: log_coeffs 0, log_values -inf
    float cv[L], vb[L];
#pragma unroll
    for (int u = 0; u < L; ++u) {
        cv[u] = u < n ? lc[base + u * D] : 0.f;
        vb[u] = u < n ? lv[base + u * D] * kLog2e : -CUDART_INF_F;
    }
    float A = 0.f, V = -CUDART_INF_F;
#pragma unroll
    for (int u = 0; u < L; ++u) {
        V = lae2(fmaf(cv[u], kLog2e, V), vb[u]);
        A = fmaf(cv[u], kLog2e, A);
    }
    sm.m[w][lane] = A;
    sm.c[w][lane] = V;
    __syncthreads();
    if (w == 0) psl_cta_offsets(sm, lane);
    lin_sync1<kCl>();
    // log2 h entering this CTA's segment: log h0 (or -inf) through the CTAs before it
    float x = linit;
    if constexpr (kCl)
        for (unsigned q = 0; q < r; ++q) x = lae2(ld_dsmem(&sm.tm[lane], q) + x, ld_dsmem(&sm.tc[lane], q));
    lin_arrive2<kCl>();
    x = lae2(sm.pm[w][lane] + x, sm.pc[w][lane]);
#pragma unroll
    for (int u = 0; u < L; ++u) {
        x = lae2(fmaf(cv[u], kLog2e, x), vb[u]);
        if (u < n) {
            __stcs(h + base + u * D, ex2_approx(x));
            if (logh != nullptr) __stcs(logh + base + u * D, x * kLn2);
        }
    }
    lin_wait2<kCl>();
}

template <int L, bool kCl>
__global__ void __launch_bounds__(32 * kLinWarps, 2)  // two CTAs per SM (clusters of 8 need them)
    psl_bwd_cl_kernel(const float *__restrict__ lc, const float *__restrict__ lv, const float *__restrict__ lh0,
                      const float *__restrict__ h, const float *__restrict__ g, float *__restrict__ dlc,
                      float *__restrict__ dlv, float *__restrict__ dlh0, int64_t T, int64_t D, int64_t groups,
                      int S) {
    __shared__ LinSmem sm;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned r = kCl ? cluster_rank() : 0u;
    const int64_t lg = blockIdx.x / S, bi = lg / groups;
    const int64_t ch = (lg - bi * groups) * 32 + lane;
    const bool act = ch < D;
    const int64_t t0 = (int64_t(r) * kLinWarps + w) * L;
    const int n = lin_steps_here(act, L, t0, T);
    const int64_t base = (bi * T + t0) * D + ch;
    const int ds = int(D);  // steps apart: 32-bit offsets
    const float h0v = (lh0 != nullptr && act) ? ex2_approx(lh0[bi * D + ch] * kLog2e) : 0.f;
    // a_t, exp(lv_t), g_t, h_{t-1} (h0 before the first step) of this warp's
    // steps, and a after its last step (zero past the end: lambda_T = 0)
    float at[L], ev[L], gv[L], hp[L];
#pragma unroll
    for (int u = 0; u < L; ++u) {
        at[u] = u < n ? ex2_approx(lc[base + u * ds] * kLog2e) : 1.f;
        ev[u] = u < n ? ex2_approx(lv[base + u * ds] * kLog2e) : 0.f;
        gv[u] = u < n ? g[base + u * ds] : 0.f;
        hp[u] = u < n ? (t0 + u >= 1 ? h[base + (u - 1) * ds] : h0v) : 0.f;
    }
    const float aft = (n > 0 && t0 + n < T) ? ex2_approx(lc[base + n * ds] * kLog2e) : 0.f;
    // step t's coefficient a_{t+1}; steps past n are the identity
    auto coef = [&](int u) { return u + 1 < n ? at[u + 1] : (u + 1 == n ? aft : 1.f); };
    float m = 1.f, c = 0.f;
#pragma unroll
    for (int u = L - 1; u >= 0; --u) {
        c = fmaf(coef(u), c, gv[u]);
        m *= coef(u);
    }
    sm.m[w][lane] = m;
    sm.c[w][lane] = c;
    __syncthreads();
    if (w == 0) lin_cta_offsets<true>(sm, lane);
    lin_sync1<kCl>();
    float x = 0.f;  // lambda past this CTA's segment
    if constexpr (kCl)
        for (int q = S - 1; q > int(r); --q)
            x = fmaf(ld_dsmem(&sm.tm[lane], unsigned(q)), x, ld_dsmem(&sm.tc[lane], unsigned(q)));
    lin_arrive2<kCl>();
    float lam = fmaf(sm.pm[w][lane], x, sm.pc[w][lane]);
#pragma unroll
    for (int u = L - 1; u >= 0; --u) {
        lam = fmaf(coef(u), lam, gv[u]);
        if (u < n) {
            __stcs(dlv + base + u * ds, lam * ev[u]);
            __stcs(dlc + base + u * ds, at[u] * lam * hp[u]);
        }
    }
    // lam is lambda_0 in the first warp of the first CTA
    if (r == 0 && w == 0 && act && dlh0 != nullptr) dlh0[bi * D + ch] = at[0] * lam * h0v;
    lin_wait2<kCl>();
}

// ---------------------------------------------------------------- several blocks a warp
// The kernels above with each warp holding R blocks of L steps, always
// launched as a cluster (of one CTA too, for short sequences in the
// recompute backward).  Kept apart from the one-block kernels, whose inputs
// stay in registers between the two walks.
// Where a thread's work lies: its channel's offset `cb` in a [B][T][D]
// tensor (element t at cb + t D), whether the channel exists, and the first
// step of its warp's R blocks.
struct LinLane {
    int lane, w;
    unsigned r;
    int64_t bi, ch, cb, t0;
    bool act;
};
template <int L>
__device__ __forceinline__ LinLane lin_lane(int64_t T, int64_t D, int64_t groups, int S, int R) {
    LinLane q;
    q.lane = threadIdx.x & 31;
    q.w = threadIdx.x >> 5;
    q.r = cluster_rank();
    const int64_t lg = blockIdx.x / S;
    q.bi = lg / groups;
    q.ch = (lg - q.bi * groups) * 32 + q.lane;
    q.act = q.ch < D;
    q.cb = q.bi * T * D + q.ch;
    q.t0 = (int64_t(q.r) * kLinWarps + q.w) * int64_t(R) * L;
    return q;
}

// Block k's raw log_coeffs and log_values into registers (steps past the
// block's end the identity; a plain function with restrict-qualified
// pointers, so the loads may be issued ahead of anything; the conversion to
// base 2 waits until the values are used, so that loading the next block
// while this one is composed stalls nothing); returns the block's step count.
template <int L>
__device__ __forceinline__ int psl_raw_block(const float *__restrict__ lc, const float *__restrict__ lv,
                                             const LinLane &q, int k, int64_t T, int64_t D, float (&cv)[L],
                                             float (&vr)[L]) {
    const int64_t tk = q.t0 + int64_t(k) * L, base = q.cb + tk * D;
    const int n = lin_steps_here(q.act, L, tk, T);
    const int ds = int(D);  // steps apart within a block: 32-bit offsets
    const float *pc = lc + base, *pv = lv + base;
#pragma unroll
    for (int u = 0; u < L; ++u) {
        cv[u] = u < n ? pc[u * ds] : 0.f;
        vr[u] = u < n ? pv[u * ds] : -CUDART_INF_F;
    }
    return n;
}

// The forward in two walks over the warp's blocks, two blocks at a time,
// with the next two loaded meanwhile (four block buffers).  The first walk
// takes each block's own map from the identity (two independent chains at a
// time) and chains those R maps into the map of the warp's blocks before
// each block, kept in dynamic shared memory (2 R floats a thread); the second
// turns that map and the state entering the warp into each block's entering
// state, so that two blocks are walked side by side as well.
template <int L>
__global__ void __launch_bounds__(32 * kLinWarps, 2)  // two CTAs per SM (clusters of 8 need them)
    psl_fwd_cl_mb_kernel(const float *__restrict__ lc, const float *__restrict__ lv, const float *__restrict__ lh0,
                      float *__restrict__ h, float *__restrict__ logh, int64_t T, int64_t D, int64_t groups,
                      int S, int R) {
    __shared__ LinSmem sm;
    extern __shared__ float pre[];  // [R][256] A, then [R][256] V: the warp's map before block k
    constexpr int NT = 32 * kLinWarps;
    float *preA = pre, *preV = pre + size_t(R) * NT;
    const LinLane q = lin_lane<L>(T, D, groups, S, R);
    const int lane = q.lane, w = q.w, tid = threadIdx.x;
    float c0[L], v0[L], c1[L], v1[L], c2[L], v2[L], c3[L], v3[L];
    // block k's raw inputs (identity steps past the warp's R blocks)
    auto ld = [&](int k, float (&cv)[L], float (&vr)[L]) {
        if (k < R) return psl_raw_block<L>(lc, lv, q, k, T, D, cv, vr);
#pragma unroll
        for (int u = 0; u < L; ++u) {
            cv[u] = 0.f;
            vr[u] = -CUDART_INF_F;
        }
        return 0;
    };
    float WA = 0.f, WV = -CUDART_INF_F;  // the warp's map of the blocks composed so far
    // blocks ka and ka + 1: their own maps side by side, then chained on
    auto compose2 = [&](int ka, const float (&ca)[L], const float (&va)[L], const float (&cb)[L],
                        const float (&vb)[L]) {
        float Aa = 0.f, Va = -CUDART_INF_F, Ab = 0.f, Vb = -CUDART_INF_F;
#pragma unroll
        for (int u = 0; u < L; ++u) {
            Va = lae2(fmaf(ca[u], kLog2e, Va), va[u] * kLog2e);
            Aa = fmaf(ca[u], kLog2e, Aa);
            Vb = lae2(fmaf(cb[u], kLog2e, Vb), vb[u] * kLog2e);
            Ab = fmaf(cb[u], kLog2e, Ab);
        }
        preA[size_t(ka) * NT + tid] = WA;
        preV[size_t(ka) * NT + tid] = WV;
        WV = lae2(Aa + WV, Va);
        WA += Aa;
        if (ka + 1 < R) {
            preA[size_t(ka + 1) * NT + tid] = WA;
            preV[size_t(ka + 1) * NT + tid] = WV;
            WV = lae2(Ab + WV, Vb);
            WA += Ab;
        }
    };
    ld(0, c0, v0);
    ld(1, c1, v1);
    for (int k = 0; k < R; k += 4) {
        if (k + 2 < R) {
            ld(k + 2, c2, v2);
            ld(k + 3, c3, v3);
        }
        compose2(k, c0, v0, c1, v1);
        if (k + 2 < R) {
            if (k + 4 < R) {
                ld(k + 4, c0, v0);
                ld(k + 5, c1, v1);
            }
            compose2(k + 2, c2, v2, c3, v3);
        }
    }
    sm.m[w][lane] = WA;
    sm.c[w][lane] = WV;
    __syncthreads();
    if (w == 0) psl_cta_offsets(sm, lane);
    lin_sync1<true>();
    // log2 h entering this CTA's segment: log h0 (or -inf) through the CTAs before it
    float x = (lh0 != nullptr && q.act) ? lh0[q.bi * D + q.ch] * kLog2e : -CUDART_INF_F;
    for (unsigned p = 0; p < q.r; ++p) x = lae2(ld_dsmem(&sm.tm[lane], p) + x, ld_dsmem(&sm.tc[lane], p));
    lin_arrive2<true>();
    x = lae2(sm.pm[w][lane] + x, sm.pc[w][lane]);  // entering the warp's blocks
    // blocks ka and ka + 1 (if any) side by side from their entering states
    auto walk2 = [&](int ka, int na, const float (&ca)[L], const float (&va)[L], int nb, const float (&cb)[L],
                     const float (&vb)[L]) {
        float xa = lae2(preA[size_t(ka) * NT + tid] + x, preV[size_t(ka) * NT + tid]);
        float xb = ka + 1 < R ? lae2(preA[size_t(ka + 1) * NT + tid] + x, preV[size_t(ka + 1) * NT + tid])
                              : -CUDART_INF_F;
        const int64_t ba = q.cb + (q.t0 + int64_t(ka) * L) * D;
        const int ds = int(D);
        float *ha = h + ba, *la = logh != nullptr ? logh + ba : nullptr;  // block ka + 1 at L * ds past them
#pragma unroll
        for (int u = 0; u < L; ++u) {
            xa = lae2(fmaf(ca[u], kLog2e, xa), va[u] * kLog2e);
            xb = lae2(fmaf(cb[u], kLog2e, xb), vb[u] * kLog2e);
            if (u < na) {
                __stcs(ha + u * ds, ex2_approx(xa));
                if (logh != nullptr) __stcs(la + u * ds, xa * kLn2);
            }
            if (u < nb) {
                __stcs(ha + (L + u) * ds, ex2_approx(xb));
                if (logh != nullptr) __stcs(la + (L + u) * ds, xb * kLn2);
            }
        }
    };
    int n0 = ld(0, c0, v0), n1 = ld(1, c1, v1), n2 = 0, n3 = 0;
    for (int k = 0; k < R; k += 4) {
        if (k + 2 < R) {
            n2 = ld(k + 2, c2, v2);
            n3 = ld(k + 3, c3, v3);
        }
        walk2(k, n0, c0, v0, n1, c1, v1);
        if (k + 2 < R) {
            if (k + 4 < R) {
                n0 = ld(k + 4, c0, v0);
                n1 = ld(k + 5, c1, v1);
            }
            walk2(k + 2, n2, c2, v2, n3, c3, v3);
        }
    }
    lin_wait2<true>();
}

// A backward's raw block: log_coeffs, g and the log_coeffs after the block
// (in *lca), with kLv log_values, with kH h_{t-1} (h0, or zero, before
// t = 0); pads give a = 1, exp(lv) = 0, g = 0.  h is read only with kH.
template <int L, bool kLv, bool kH>
__device__ __forceinline__ int psl_bwd_raw(const float *__restrict__ lc, const float *__restrict__ lv,
                                           const float *__restrict__ h, const float *__restrict__ g, const LinLane &q,
                                           int k, int64_t T, int64_t D, float h0v, float (&lcr)[L], float (&lvr)[L],
                                           float (&gr)[L], float (&hr)[L], float *lca) {
    const int64_t tk = q.t0 + int64_t(k) * L, base = q.cb + tk * D;
    const int n = lin_steps_here(q.act, L, tk, T);
    const int ds = int(D);  // steps apart within a block: 32-bit offsets
    const float *plc = lc + base, *pg = g + base;
#pragma unroll
    for (int u = 0; u < L; ++u) {
        lcr[u] = u < n ? plc[u * ds] : 0.f;
        gr[u] = u < n ? pg[u * ds] : 0.f;
        if constexpr (kLv) lvr[u] = u < n ? lv[base + u * ds] : -CUDART_INF_F;
        if constexpr (kH) hr[u] = u < n ? (tk + u >= 1 ? h[base + (u - 1) * ds] : h0v) : 0.f;
    }
    *lca = (n > 0 && tk + n < T) ? plc[n * ds] : -CUDART_INF_F;
    return n;
}

// The saved-h backward with the blocks double-buffered as in the forward
// (raw inputs of the next block loaded while a block is walked; 8-step
// blocks, so that two buffers of four inputs fit the registers).
template <int L>
__global__ void __launch_bounds__(32 * kLinWarps, 2)  // two CTAs per SM (clusters of 8 need them)
    psl_bwd_cl_mb_kernel(const float *__restrict__ lc, const float *__restrict__ lv, const float *__restrict__ lh0,
                      const float *__restrict__ h, const float *__restrict__ g, float *__restrict__ dlc,
                      float *__restrict__ dlv, float *__restrict__ dlh0, int64_t T, int64_t D, int64_t groups,
                      int S, int R) {
    __shared__ LinSmem sm;
    const LinLane q = lin_lane<L>(T, D, groups, S, R);
    const int lane = q.lane, w = q.w;
    const float h0v = (lh0 != nullptr && q.act) ? ex2_approx(lh0[q.bi * D + q.ch] * kLog2e) : 0.f;
    float lc0[L], lv0[L], g0[L], h0r[L], lc1[L], lv1[L], g1[L], h1r[L], lca0 = 0.f, lca1 = 0.f;
    int n0 = 0, n1 = 0;
    // a of a block's steps and a after it; step u's coefficient a_{t+1}
    auto coefs = [&](const float (&lcr)[L], float lca, int n, float (&cf)[L], float (&at)[L]) {
#pragma unroll
        for (int u = 0; u < L; ++u) at[u] = ex2_approx(lcr[u] * kLog2e);
        const float aft = ex2_approx(lca * kLog2e);
#pragma unroll
        for (int u = 0; u < L; ++u) cf[u] = u + 1 < n ? at[u + 1 < L ? u + 1 : L - 1] : (u + 1 == n ? aft : 1.f);
    };
    float m = 1.f, c = 0.f;
    auto compose = [&](const float (&lcr)[L], const float (&gr)[L], float lca, int n) {
        float cf[L], at[L];
        coefs(lcr, lca, n, cf, at);
#pragma unroll
        for (int u = L - 1; u >= 0; --u) {
            c = fmaf(cf[u], c, gr[u]);
            m *= cf[u];
        }
    };
    auto load_map = [&](int k, float (&lcr)[L], float (&gr)[L], float (&lvr)[L], float (&hr)[L], float *lca) {
        return psl_bwd_raw<L, false, false>(lc, lv, h, g, q, k, T, D, h0v, lcr, lvr, gr, hr, lca);
    };
    // blocks R-1 .. 0, two at a time
    n0 = load_map(R - 1, lc0, g0, lv0, h0r, &lca0);
    for (int k = R - 1; k >= 0; k -= 2) {
        if (k >= 1) n1 = load_map(k - 1, lc1, g1, lv1, h1r, &lca1);
        compose(lc0, g0, lca0, n0);
        if (k >= 1) {
            if (k >= 2) n0 = load_map(k - 2, lc0, g0, lv0, h0r, &lca0);
            compose(lc1, g1, lca1, n1);
        }
    }
    sm.m[w][lane] = m;
    sm.c[w][lane] = c;
    __syncthreads();
    if (w == 0) lin_cta_offsets<true>(sm, lane);
    lin_sync1<true>();
    float x = 0.f;  // lambda past this CTA's segment
    for (int p = S - 1; p > int(q.r); --p)
        x = fmaf(ld_dsmem(&sm.tm[lane], unsigned(p)), x, ld_dsmem(&sm.tc[lane], unsigned(p)));
    lin_arrive2<true>();
    float lam = fmaf(sm.pm[w][lane], x, sm.pc[w][lane]);
    auto walk = [&](int k, int n, const float (&lcr)[L], const float (&lvr)[L], const float (&gr)[L],
                    const float (&hr)[L], float lca) {
        float cf[L], at[L];
        coefs(lcr, lca, n, cf, at);
        const int64_t base = q.cb + (q.t0 + int64_t(k) * L) * D;
        const int ds = int(D);
        float *pv = dlv + base, *pc = dlc + base;
#pragma unroll
        for (int u = L - 1; u >= 0; --u) {
            lam = fmaf(cf[u], lam, gr[u]);
            if (u < n) {
                __stcs(pv + u * ds, lam * ex2_approx(lvr[u] * kLog2e));
                __stcs(pc + u * ds, at[u] * lam * hr[u]);
            }
        }
        // lam is lambda_0 at block 0 of the first warp of the first CTA
        if (k == 0 && q.r == 0 && w == 0 && q.act && dlh0 != nullptr) dlh0[q.bi * D + q.ch] = at[0] * lam * h0v;
    };
    auto load = [&](int k, float (&lcr)[L], float (&lvr)[L], float (&gr)[L], float (&hr)[L], float *lca) {
        return psl_bwd_raw<L, true, true>(lc, lv, h, g, q, k, T, D, h0v, lcr, lvr, gr, hr, lca);
    };
    n0 = load(R - 1, lc0, lv0, g0, h0r, &lca0);
    for (int k = R - 1; k >= 0; k -= 2) {
        if (k >= 1) n1 = load(k - 1, lc1, lv1, g1, h1r, &lca1);
        walk(k, n0, lc0, lv0, g0, h0r, lca0);
        if (k >= 1) {
            if (k >= 2) n0 = load(k - 2, lc0, lv0, g0, h0r, &lca0);
            walk(k - 1, n1, lc1, lv1, g1, h1r, lca1);
        }
    }
    lin_wait2<true>();
}

// The recompute-mode backward with several blocks a warp, in two passes over
// the blocks, each double-buffered as above.  The first (left to right)
// composes the forward's log-space map and the backward's affine map
// (lambda_first = m lambda_after + c, extended a step at a time on the
// right: c += m g_t, m *= a_{t+1}) and keeps, per block, the forward map of
// the warp's blocks before it in dynamic shared memory (2 R floats a
// thread).  The second (right to left) turns that map and the state entering
// the warp into the block's entering state, rebuilds the block's h_{t-1} in
// registers and walks the backward through it.
template <int L>
__global__ void __launch_bounds__(32 * kLinWarps, 2)  // two CTAs per SM (clusters of 8 need them)
    psl_bwd_rc_cl_mb_kernel(const float *__restrict__ lc, const float *__restrict__ lv, const float *__restrict__ lh0,
                         const float *__restrict__ g, float *__restrict__ dlc, float *__restrict__ dlv,
                         float *__restrict__ dlh0, int64_t T, int64_t D, int64_t groups, int S, int R) {
    __shared__ LinSmem fm, bm;  // the forward's maps, the backward's
    extern __shared__ float pre[];  // [R][256] A then [R][256] V of the blocks before each block
    float *preA = pre, *preV = pre + size_t(R) * (32 * kLinWarps);
    const LinLane q = lin_lane<L>(T, D, groups, S, R);
    const int lane = q.lane, w = q.w, tid = threadIdx.x;
    const float l0 = (lh0 != nullptr && q.act) ? lh0[q.bi * D + q.ch] * kLog2e : -CUDART_INF_F;
    float lc0[L], lv0[L], g0[L], lc1[L], lv1[L], g1[L], hd[L], lca0 = 0.f, lca1 = 0.f;
    int n0 = 0, n1 = 0;
    auto coefs = [&](const float (&lcr)[L], float lca, int n, float (&cf)[L], float (&at)[L]) {
#pragma unroll
        for (int u = 0; u < L; ++u) at[u] = ex2_approx(lcr[u] * kLog2e);
        const float aft = ex2_approx(lca * kLog2e);
#pragma unroll
        for (int u = 0; u < L; ++u) cf[u] = u + 1 < n ? at[u + 1 < L ? u + 1 : L - 1] : (u + 1 == n ? aft : 1.f);
    };
    auto load = [&](int k, float (&lcr)[L], float (&lvr)[L], float (&gr)[L], float *lca) {
        return psl_bwd_raw<L, true, false>(lc, lv, nullptr, g, q, k, T, D, 0.f, lcr, lvr, gr, hd, lca);
    };
    float A = 0.f, V = -CUDART_INF_F, m = 1.f, c = 0.f;
    auto compose = [&](int k, const float (&lcr)[L], const float (&lvr)[L], const float (&gr)[L], float lca, int n) {
        preA[size_t(k) * (32 * kLinWarps) + tid] = A;
        preV[size_t(k) * (32 * kLinWarps) + tid] = V;
        float cf[L], at[L];
        coefs(lcr, lca, n, cf, at);
#pragma unroll
        for (int u = 0; u < L; ++u) {
            V = lae2(fmaf(lcr[u], kLog2e, V), lvr[u] * kLog2e);
            A = fmaf(lcr[u], kLog2e, A);
            c = fmaf(m, gr[u], c);
            m *= cf[u];
        }
    };
    n0 = load(0, lc0, lv0, g0, &lca0);
    for (int k = 0; k < R; k += 2) {
        if (k + 1 < R) n1 = load(k + 1, lc1, lv1, g1, &lca1);
        compose(k, lc0, lv0, g0, lca0, n0);
        if (k + 1 < R) {
            if (k + 2 < R) n0 = load(k + 2, lc0, lv0, g0, &lca0);
            compose(k + 1, lc1, lv1, g1, lca1, n1);
        }
    }
    fm.m[w][lane] = A;
    fm.c[w][lane] = V;
    bm.m[w][lane] = m;
    bm.c[w][lane] = c;
    __syncthreads();
    if (w == 0) {
        psl_cta_offsets(fm, lane);
        lin_cta_offsets<true>(bm, lane);
    }
    lin_sync1<true>();
    float x = l0, y = 0.f;  // log2 h entering the CTA's segment, lambda past it
    for (unsigned p = 0; p < q.r; ++p) x = lae2(ld_dsmem(&fm.tm[lane], p) + x, ld_dsmem(&fm.tc[lane], p));
    for (int p = S - 1; p > int(q.r); --p)
        y = fmaf(ld_dsmem(&bm.tm[lane], unsigned(p)), y, ld_dsmem(&bm.tc[lane], unsigned(p)));
    lin_arrive2<true>();
    x = lae2(fm.pm[w][lane] + x, fm.pc[w][lane]);  // log2 h entering the warp's segment
    float lam = fmaf(bm.pm[w][lane], y, bm.pc[w][lane]);
    auto walk = [&](int k, int n, const float (&lcr)[L], const float (&lvr)[L], const float (&gr)[L], float lca) {
        // the forward over this block: h_{t-1} of each step (h0, or zero, before t = 0)
        float xk = k == 0 ? x
                          : lae2(preA[size_t(k) * (32 * kLinWarps) + tid] + x, preV[size_t(k) * (32 * kLinWarps) + tid]);
        float hp[L], cf[L], at[L];
#pragma unroll
        for (int u = 0; u < L; ++u) {
            hp[u] = ex2_approx(xk);
            xk = lae2(fmaf(lcr[u], kLog2e, xk), lvr[u] * kLog2e);
        }
        coefs(lcr, lca, n, cf, at);
        const int64_t base = q.cb + (q.t0 + int64_t(k) * L) * D;
        const int ds = int(D);
        float *pv = dlv + base, *pc = dlc + base;
#pragma unroll
        for (int u = L - 1; u >= 0; --u) {
            lam = fmaf(cf[u], lam, gr[u]);
            if (u < n) {
                __stcs(pv + u * ds, lam * ex2_approx(lvr[u] * kLog2e));
                __stcs(pc + u * ds, at[u] * lam * hp[u]);
            }
        }
        // lam is lambda_0 and hp[0] is h0 at block 0 of the first warp of the first CTA
        if (k == 0 && q.r == 0 && w == 0 && q.act && dlh0 != nullptr) dlh0[q.bi * D + q.ch] = at[0] * lam * hp[0];
    };
    n0 = load(R - 1, lc0, lv0, g0, &lca0);
    for (int k = R - 1; k >= 0; k -= 2) {
        if (k >= 1) n1 = load(k - 1, lc1, lv1, g1, &lca1);
        walk(k, n0, lc0, lv0, g0, lca0);
        if (k >= 1) {
            if (k >= 2) n0 = load(k - 2, lc0, lv0, g0, &lca0);
            walk(k - 1, n1, lc1, lv1, g1, lca1);
        }
    }
    lin_wait2<true>();
}

struct LinPlan {
    int L, S;
};
// L = 8 steps a warp up to T = 512, 16 above; as many CTAs as the segments need.
LinPlan lin_plan(int64_t T) {
    LinPlan p;
    p.L = T <= int64_t(8) * kLinWarps * kLinMaxCta ? 8 : 16;
    p.S = int((T + int64_t(p.L) * kLinWarps - 1) / (int64_t(p.L) * kLinWarps));
    return p;
}
// Runs launch(plan): with fewer than 16 lane groups and T > 512 first in
// 8-step blocks on clusters of up to 16 CTAs (the non-portable size: twice
// the SMs for a few long sequences), falling back to lin_plan(T) if that
// launch fails.
template <typename F>
cudaError_t with_lin_plan(int64_t B, int64_t groups, int64_t T, F launch) {
    if (B * groups < 16 && T > int64_t(8) * kLinWarps * kLinMaxCta) {
        LinPlan w;
        w.L = 8;
        w.S = int((T + int64_t(8) * kLinWarps - 1) / (int64_t(8) * kLinWarps));
        if (launch(w) == cudaSuccess) return cudaSuccess;
        (void)cudaGetLastError();  // a launch-configuration error: not sticky
    }
    return launch(lin_plan(T));
}

// T in [1, 32768]: R blocks of L steps a warp, S CTAs a cluster, and
// smem_per_block bytes of dynamic shared memory a CTA for each of the R.
// With few lane groups (fewer than 16: fewer than 128 CTAs at 8 a cluster)
// a long sequence takes clusters of up to 16 CTAs (the non-portable size),
// twice the SMs (at 16 groups and more the wider clusters measured slower);
// if such a cluster cannot be launched the call falls back to 8.
template <int L, typename... KArgs, typename... Args>
cudaError_t launch_mb(void (*kern)(KArgs...), size_t smem_per_block, int64_t B, int64_t T, int64_t D,
                      cudaStream_t s, Args... args) {
    if (T > kLinMaxTBlocks) return cudaErrorInvalidConfiguration;
    const int64_t groups = (D + 31) / 32, cta_steps = int64_t(L) * kLinWarps;
    auto go = [&](int smax) -> cudaError_t {
        const int R = int((T + cta_steps * smax - 1) / (cta_steps * smax));
        const int S = int((T + cta_steps * R - 1) / (cta_steps * R));
        const int64_t blocks = B * groups * S;
        if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
        if (blocks == 0) return cudaSuccess;
        const size_t smem = smem_per_block * size_t(R);
        cudaError_t e;
        if (smem > 48 * 1024) {  // past the default limit (at most 128 KB: R <= 64)
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
                return e;
        }
        return launch_cluster(kern, blocks, 32 * kLinWarps, smem, S, s, args..., T, D, groups, S, R);
    };
    if (B * groups * kLinMaxCta < 128 && T > cta_steps * kLinMaxCta) {
        if (go(kLinMaxCtaWide) == cudaSuccess) return cudaSuccess;
        (void)cudaGetLastError();  // a launch-configuration error: not sticky
    }
    return go(kLinMaxCta);
}

}  // namespace

// Few channel groups (under 2048 warps of channels, where one thread walking
// a channel's whole sequence leaves the GPU latency-bound), and T <= 1024 for
// linear_scan (past that the three-launch chunked k = 1 path measured faster
// than several blocks a warp), T <= 32768 for parallel_scan_log.
static bool few_channel_groups(int64_t B, int64_t D) { return B >= 0 && D >= 0 && B * ((D + 31) / 32) < 2048; }
bool lin_supported(int64_t B, int64_t T, int64_t D) { return T >= 1 && T <= kLinMaxT && few_channel_groups(B, D); }
bool psl_cl_supported(int64_t B, int64_t T, int64_t D) {
    return T >= 1 && T <= kLinMaxTBlocks && few_channel_groups(B, D);
}

cudaError_t launch_lin_fwd(const float *a, const float *b, const float *h0, float *h, int64_t B, int64_t T,
                           int64_t D, cudaStream_t s) {
    const int64_t groups = (D + 31) / 32;
    if (T < 1 || T > kLinMaxT) return cudaErrorInvalidConfiguration;
#define LIN_FWD(L_, CL_) \
    launch_cluster(lin_fwd_kernel<L_, CL_>, blocks, 32 * kLinWarps, 0, p.S, s, a, b, h0, h, T, D, groups, p.S)
    // the standard plan only: the wider clusters measured slower for this
    // short kernel (B=1 T=1024 D=64 5.0 -> 5.8 us)
    const LinPlan p = lin_plan(T);
    const int64_t blocks = B * groups * p.S;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    if (blocks == 0) return cudaSuccess;
    if (p.L == 16) return LIN_FWD(16, true);  // T > 512: always more than one CTA
    return p.S == 1 ? LIN_FWD(8, false) : LIN_FWD(8, true);
#undef LIN_FWD
}

cudaError_t launch_lin_bwd(const float *a, const float *h0, const float *h, const float *g, float *da, float *db,
                           float *dh0, int64_t B, int64_t T, int64_t D, cudaStream_t s) {
    const int64_t groups = (D + 31) / 32;
    if (T < 1 || T > kLinMaxT) return cudaErrorInvalidConfiguration;
#define LIN_BWD(L_, CL_)                                                                                       \
    launch_cluster(lin_bwd_kernel<L_, CL_>, blocks, 32 * kLinWarps, 0, p.S, s, a, h0, h, g, da, db, dh0, T, D, groups, \
                   p.S)
    return with_lin_plan(B, groups, T, [&](const LinPlan &p) -> cudaError_t {
        const int64_t blocks = B * groups * p.S;
        if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
        if (blocks == 0) return cudaSuccess;
        if (p.L == 16) return LIN_BWD(16, true);  // T > 512: always more than one CTA
        return p.S == 1 ? LIN_BWD(8, false) : LIN_BWD(8, true);
    });
#undef LIN_BWD
}

cudaError_t launch_psl_fwd_cl(const float *lc, const float *lv, const float *lh0, float *h, float *logh, int64_t B,
                              int64_t T, int64_t D, cudaStream_t s) {
    if (T > kLinMaxT)
        return launch_mb<8>(psl_fwd_cl_mb_kernel<8>, 2 * sizeof(float) * 32 * kLinWarps, B, T, D, s, lc, lv, lh0, h,
                            logh);
    const int64_t groups = (D + 31) / 32;
    if (T < 1) return cudaErrorInvalidConfiguration;
#define PSL_FWD(L_, CL_)                                                                                     \
    launch_cluster(psl_fwd_cl_kernel<L_, CL_>, blocks, 32 * kLinWarps, 0, p.S, s, lc, lv, lh0, h, logh, T, D, \
                   groups, p.S)
    return with_lin_plan(B, groups, T, [&](const LinPlan &p) -> cudaError_t {
        const int64_t blocks = B * groups * p.S;
        if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
        if (blocks == 0) return cudaSuccess;
        if (p.L == 16) return PSL_FWD(16, true);  // T > 512: always more than one CTA
        return p.S == 1 ? PSL_FWD(8, false) : PSL_FWD(8, true);
    });
#undef PSL_FWD
}

cudaError_t launch_psl_bwd_cl(const float *lc, const float *lv, const float *lh0, const float *h, const float *g,
                              float *dlc, float *dlv, float *dlh0, int64_t B, int64_t T, int64_t D, cudaStream_t s) {
    if (T > kLinMaxT) return launch_mb<8>(psl_bwd_cl_mb_kernel<8>, 0, B, T, D, s, lc, lv, lh0, h, g, dlc, dlv, dlh0);
    const int64_t groups = (D + 31) / 32;
    if (T < 1) return cudaErrorInvalidConfiguration;
#define PSL_BWD(L_, CL_)                                                                                     \
    launch_cluster(psl_bwd_cl_kernel<L_, CL_>, blocks, 32 * kLinWarps, 0, p.S, s, lc, lv, lh0, h, g, dlc, dlv, \
                   dlh0, T, D, groups, p.S)
    return with_lin_plan(B, groups, T, [&](const LinPlan &p) -> cudaError_t {
        const int64_t blocks = B * groups * p.S;
        if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
        if (blocks == 0) return cudaSuccess;
        if (p.L == 16) return PSL_BWD(16, true);  // T > 512: always more than one CTA
        return p.S == 1 ? PSL_BWD(8, false) : PSL_BWD(8, true);
    });
#undef PSL_BWD
}

cudaError_t launch_psl_bwd_rc_cl(const float *lc, const float *lv, const float *lh0, const float *g, float *dlc,
                                 float *dlv, float *dlh0, int64_t B, int64_t T, int64_t D, cudaStream_t s) {
    // several-block kernel at every T (also where the forward and the saved-h
    // backward take one block a warp: its two walks over 8-step blocks beat a
    // one-block recompute kernel at every shape measured)
    if (T < 1) return cudaErrorInvalidConfiguration;
    return launch_mb<8>(psl_bwd_rc_cl_mb_kernel<8>, 2 * sizeof(float) * 32 * kLinWarps, B, T, D, s, lc, lv, lh0, g,
                        dlc, dlv, dlh0);
}

}  // namespace mgs
