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
// max(x, y) + log1p(exp(-|x - y|)).
// Backward walks t downwards in linear space (a_t = exp(log_coeffs_t) in (0, 1]
// for gates), lambda_t = g_t + a_{t+1} lambda_{t+1}.
//
// A warp owns 128 adjacent channels of one batch row (4 per thread, float4);
// each time step's rows arrive by 1-D TMA bulk copies into a per-warp ring.
#include <math_constants.h>

#include "mgs_launch.h"

namespace mgs {
namespace {

constexpr int kChan = 128;  // channels per warp
constexpr int kWarpsPerBlock = 1;
__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int NT, int TS, int NS>  // NT row-tensors per step
struct PslLayout {
    static constexpr int STEPF = NT * kChan;
    static constexpr size_t ring_bytes = size_t(NS) * TS * STEPF * sizeof(float);
    static constexpr size_t warp_bytes = align_up(ring_bytes + NS * sizeof(uint64_t), 128);
};

constexpr int kFwdTS = 8, kFwdNS = 4;  // 2 tensors x 512 B x 8 steps = 8 KB per stage
constexpr int kBwdTS = 4, kBwdNS = 4;  // 4 tensors x 512 B x 4 steps = 8 KB per stage

// The correction term log1p(exp(-|x - y|)) lies in [0, log 2]; computing it
// with the MUFU approximations (__expf, __logf) costs an absolute error of
// about 2e-7 in log h_t whatever the magnitude of x and y, i.e. a relative
// error of that size in h_t, well inside the fp32 parity bound.
__device__ __forceinline__ float logaddexp_f(float x, float y) {
    const float m = fmaxf(x, y);
    const float r = m + __logf(1.f + __expf(-fabsf(x - y)));
    // both -inf: the sum of two zeros is zero (avoid inf - inf)
    return (m == -CUDART_INF_F) ? m : r;
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// ---------------------------------------------------------------- forward
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    psl_fwd_kernel(const float *__restrict__ lc, const float *__restrict__ lv,
                   const float *__restrict__ lh0, float *__restrict__ h,
                   float *__restrict__ logh, int64_t B, int64_t T, int64_t D,
                   int64_t groups_per_b, DevCtl ctl) {
    using L = PslLayout<2, kFwdTS, kFwdNS>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = int64_t(blockIdx.x) * kWarpsPerBlock + warp;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw + size_t(warp) * L::warp_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + size_t(warp) * L::warp_bytes + L::ring_bytes);

    const int64_t bi = g / groups_per_b;
    const int64_t c0 = (g % groups_per_b) * kChan;
    const int nc = int(min64(kChan, D - c0));
    const bool active = 4 * lane < nc;
    const uint32_t row_bytes = uint32_t(nc) * 4u;
    const int64_t nblk = (T + kFwdTS - 1) / kFwdTS;

    WarpRing<kFwdNS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {
        const int64_t t0 = j * kFwdTS;
        const int n = int(min64(kFwdTS, T - t0));
        mbar_arrive_expect_tx(&bars[s], uint32_t(n) * 2u * row_bytes);
        for (int u = 0; u < n; ++u) {
            const int64_t off = (bi * T + t0 + u) * D + c0;
            float *st = ring + (size_t(s) * kFwdTS + u) * L::STEPF;
            bulk_g2s(st, lc + off, row_bytes, &bars[s], pol);
            bulk_g2s(st + kChan, lv + off, row_bytes, &bars[s], pol);
        }
    };
    const int npro = int(min64(kFwdNS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float4 Lg;  // log h_{t-1} for the thread's four channels
    if (lh0 != nullptr && active) {
        Lg = ld4(lh0 + bi * D + c0 + 4 * lane);
    } else {
        Lg = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
    }
    const int64_t out0 = bi * T * D + c0 + 4 * lane;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % kFwdNS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t t0 = j * kFwdTS;
        const int n = int(min64(kFwdTS, T - t0));
        const float *st = ring + size_t(s) * kFwdTS * L::STEPF;
#pragma unroll 4
        for (int u = 0; u < n; ++u) {
            const float4 a = ld4(st + u * L::STEPF + 4 * lane);
            const float4 v = ld4(st + u * L::STEPF + kChan + 4 * lane);
            Lg.x = logaddexp_f(a.x + Lg.x, v.x);
            Lg.y = logaddexp_f(a.y + Lg.y, v.y);
            Lg.z = logaddexp_f(a.z + Lg.z, v.z);
            Lg.w = logaddexp_f(a.w + Lg.w, v.w);
            if (active) {
                const int64_t o = out0 + (t0 + u) * D;
                st_cs4(h + o, make_float4(expf(Lg.x), expf(Lg.y), expf(Lg.z), expf(Lg.w)));
                if (logh != nullptr) st_cs4(logh + o, Lg);
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
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    psl_bwd_kernel(const float *__restrict__ lc, const float *__restrict__ lv,
                   const float *__restrict__ lh0, const float *__restrict__ h,
                   const float *__restrict__ gh, float *__restrict__ dlc,
                   float *__restrict__ dlv, float *__restrict__ dlh0, int64_t B, int64_t T,
                   int64_t D, int64_t groups_per_b, DevCtl ctl) {
    using L = PslLayout<4, kBwdTS, kBwdNS>;  // lc_t, lv_t, g_t, h_{t-1}
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = int64_t(blockIdx.x) * kWarpsPerBlock + warp;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw + size_t(warp) * L::warp_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + size_t(warp) * L::warp_bytes + L::ring_bytes);

    const int64_t bi = g / groups_per_b;
    const int64_t c0 = (g % groups_per_b) * kChan;
    const int nc = int(min64(kChan, D - c0));
    const bool active = 4 * lane < nc;
    const uint32_t row_bytes = uint32_t(nc) * 4u;
    const int64_t nblk = (T + kBwdTS - 1) / kBwdTS;

    WarpRing<kBwdNS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {
        const int64_t tt = T - 1 - j * kBwdTS;
        const int n = int(min64(kBwdTS, tt + 1));
        const int with_h = (tt - n + 1 >= 1) ? n : n - 1;
        mbar_arrive_expect_tx(&bars[s], uint32_t(3 * n + with_h) * row_bytes);
        for (int u = 0; u < n; ++u) {
            const int64_t t = tt - u;
            const int64_t off = (bi * T + t) * D + c0;
            float *st = ring + (size_t(s) * kBwdTS + u) * L::STEPF;
            bulk_g2s(st, lc + off, row_bytes, &bars[s], pol);
            bulk_g2s(st + kChan, lv + off, row_bytes, &bars[s], pol);
            bulk_g2s(st + 2 * kChan, gh + off, row_bytes, &bars[s], pol);
            if (t >= 1) bulk_g2s(st + 3 * kChan, h + off - D, row_bytes, &bars[s], pol);
        }
    };
    const int npro = int(min64(kBwdNS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float4 h0v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lh0 != nullptr && active) {
        const float4 l = ld4(lh0 + bi * D + c0 + 4 * lane);
        h0v = make_float4(expf(l.x), expf(l.y), expf(l.z), expf(l.w));
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
        const float *st = ring + size_t(s) * kBwdTS * L::STEPF;
#pragma unroll 4
        for (int u = 0; u < n; ++u) {
            const int64_t t = tt - u;
            const float *su = st + u * L::STEPF + 4 * lane;
            const float4 c = ld4(su), v = ld4(su + kChan), gg = ld4(su + 2 * kChan);
            const float4 hp = (t >= 1) ? ld4(su + 3 * kChan) : h0v;
            const float4 a = make_float4(expf(c.x), expf(c.y), expf(c.z), expf(c.w));
            const float4 lam = make_float4(gg.x + nx.x, gg.y + nx.y, gg.z + nx.z, gg.w + nx.w);
            nx = make_float4(a.x * lam.x, a.y * lam.y, a.z * lam.z, a.w * lam.w);
            if (active) {
                const int64_t o = out0 + t * D;
                st_cs4(dlv + o, make_float4(lam.x * expf(v.x), lam.y * expf(v.y), lam.z * expf(v.z),
                                            lam.w * expf(v.w)));
                st_cs4(dlc + o, make_float4(nx.x * hp.x, nx.y * hp.y, nx.z * hp.z, nx.w * hp.w));
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

}  // namespace

cudaError_t launch_psl_fwd(const float *lc, const float *lv, const float *lh0, float *h,
                           float *logh, int64_t B, int64_t T, int64_t D, const DevCtl &ctl,
                           cudaStream_t s) {
    using L = PslLayout<2, kFwdTS, kFwdNS>;
    const int64_t gpb = (D + kChan - 1) / kChan;
    const int smem = int(L::warp_bytes * kWarpsPerBlock);
    cudaError_t e = ensure_smem_attr((const void *)psl_fwd_kernel, smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (B * gpb + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    psl_fwd_kernel<<<dim3(unsigned(blocks)), kWarpsPerBlock * 32, smem, s>>>(lc, lv, lh0, h, logh, B, T, D, gpb, ctl);
    return cudaGetLastError();
}

cudaError_t launch_psl_bwd(const float *lc, const float *lv, const float *lh0, const float *h,
                           const float *gh, float *dlc, float *dlv, float *dlh0, int64_t B,
                           int64_t T, int64_t D, const DevCtl &ctl, cudaStream_t s) {
    using L = PslLayout<4, kBwdTS, kBwdNS>;
    const int64_t gpb = (D + kChan - 1) / kChan;
    const int smem = int(L::warp_bytes * kWarpsPerBlock);
    cudaError_t e = ensure_smem_attr((const void *)psl_bwd_kernel, smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (B * gpb + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    psl_bwd_kernel<<<dim3(unsigned(blocks)), kWarpsPerBlock * 32, smem, s>>>(lc, lv, lh0, h, gh, dlc, dlv, dlh0, B, T, D, gpb, ctl);
    return cudaGetLastError();
}

}  // namespace mgs
