// Givens-mesh affine and matrix scans: matrix_affine_scan and matrix_scan whose
// k x k transition is GivensMinGRU's brick-wall rotation mesh, fed by its
// k(k-1)/2 angles instead of the materialised matrix ("mingru-scans" home
// page, lineage paragraph: the Clements et al. mesh of Golub & Van Loan plane
// rotations; "Run the benchmarks", Step 3: the angle-fused backward).
//
//   G(theta) = L_k ... L_1, layer l rotating pairs (0,1),(2,3),.. (odd l) or
//   (1,2),(3,4),.. (even l); a rotation maps (x_p, x_{p+1}) to
//   (c x_p - s x_{p+1}, s x_p + c x_{p+1}).
//   affine:  h_t = G(theta_t) diag(a_t) h_{t-1} + b_t      (a optional)
//   matrix:  P_t = G(theta_t) P_{t-1},  P_0 = I
//
// Neither direction ever forms A_t or dA_t: the forward applies the 28
// rotations (k = 8) to the state, and the backward gets each angle's
// gradient from the rotated state and the adjoint at that rotation,
//   d theta = mu_{p+1} x_p - mu_p x_{p+1}   ((x, mu) just after the rotation),
// since d/dtheta of a rotation's output (x_p, x_{p+1}) is (-x_{p+1}, x_p).
// HBM bytes per step (k = 8) drop from 4(k^2 + 2k) = 320 to 4(28 + 3k) = 208
// forward and from 608 to 4(2*28 + 5k) = 384 backward for the affine scan.
//
// Mapping.  Affine scan: one thread per (batch, head) lane holds the whole
// state in registers, so the rotations need no exchange between threads; a
// warp takes LPW consecutive heads of one batch row (LPW chosen per shape so
// that there are enough warps to fill the GPU).  Matrix scan: eight threads
// per lane, thread j owning column j of P_t, four lanes per warp.  In both,
// each stage of TS steps arrives by tiled TMA loads into a per-warp ring, and
// the whole warp first turns the stage's angles into cosines and sines (from
// the half-angle tangent, so that the rotations carry no systematic norm
// error), which the recurrence threads then read.
#include "mgs_tiles.cuh"

namespace mgs {
namespace {

constexpr int GK = 8;                  // coordinates per head
constexpr int GN = GK * (GK - 1) / 2;  // angles per head and step
constexpr int kItems = 64;             // (lane, step) items per affine-scan stage
constexpr int kGasNS = 3;              // affine-scan stages in flight
constexpr int kGmsLanes = 4;           // heads per warp in the matrix scan
constexpr int kGmsFwdTS = 16, kGmsFwdNS = 3;
constexpr int kGmsBwdTS = 8, kGmsBwdNS = 2;

// Index of the first angle of layer l (0-based): layers alternate 4 and 3 pairs.
__host__ __device__ constexpr int layer_base(int l) { return (l / 2) * 7 + (l % 2) * 4; }
__host__ __device__ constexpr int layer_pairs(int l) { return (l % 2) ? 3 : 4; }

// (x, y) <- (c x - s y, s x + c y)
__device__ __forceinline__ void rot_fwd(float &x, float &y, float c, float s) {
    const float nx = fmaf(c, x, -s * y);
    y = fmaf(s, x, c * y);
    x = nx;
}
// transposed rotation: (x, y) <- (c x + s y, -s x + c y)
__device__ __forceinline__ void rot_bwd(float &x, float &y, float c, float s) {
    const float nx = fmaf(c, x, s * y);
    y = fmaf(-s, x, c * y);
    x = nx;
}

template <int N>
__device__ __forceinline__ void lds_vec(const float *p, float (&r)[N]) {
#pragma unroll
    for (int c = 0; c < N / 4; ++c) {
        const float4 q = reinterpret_cast<const float4 *>(p)[c];
        r[4 * c] = q.x;
        r[4 * c + 1] = q.y;
        r[4 * c + 2] = q.z;
        r[4 * c + 3] = q.w;
    }
}

template <int N>
__device__ __forceinline__ void stg_vec_cs(float *p, const float (&r)[N]) {
#pragma unroll
    for (int c = 0; c < N / 4; ++c) st_cs4(p + 4 * c, make_float4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]));
}

// h <- G h, layer 1 first (cs: cosines, sn: sines in angle order).
__device__ __forceinline__ void mesh_apply(float (&x)[GK], const float (&cs)[GN], const float (&sn)[GN]) {
#pragma unroll
    for (int l = 0; l < GK; ++l)
#pragma unroll
        for (int q = 0; q < layer_pairs(l); ++q) {
            const int p = (l & 1) + 2 * q, n = layer_base(l) + q;
            rot_fwd(x[p], x[p + 1], cs[n], sn[n]);
        }
}

// cos and sin of an angle as rational functions of the half-angle tangent
// t = tan(theta/2): c = (1 - t^2) / (1 + t^2), s = 2t / (1 + t^2), every step
// rounded to nearest.  What this buys is zero-mean rounding in c^2 + s^2 - 1.
// sincosf itself is accurate to about an ulp, but over uniform angles its
// pairs carry c^2 + s^2 - 1 = +1.8e-8 on average (measured on this GPU); a
// product of T = 1024 steps of 28 rotations compounds that bias into a 4e-5
// relative growth of the state, four times the parity tolerance.  The ratio
// t = sin/cos of the half angle cancels any common scale error of sincosf,
// and its angle error has no measurable mean.
__device__ __forceinline__ void unbiased_cos_sin(float theta, float &c, float &s) {
    float sh, ch;
    sincosf(0.5f * theta, &sh, &ch);
    const float t = __fdiv_rn(sh, ch);
    if (fabsf(t) > 1e18f) {  // half angle at a pole of tan: theta = pi (mod 2 pi)
        c = -1.f;
        s = 0.f;
        return;
    }
    const float r = __frcp_rn(fmaf(t, t, 1.f));
    c = fmaf(-t, t, 1.f) * r;
    s = (2.f * t) * r;
}

// The n angles at th (n a multiple of 4, 16-byte aligned) -> cosines in place
// and sines to sn; the whole warp shares the work.
__device__ __forceinline__ void stage_sincos(float *th, float *sn, int n, int lane) {
    for (int i = 4 * lane; i < n; i += 128) {
        const float4 t = *reinterpret_cast<const float4 *>(th + i);
        float4 c, s;
        unbiased_cos_sin(t.x, c.x, s.x);
        unbiased_cos_sin(t.y, c.y, s.y);
        unbiased_cos_sin(t.z, c.z, s.z);
        unbiased_cos_sin(t.w, c.w, s.w);
        *reinterpret_cast<float4 *>(th + i) = c;
        *reinterpret_cast<float4 *>(sn + i) = s;
    }
}

// 3-D map over [rows][H][E] floats, boxes of E x lanes x ts.
cudaError_t make_head_map(CUtensorMap *m, const float *base, int64_t rows, int64_t H, int E, int lanes,
                          int ts) {
    const uint64_t dims[3] = {uint64_t(E), uint64_t(H), uint64_t(rows)};
    const uint64_t str[2] = {uint64_t(E) * 4u, uint64_t(H) * E * 4u};
    const uint32_t box[3] = {uint32_t(E), uint32_t(lanes), uint32_t(ts)};
    return make_tmap(m, base, 3, dims, str, box);
}

// Per-warp shared memory of the affine scan: kGasNS stages of
// [theta ts*lpw*GN][vector inputs nv x ts*lpw*GK], a sine scratch of
// ts*lpw*GN floats, then the barriers.
struct GasSmem {
    int th_f, vec_f, stage_f, ring_f, sin_f;
    __host__ __device__ GasSmem(int lpw, int ts, int nv) {
        th_f = ts * lpw * GN;
        vec_f = ts * lpw * GK;
        stage_f = int(align_up(size_t(th_f + nv * vec_f), 32));
        ring_f = kGasNS * stage_f;
        sin_f = th_f;
    }
    __host__ __device__ size_t bytes() const { return size_t(ring_f + sin_f) * 4 + kGasNS * sizeof(uint64_t); }
};

// ---------------------------------------------------------------- affine forward
__global__ void __launch_bounds__(32)
    gas_fwd_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const float *__restrict__ h0, float *__restrict__ h,
                   int64_t B, int64_t T, int64_t H, int64_t groups_per_b, int lpw, int ts, int has_a,
                   DevCtl ctl) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const GasSmem L(lpw, ts, has_a ? 2 : 1);
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    float *sn = ring + L.ring_f;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sn + L.sin_f);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * lpw;
    const int nl = int(min64(lpw, H - head0));
    const int64_t nblk = (T + ts - 1) / ts;
    const int row0 = int(bi * T);
    const int b_off = L.th_f + (has_a ? L.vec_f : 0);
    const uint32_t stage_tx = uint32_t(L.th_f + (has_a ? 2 : 1) * L.vec_f) * 4u;

    WarpRing<kGasNS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmTh);
        prefetch_tmap(&tmB);
        if (has_a) prefetch_tmap(&tmA);
    }
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L.stage_f;
        const int r = row0 + int(j * ts);
        mbar_arrive_expect_tx(&bars[s], stage_tx);
        tma_load_3d(st, &tmTh, 0, head0, r, &bars[s], pol);
        if (has_a) tma_load_3d(st + L.th_f, &tmA, 0, head0, r, &bars[s], pol);
        tma_load_3d(st + b_off, &tmB, 0, head0, r, &bars[s], pol);
    };
    const int npro = int(min64(kGasNS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    const bool active = lane < nl;
    float x[GK];
    if (active && h0 != nullptr) {
        lds_vec<GK>(h0 + (bi * H + head0 + lane) * GK, x);  // 16-byte aligned global loads
    } else {
#pragma unroll
        for (int i = 0; i < GK; ++i) x[i] = 0.f;
    }
    float *hp = h + ((bi * T) * H + head0 + lane) * GK;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % kGasNS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(ts, T - j * ts));
        float *st = ring + size_t(s) * L.stage_f;
        stage_sincos(st, sn, n * lpw * GN, lane);
        __syncwarp();
        if (active) {
            for (int u = 0; u < n; ++u) {
                const int item = u * lpw + lane;
                float cs[GN], sv[GN], bv[GK];
                lds_vec<GN>(st + item * GN, cs);
                lds_vec<GN>(sn + item * GN, sv);
                lds_vec<GK>(st + b_off + item * GK, bv);
                if (has_a) {
                    float av[GK];
                    lds_vec<GK>(st + L.th_f + item * GK, av);
#pragma unroll
                    for (int i = 0; i < GK; ++i) x[i] *= av[i];
                }
                mesh_apply(x, cs, sv);
#pragma unroll
                for (int i = 0; i < GK; ++i) x[i] += bv[i];
                stg_vec_cs<GK>(hp, x);
                hp += H * GK;
            }
        }
        __syncwarp();
        if (j + kGasNS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + kGasNS);
            }
            rg.armed(s);
        }
    }
}

// ---------------------------------------------------------------- affine backward
// Walks t downwards.  Per step and lane:
//   lambda = g_t + carry,  db_t = lambda,
//   x = a_t * h_{t-1} rotated layer by layer (each layer's output kept),
//   mu = lambda taken back through the layers (transposed rotations), giving
//   every angle's gradient on the way,
//   da_t = mu_0 * h_{t-1},  carry = a_t * mu_0 (= A_t^T lambda_t);
// dh0 = the last carry.
__global__ void __launch_bounds__(32)
    gas_bwd_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmH,
                   const float *__restrict__ h0, float *__restrict__ dth, float *__restrict__ da,
                   float *__restrict__ db, float *__restrict__ dh0, int64_t B, int64_t T, int64_t H,
                   int64_t groups_per_b, int lpw, int ts, int has_a, DevCtl ctl) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int nv = has_a ? 3 : 2;  // a, g, h_{t-1}
    const GasSmem L(lpw, ts, nv);
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    float *sn = ring + L.ring_f;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sn + L.sin_f);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * lpw;
    const int nl = int(min64(lpw, H - head0));
    const int64_t nblk = (T + ts - 1) / ts;
    const int g_off = L.th_f + (has_a ? L.vec_f : 0), h_off = g_off + L.vec_f;
    const uint32_t stage_tx = uint32_t(L.th_f + nv * L.vec_f) * 4u;

    WarpRing<kGasNS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmTh);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmH);
        if (has_a) prefetch_tmap(&tmA);
    }
    // Block j covers in-batch rows T-(j+1)*ts .. T-1-j*ts (rows below 0 are
    // skipped); the h box starts one row earlier and holds h_{t-1}.
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L.stage_f;
        const int r = int(bi * T + T - (j + 1) * ts);
        mbar_arrive_expect_tx(&bars[s], stage_tx);
        tma_load_3d(st, &tmTh, 0, head0, r, &bars[s], pol);
        if (has_a) tma_load_3d(st + L.th_f, &tmA, 0, head0, r, &bars[s], pol);
        tma_load_3d(st + g_off, &tmG, 0, head0, r, &bars[s], pol);
        tma_load_3d(st + h_off, &tmH, 0, head0, r - 1, &bars[s], pol);
    };
    const int npro = int(min64(kGasNS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    const bool active = lane < nl;
    float h0v[GK], carry[GK];
#pragma unroll
    for (int i = 0; i < GK; ++i) {
        h0v[i] = 0.f;
        carry[i] = 0.f;
    }
    if (active && h0 != nullptr) lds_vec<GK>(h0 + (bi * H + head0 + lane) * GK, h0v);

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % kGasNS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tb = T - (j + 1) * ts;       // in-batch row of box row 0
        const int u0 = int(tb < 0 ? -tb : 0);      // first valid box row
        float *st = ring + size_t(s) * L.stage_f;
        stage_sincos(st + u0 * lpw * GN, sn + u0 * lpw * GN, (ts - u0) * lpw * GN, lane);
        __syncwarp();
        if (active) {
            for (int u = ts - 1; u >= u0; --u) {
                const int64_t t = tb + u;
                const int item = u * lpw + lane;
                float cs[GN], sv[GN], lam[GK], hp[GK];
                lds_vec<GN>(st + item * GN, cs);
                lds_vec<GN>(sn + item * GN, sv);
                lds_vec<GK>(st + g_off + item * GK, lam);
                if (t >= 1) {
                    lds_vec<GK>(st + h_off + item * GK, hp);
                } else {
#pragma unroll
                    for (int i = 0; i < GK; ++i) hp[i] = h0v[i];
                }
#pragma unroll
                for (int i = 0; i < GK; ++i) lam[i] += carry[i];
                const int64_t o = ((bi * T + t) * H + head0 + lane);
                stg_vec_cs<GK>(db + o * GK, lam);
                float av[GK];
                if (has_a) {
                    lds_vec<GK>(st + L.th_f + item * GK, av);
                } else {
#pragma unroll
                    for (int i = 0; i < GK; ++i) av[i] = 1.f;
                }
                // forward through the mesh, keeping every layer's output
                float xl[GK][GK];
#pragma unroll
                for (int i = 0; i < GK; ++i) xl[0][i] = av[i] * hp[i];
#pragma unroll
                for (int l = 0; l < GK; ++l) {
                    if (l > 0) {
#pragma unroll
                        for (int i = 0; i < GK; ++i) xl[l][i] = xl[l - 1][i];
                    }
#pragma unroll
                    for (int q = 0; q < layer_pairs(l); ++q) {
                        const int p = (l & 1) + 2 * q, n = layer_base(l) + q;
                        rot_fwd(xl[l][p], xl[l][p + 1], cs[n], sv[n]);
                    }
                }
                // adjoint back through the layers
                float dthv[GN];
#pragma unroll
                for (int l = GK - 1; l >= 0; --l) {
#pragma unroll
                    for (int q = 0; q < layer_pairs(l); ++q) {
                        const int p = (l & 1) + 2 * q, n = layer_base(l) + q;
                        dthv[n] = fmaf(lam[p + 1], xl[l][p], -lam[p] * xl[l][p + 1]);
                        rot_bwd(lam[p], lam[p + 1], cs[n], sv[n]);
                    }
                }
                stg_vec_cs<GN>(dth + o * GN, dthv);
                if (da != nullptr) {
                    float dav[GK];
#pragma unroll
                    for (int i = 0; i < GK; ++i) dav[i] = lam[i] * hp[i];
                    stg_vec_cs<GK>(da + o * GK, dav);
                }
#pragma unroll
                for (int i = 0; i < GK; ++i) carry[i] = av[i] * lam[i];
            }
        }
        __syncwarp();
        if (j + kGasNS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + kGasNS);
            }
            rg.armed(s);
        }
    }
    if (active && dh0 != nullptr) {
        float *p = dh0 + (bi * H + head0 + lane) * GK;
        *reinterpret_cast<float4 *>(p) = make_float4(carry[0], carry[1], carry[2], carry[3]);
        *reinterpret_cast<float4 *>(p + 4) = make_float4(carry[4], carry[5], carry[6], carry[7]);
    }
}

// ---------------------------------------------------------------- matrix forward
// Thread j of a lane's 8-thread group carries column j of P_t.
__global__ void __launch_bounds__(32)
    gms_fwd_kernel(const __grid_constant__ CUtensorMap tmTh, float *__restrict__ P, int64_t B, int64_t T,
                   int64_t H, int64_t groups_per_b, DevCtl ctl) {
    constexpr int TS = kGmsFwdTS, NS = kGmsFwdNS;
    constexpr int STAGEF = TS * kGmsLanes * GN;  // one theta box (a multiple of 32 floats)
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    float *sn = ring + NS * STAGEF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sn + STAGEF);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * kGmsLanes;
    const int sub = lane >> 3, col = lane & 7;
    const bool active = head0 + sub < H;
    const int64_t nblk = (T + TS - 1) / TS;
    const int row0 = int(bi * T);

    WarpRing<NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) prefetch_tmap(&tmTh);
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        mbar_arrive_expect_tx(&bars[s], uint32_t(STAGEF * 4));
        tma_load_3d(ring + size_t(s) * STAGEF, &tmTh, 0, head0, row0 + int(j * TS), &bars[s], pol);
    };
    const int npro = int(min64(NS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float v[GK];
#pragma unroll
    for (int i = 0; i < GK; ++i) v[i] = (i == col) ? 1.f : 0.f;
    float *pp = P + ((bi * T) * H + head0 + sub) * (GK * GK) + col;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int n = int(min64(TS, T - j * TS));
        float *st = ring + size_t(s) * STAGEF;
        stage_sincos(st, sn, n * kGmsLanes * GN, lane);
        __syncwarp();
        for (int u = 0; u < n; ++u) {
            const int item = u * kGmsLanes + sub;
            float cs[GN], sv[GN];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(sn + item * GN, sv);
            mesh_apply(v, cs, sv);
            if (active) {
#pragma unroll
                for (int i = 0; i < GK; ++i) st_cs(pp + i * GK, v[i]);
            }
            pp += H * GK * GK;
        }
        __syncwarp();
        if (j + NS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + NS);
            }
            rg.armed(s);
        }
    }
}

// ---------------------------------------------------------------- matrix backward
// Per step and column j (t downwards): Lambda = G_t[:, j] + carry; x = P_t[:, j];
// both go back through the layers by transposed rotations (x recovers the
// column before each layer, exact up to rounding since the mesh is
// orthogonal), each thread adding its column's share of every angle's
// gradient; the eight shares are summed by a butterfly reduce-scatter that
// leaves angles 4j .. 4j+3 with thread j.  carry = A_t^T Lambda[:, j].
__global__ void __launch_bounds__(32)
    gms_bwd_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmP,
                   const __grid_constant__ CUtensorMap tmG, float *__restrict__ dth, int64_t B, int64_t T,
                   int64_t H, int64_t groups_per_b, DevCtl ctl) {
    constexpr int TS = kGmsBwdTS, NS = kGmsBwdNS;
    using TM = MatTile<GK, true>;  // swizzled: conflict-free column reads
    constexpr int MATF = TS * TM::MF, THF = TS * kGmsLanes * GN;
    constexpr int STAGEF = int(align_up(size_t(2 * MATF + THF), TM::kAlign / 4));
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    unsigned char *sbase = align_smem(smem_raw, TM::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    float *sn = ring + NS * STAGEF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sn + THF);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * kGmsLanes;
    const int sub = lane >> 3, col = lane & 7;
    const bool active = head0 + sub < H;
    const int64_t nblk = (T + TS - 1) / TS;

    WarpRing<NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        prefetch_tmap(&tmTh);
        prefetch_tmap(&tmP);
        prefetch_tmap(&tmG);
    }
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * STAGEF;
        const int r = int(bi * T + T - (j + 1) * TS);
        mbar_arrive_expect_tx(&bars[s], uint32_t((2 * MATF + THF) * 4));
        TM::load(st, &tmP, head0, r, &bars[s], pol);
        TM::load(st + MATF, &tmG, head0, r, &bars[s], pol);
        tma_load_3d(st + 2 * MATF, &tmTh, 0, head0, r, &bars[s], pol);
    };
    const int npro = int(min64(NS, nblk));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float carry[GK];
#pragma unroll
    for (int i = 0; i < GK; ++i) carry[i] = 0.f;

    for (int64_t j = 0; j < nblk; ++j) {
        const int s = int(j % NS);
        if (!rg.wait(s, ctl)) {
            if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
            rg.drain(ctl, lane);
            return;
        }
        const int64_t tb = T - (j + 1) * TS;
        const int u0 = int(tb < 0 ? -tb : 0);
        float *st = ring + size_t(s) * STAGEF;
        float *sth = st + 2 * MATF;
        stage_sincos(sth + u0 * kGmsLanes * GN, sn + u0 * kGmsLanes * GN, (TS - u0) * kGmsLanes * GN, lane);
        __syncwarp();
        for (int u = TS - 1; u >= u0; --u) {
            const int64_t t = tb + u;
            const TileRef<GK, true> Pt{st, u, sub}, Gt{st + MATF, u, sub};
            const int item = u * kGmsLanes + sub;
            float cs[GN], sv[GN], lam[GK], x[GK];
            lds_vec<GN>(sth + item * GN, cs);
            lds_vec<GN>(sn + item * GN, sv);
#pragma unroll
            for (int i = 0; i < GK; ++i) {
                lam[i] = Gt.at(i, col) + carry[i];
                x[i] = Pt.at(i, col);
            }
            float d[32];
#pragma unroll
            for (int l = GK - 1; l >= 0; --l) {
#pragma unroll
                for (int q = 0; q < layer_pairs(l); ++q) {
                    const int p = (l & 1) + 2 * q, n = layer_base(l) + q;
                    d[n] = fmaf(lam[p + 1], x[p], -lam[p] * x[p + 1]);
                    rot_bwd(x[p], x[p + 1], cs[n], sv[n]);
                    rot_bwd(lam[p], lam[p + 1], cs[n], sv[n]);
                }
            }
#pragma unroll
            for (int n = GN; n < 32; ++n) d[n] = 0.f;
            // butterfly reduce-scatter over the 8 columns: 32 -> 4 values
#pragma unroll
            for (int o = 4, half = 16; o >= 1; o >>= 1, half >>= 1) {
                const bool up = (col & o) != 0;
#pragma unroll
                for (int c = 0; c < half; ++c) {
                    const float send = up ? d[c] : d[c + half];
                    const float keep = up ? d[c + half] : d[c];
                    d[c] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (active && col < GN / 4)
                st_cs4(dth + ((bi * T + t) * H + head0 + sub) * GN + 4 * col, make_float4(d[0], d[1], d[2], d[3]));
#pragma unroll
            for (int i = 0; i < GK; ++i) carry[i] = lam[i];
        }
        __syncwarp();
        if (j + NS < nblk) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + NS);
            }
            rg.armed(s);
        }
    }
}

// Lanes per warp for the affine scan: the fewest (each lane is one thread)
// that still gives about one warp per SM sub-partition or fewer, capped by
// the heads of one batch row.
int gas_lanes_per_warp(int64_t B, int64_t H) {
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (B * H + 4 * sms - 1) / (4 * int64_t(sms));
    int lpw = 1;
    while (lpw < want && lpw < 32) lpw *= 2;
    while (lpw > 1 && lpw / 2 >= H) lpw /= 2;
    return lpw;
}

}  // namespace

cudaError_t launch_gas_fwd(const float *theta, const float *a, const float *b, const float *h0, float *h,
                           int64_t B, int64_t T, int64_t H, const DevCtl &ctl, cudaStream_t s) {
    const int lpw = gas_lanes_per_warp(B, H), ts = kItems / lpw;
    const int64_t rows = B * T;
    CUtensorMap tTh, tA, tB;
    cudaError_t e;
    if ((e = make_head_map(&tTh, theta, rows, H, GN, lpw, ts)) != cudaSuccess) return e;
    if ((e = make_head_map(&tB, b, rows, H, GK, lpw, ts)) != cudaSuccess) return e;
    if (a != nullptr) {
        if ((e = make_head_map(&tA, a, rows, H, GK, lpw, ts)) != cudaSuccess) return e;
    } else {
        tA = tB;
    }
    const int64_t gpb = (H + lpw - 1) / lpw, blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(GasSmem(lpw, ts, a ? 2 : 1).bytes());
    if ((e = ensure_smem_attr((const void *)gas_fwd_kernel, smem)) != cudaSuccess) return e;
    gas_fwd_kernel<<<dim3(unsigned(blocks)), 32, smem, s>>>(tTh, tA, tB, h0, h, B, T, H, gpb, lpw, ts,
                                                            a != nullptr, ctl);
    return cudaGetLastError();
}

cudaError_t launch_gas_bwd(const float *theta, const float *a, const float *h0, const float *h, const float *gh,
                           float *dth, float *da, float *db, float *dh0, int64_t B, int64_t T, int64_t H,
                           const DevCtl &ctl, cudaStream_t s) {
    const int lpw = gas_lanes_per_warp(B, H), ts = kItems / lpw;
    const int64_t rows = B * T;
    CUtensorMap tTh, tA, tG, tH;
    cudaError_t e;
    if ((e = make_head_map(&tTh, theta, rows, H, GN, lpw, ts)) != cudaSuccess) return e;
    if ((e = make_head_map(&tG, gh, rows, H, GK, lpw, ts)) != cudaSuccess) return e;
    if ((e = make_head_map(&tH, h, rows, H, GK, lpw, ts)) != cudaSuccess) return e;
    if (a != nullptr) {
        if ((e = make_head_map(&tA, a, rows, H, GK, lpw, ts)) != cudaSuccess) return e;
    } else {
        tA = tG;
    }
    const int64_t gpb = (H + lpw - 1) / lpw, blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(GasSmem(lpw, ts, a ? 3 : 2).bytes());
    if ((e = ensure_smem_attr((const void *)gas_bwd_kernel, smem)) != cudaSuccess) return e;
    gas_bwd_kernel<<<dim3(unsigned(blocks)), 32, smem, s>>>(tTh, tA, tG, tH, h0, dth, da, db, dh0, B, T, H, gpb,
                                                            lpw, ts, a != nullptr, ctl);
    return cudaGetLastError();
}

cudaError_t launch_gms_fwd(const float *theta, float *P, int64_t B, int64_t T, int64_t H, const DevCtl &ctl,
                           cudaStream_t s) {
    CUtensorMap tTh;
    cudaError_t e;
    if ((e = make_head_map(&tTh, theta, B * T, H, GN, kGmsLanes, kGmsFwdTS)) != cudaSuccess) return e;
    const int64_t gpb = (H + kGmsLanes - 1) / kGmsLanes, blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    constexpr int STAGEF = kGmsFwdTS * kGmsLanes * GN;
    const int smem = int((kGmsFwdNS + 1) * STAGEF * 4 + kGmsFwdNS * sizeof(uint64_t));
    if ((e = ensure_smem_attr((const void *)gms_fwd_kernel, smem)) != cudaSuccess) return e;
    gms_fwd_kernel<<<dim3(unsigned(blocks)), 32, smem, s>>>(tTh, P, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

cudaError_t launch_gms_bwd(const float *theta, const float *P, const float *G, float *dth, int64_t B, int64_t T,
                           int64_t H, const DevCtl &ctl, cudaStream_t s) {
    using TM = MatTile<GK, true>;
    CUtensorMap tTh, tP, tG;
    cudaError_t e;
    if ((e = make_head_map(&tTh, theta, B * T, H, GN, kGmsLanes, kGmsBwdTS)) != cudaSuccess) return e;
    if ((e = TM::make(&tP, P, B * T, H, kGmsBwdTS)) != cudaSuccess) return e;
    if ((e = TM::make(&tG, G, B * T, H, kGmsBwdTS)) != cudaSuccess) return e;
    const int64_t gpb = (H + kGmsLanes - 1) / kGmsLanes, blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    constexpr int MATF = kGmsBwdTS * TM::MF, THF = kGmsBwdTS * kGmsLanes * GN;
    constexpr int STAGEF = int(align_up(size_t(2 * MATF + THF), TM::kAlign / 4));
    const int smem = int(size_t(kGmsBwdNS * STAGEF + THF) * 4 + kGmsBwdNS * sizeof(uint64_t) + TM::kAlign);
    if ((e = ensure_smem_attr((const void *)gms_bwd_kernel, smem)) != cudaSuccess) return e;
    gms_bwd_kernel<<<dim3(unsigned(blocks)), 32, smem, s>>>(tTh, tP, tG, dth, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

}  // namespace mgs
