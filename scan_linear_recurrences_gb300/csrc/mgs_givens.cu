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
// Mapping.  Each block is one recurrence warp and three angle warps.  The
// angles cost far more than the rotations (28 cosine/sine pairs per lane and
// step against 112 multiply-adds), but they do not depend on the state, so
// the angle warps convert stage j+1's angles (to cosines and sines, from the
// half-angle tangent so that the rotations carry no systematic norm error)
// while the recurrence warp runs stage j.  Affine scan: one thread of the
// recurrence warp per (batch, head) lane holds the whole state in registers,
// so the rotations need no exchange between threads; a block takes LPW
// consecutive heads of one batch row (LPW chosen per shape so that there are
// enough blocks to fill the GPU).  Matrix scan: eight threads per lane,
// thread j owning column j of P_t, four lanes per block.  Each stage of TS
// steps arrives by tiled TMA loads into a per-block ring.
#include "mgs_chunk.cuh"
#include "mgs_ffsincos.cuh"

namespace mgs {
namespace {

constexpr int GK = 8;                  // coordinates per head
constexpr int GN = GK * (GK - 1) / 2;  // angles per head and step
constexpr int kItems = 64;             // (lane, step) items per affine-scan stage
constexpr int kNS = 3;                 // stages in flight
// Threads per block of the fused kernels: one recurrence warp and the angle
// warps, three in the forward kernels and four in the backward ones, whose
// angle warps also run the affine scan's forward pass through the layers
// (measured at the lab shape: affine backward 31.0 -> 24.8 us with the fourth
// warp; the forward kernels gain nothing from a fourth or fifth).
constexpr int kBlockF = 128, kBlockB = 160;
constexpr int kProdF = kBlockF - 32, kProdB = kBlockB - 32;  // angle threads
constexpr int kGasMaxLanes = 8;        // affine-scan lanes per recurrence warp, at most
constexpr int kGmsLanes = 4;           // heads per block in the matrix scan (8 threads each)
constexpr int kGmsFwdTS = 16, kGmsBwdTS = 8;

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
// 1/x for normal positive x below 2^126: the hardware approximation refined
// by one Newton-Raphson step, r1 = r0 + r0 (1 - x r0) with the residual taken
// by a fused multiply-add, which leaves only the final rounding (to nearest).
__device__ __forceinline__ float recip_nr(float x) {
    float r0;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(x));
    return fmaf(r0, fmaf(-x, r0, 1.f), r0);
}

// kFast: the half angle's sine and cosine from the hardware approximation
// (__sincosf, absolute error about 2^-21 on [-pi, pi]) instead of sincosf.
// The construction keeps c^2 + s^2 - 1 unbiased either way; what the faster
// form adds is an angle error near 1e-6 rad.  The gated affine scan contracts
// it (|a| < 1), so it takes kFast; the matrix scans, a product of T orthogonal
// meshes with nothing to contract the errors, keep sincosf.
template <bool kFast = false>
__device__ __forceinline__ void unbiased_cos_sin(float theta, float &c, float &s) {
    float sh, ch;
    if constexpr (kFast)
        __sincosf(0.5f * theta, &sh, &ch);
    else
        sincosf(0.5f * theta, &sh, &ch);
    // |cos| of the half angle: at least 2^-100 away from a pole (theta = pi
    // mod 2 pi gives |t| <= 1e30, where c = -1 and s = 0 to fp32 precision)
    const float ach = fmaxf(fabsf(ch), 1e-30f);
    const float t = fminf(fmaxf(copysignf(sh * recip_nr(ach), sh * ch), -1e18f), 1e18f);
    const float r = recip_nr(fmaf(t, t, 1.f));
    c = fmaf(-t, t, 1.f) * r;
    s = (2.f * t) * r;
}

// Angles [lo, hi) of a stage converted by the block's NP angle threads
// (pt = 0 .. NP-1): cosines in place, sines to sn; consecutive threads take
// consecutive words.
// Four angles per thread and round are independent chains, which the
// scheduler interleaves (one chain alone is a long run of dependent ops).
template <int NP, bool kFast = false>
__device__ __forceinline__ void angle_range(float *th, float *sn, int lo, int hi, int pt) {
    constexpr int kProd = NP;
    int i = lo + pt;
    for (; i + 3 * kProd < hi; i += 4 * kProd) {
        float x[4], c[4], s[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) x[q] = th[i + q * kProd];
#pragma unroll
        for (int q = 0; q < 4; ++q) unbiased_cos_sin<kFast>(x[q], c[q], s[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            th[i + q * kProd] = c[q];
            sn[i + q * kProd] = s[q];
        }
    }
    for (; i < hi; i += kProd) {
        float c, s;
        unbiased_cos_sin<kFast>(th[i], c, s);
        th[i] = c;
        sn[i] = s;
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

// Block pipeline shared by the four kernels.  A block is one recurrence warp
// (warp 0) and three angle warps.  Iteration `it` of the main loop:
//   angle warps: wait for stage it's bulk copies, convert its angles;
//   warp 0:      run the recurrence over stage it-1 (converted last time);
//   all:         __syncthreads; then stage it-1's slot is refilled with the
//                block kNS ahead.
// The angle warps own the ring's barriers: only they wait on the copies, and
// the block barrier hands the landed (and converted) data on to warp 0.  A
// wait that gives up sets the block's abort word, so every thread leaves at
// the same barrier, after the angle warps have drained the copies in flight.
struct BlockRing {
    WarpRing<kNS> rg;
    uint64_t *bars;
    int *abort_word;
    __device__ __forceinline__ void init(uint64_t *b, int *ab, int tid) {
        bars = b;
        abort_word = ab;
        if (tid == 0) {
            for (int s = 0; s < kNS; ++s) mbar_init(&bars[s], 1);
            fence_barrier_init();
            *abort_word = 0;
        }
        __syncthreads();
        rg.bar = bars;
        rg.inflight = 0;
        rg.phase = 0;
    }
};

#define MGS_BLOCK_ABORT_CHECK(br, producer, lane)                 \
    if (*(br).abort_word != 0) {                                  \
        if (producer) (br).rg.drain(ctl, lane);                   \
        return;                                                   \
    }

// Per-block shared memory of the affine scan: kNS stages of
// [theta ts*lpw*GN][vector inputs nv x ts*lpw*GK], two sine buffers of
// ts*lpw*GN floats, in the backward two buffers of rotated pairs of
// 2*ts*lpw*GN floats, the barriers and the abort word.
// The backward adds two buffers of the rotated-state pairs (xp_f floats each).
// In the exact-orthogonal mode (no gate, see below) two more buffers of
// ts*lpw*GN floats per stage parity hold the low parts of the cosines and
// sines, and the table of cos_sin_ff sits in front of the barriers.
struct GasSmem {
    int th_f, vec_f, stage_f, ring_f, sin_f, xp_f, lo_f, tab_f;
    __host__ __device__ GasSmem(int lpw, int ts, int nv, bool with_xp = false, bool xo = false) {
        th_f = ts * lpw * GN;
        vec_f = ts * lpw * GK;
        stage_f = int(align_up(size_t(th_f + nv * vec_f), 32));
        ring_f = kNS * stage_f;
        sin_f = th_f;
        xp_f = with_xp ? 2 * th_f : 0;
        lo_f = xo ? 2 * th_f : 0;
        tab_f = xo ? 4 * SinCosTable::kEntries : 0;
    }
    __host__ __device__ size_t bytes() const {
        return size_t(ring_f + 2 * sin_f + 2 * xp_f + 2 * lo_f + tab_f) * 4 + kNS * sizeof(uint64_t) + 16;
    }
};

// Exact-orthogonal mode.  Without the gate a the transition G(theta) is
// orthogonal: nothing contracts, the state and the adjoint grow like sqrt(T)
// and the angle gradients like T, so the rounding of fp32 cosines and sines
// (each rotation off by up to half an ulp, 3e-8, in angle) accumulates into
// angle-gradient errors of several 1e-3 at T ~ 500.  There the kernels take
// the cosines and sines as hi + lo pairs from cos_sin_ff (error ~1e-11) and
// carry the recurrence state (forward) and the adjoint (backward) as hi + lo
// pairs, rounding to fp32 only what they store.
template <int NP>
__device__ __forceinline__ void angle_range_ff(float *th, float *sn, float *clo, float *slo, int lo, int hi, int pt,
                                               const float4 *tab) {
    int i = lo + pt;
    for (; i + NP < hi; i += 2 * NP) {
        float c0, c0l, s0, s0l, c1, c1l, s1, s1l;
        cos_sin_ff(th[i], tab, c0, c0l, s0, s0l);
        cos_sin_ff(th[i + NP], tab, c1, c1l, s1, s1l);
        th[i] = c0; sn[i] = s0; clo[i] = c0l; slo[i] = s0l;
        th[i + NP] = c1; sn[i + NP] = s1; clo[i + NP] = c1l; slo[i + NP] = s1l;
    }
    for (; i < hi; i += NP) {
        float c, cl, sv, sl;
        cos_sin_ff(th[i], tab, c, cl, sv, sl);
        th[i] = c; sn[i] = sv; clo[i] = cl; slo[i] = sl;
    }
}

// Copies the cos_sin_ff table from the kernel parameters into shared memory
// (indexed reads of parameter space serialise across a warp).
__device__ __forceinline__ void load_table(float4 *dst, const SinCosTable &tab, int tid, int nthreads) {
    for (int i = tid; i < SinCosTable::kEntries; i += nthreads) dst[i] = tab.e[i];
}

// ---------------------------------------------------------------- affine forward
// XO: the exact-orthogonal mode (has_a must be 0), see angle_range_ff.
template <bool XO>
__global__ void __launch_bounds__(kBlockF)
    gas_fwd_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const float *__restrict__ h0, float *__restrict__ h,
                   int64_t B, int64_t T, int64_t H, int64_t groups_per_b, int lpw, int ts, int has_a,
                   const __grid_constant__ SinCosTable tab, DevCtl ctl) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const GasSmem L(lpw, ts, has_a ? 2 : 1, false, XO);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp != 0;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    float *snb = ring + L.ring_f;  // two sine buffers
    float *lob = snb + 2 * L.sin_f;  // XO: two buffers of (cosine lo, sine lo)
    float4 *tabs = reinterpret_cast<float4 *>(lob + 2 * L.lo_f);
    uint64_t *bars = reinterpret_cast<uint64_t *>(tabs + (XO ? SinCosTable::kEntries : 0));
    if constexpr (XO) load_table(tabs, tab, tid, kBlockF);
    BlockRing br;
    br.init(bars, reinterpret_cast<int *>(bars + kNS), tid);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * lpw;
    const int nl = int(min64(lpw, H - head0));
    const int64_t nblk = (T + ts - 1) / ts;
    const int row0 = int(bi * T);
    const int b_off = L.th_f + (has_a ? L.vec_f : 0);
    const uint32_t stage_tx = uint32_t(L.th_f + (has_a ? 2 : 1) * L.vec_f) * 4u;
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {  // thread kBlockF-1 only
        float *st = ring + size_t(s) * L.stage_f;
        const int r = row0 + int(j * ts);
        mbar_arrive_expect_tx(&bars[s], stage_tx);
        tma_load_3d(st, &tmTh, 0, head0, r, &bars[s], pol);
        if (has_a) tma_load_3d(st + L.th_f, &tmA, 0, head0, r, &bars[s], pol);
        tma_load_3d(st + b_off, &tmB, 0, head0, r, &bars[s], pol);
    };
    const int npro = int(min64(kNS, nblk));
    if (tid == kBlockF - 1) {
        prefetch_tmap(&tmTh);
        prefetch_tmap(&tmB);
        if (has_a) prefetch_tmap(&tmA);
        for (int s = 0; s < npro; ++s) issue(s, s);
    }
    if (producer)
        for (int s = 0; s < npro; ++s) br.rg.armed(s);

    const bool active = !producer && lane < nl;
    float x[GK], xl[GK];  // state (XO: hi parts; xl the lo parts)
    if (active && h0 != nullptr) {
        lds_vec<GK>(h0 + (bi * H + head0 + lane) * GK, x);  // 16-byte aligned global loads
    } else {
#pragma unroll
        for (int i = 0; i < GK; ++i) x[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < GK; ++i) xl[i] = 0.f;
    float *hp = h + ((bi * T) * H + head0 + lane) * GK;

    for (int64_t it = 0; it <= nblk; ++it) {
        if (producer && it < nblk) {
            const int s = int(it % kNS);
            if (br.rg.wait(s, ctl)) {
                const int hi = int(min64(ts, T - it * ts)) * lpw * GN;
                if constexpr (XO) {
                    float *lo = lob + (it & 1) * L.lo_f;
                    angle_range_ff<kProdF>(ring + size_t(s) * L.stage_f, snb + (it & 1) * L.sin_f, lo, lo + L.sin_f,
                                           0, hi, tid - 32, tabs);
                } else {
                    angle_range<kProdF, true>(ring + size_t(s) * L.stage_f, snb + (it & 1) * L.sin_f, 0, hi, tid - 32);
                }
            } else {
                if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
                *br.abort_word = 1;
            }
        }
        if (active && it >= 1) {
            const int64_t j = it - 1;
            const float *st = ring + size_t(j % kNS) * L.stage_f;
            const float *sc = snb + (j & 1) * L.sin_f;
            const int n = int(min64(ts, T - j * ts));
            if constexpr (XO) {
                const float *lo = lob + (j & 1) * L.lo_f;
                for (int u = 0; u < n; ++u) {
                    const int item = u * lpw + lane;
                    const float *cp = st + item * GN, *sp = sc + item * GN;
                    const float *clp = lo + item * GN, *slp = lo + L.sin_f + item * GN;
                    float bv[GK];
                    lds_vec<GK>(st + b_off + item * GK, bv);
#pragma unroll
                    for (int l = 0; l < GK; ++l)
#pragma unroll
                        for (int q = 0; q < layer_pairs(l); ++q) {
                            const int p = (l & 1) + 2 * q, nn = layer_base(l) + q;
                            ff_rot_fwd(x[p], xl[p], x[p + 1], xl[p + 1], cp[nn], clp[nn], sp[nn], slp[nn]);
                        }
#pragma unroll
                    for (int i = 0; i < GK; ++i) ff_add(x[i], xl[i], bv[i]);
                    stg_vec_cs<GK>(hp, x);
                    hp += H * GK;
                }
            } else
            for (int u = 0; u < n; ++u) {
                const int item = u * lpw + lane;
                float cs[GN], sv[GN], bv[GK];
                lds_vec<GN>(st + item * GN, cs);
                lds_vec<GN>(sc + item * GN, sv);
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
        __syncthreads();
        MGS_BLOCK_ABORT_CHECK(br, producer, lane);
        if (it >= 1 && it - 1 + kNS < nblk) {
            const int s = int((it - 1) % kNS);
            if (tid == kBlockF - 1) {
                fence_proxy_async_smem();
                issue(s, it - 1 + kNS);
            }
            if (producer) br.rg.armed(s);
        }
    }
}

// ---------------------------------------------------------------- affine backward
// Walks t downwards.  Per step and lane:
//   lambda = g_t + carry,  db_t = lambda,
//   x = a_t * h_{t-1} rotated layer by layer (each rotation's output pair kept),
//   mu = lambda taken back through the layers (transposed rotations), giving
//   every angle's gradient on the way,
//   da_t = mu_0 * h_{t-1},  carry = a_t * mu_0 (= A_t^T lambda_t);
// dh0 = the last carry.  The forward pass through the layers depends only on
// inputs (h_{t-1}, a_t, theta_t), not on the carry, so the angle warps run it
// for the next stage together with its angle conversion and leave the 28
// rotated pairs per step in shared memory; the recurrence warp's chain per
// step is then only the transposed rotations of mu.
// XO: the exact-orthogonal mode (has_a must be 0): cosines and sines as
// hi + lo pairs and the adjoint carried as hi + lo pairs; the forward pass
// through the layers (which only enters the angle gradients, rounded to
// fp32 anyway) uses the hi parts.
template <bool XO>
__global__ void __launch_bounds__(kBlockB)
    gas_bwd_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmH,
                   const float *__restrict__ h0, float *__restrict__ dth, float *__restrict__ da,
                   float *__restrict__ db, float *__restrict__ dh0, int64_t B, int64_t T, int64_t H,
                   int64_t groups_per_b, int lpw, int ts, int has_a, const __grid_constant__ SinCosTable tab,
                   DevCtl ctl) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int nv = has_a ? 3 : 2;  // a, g, h_{t-1}
    const GasSmem L(lpw, ts, nv, true, XO);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp != 0;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    float *snb = ring + L.ring_f;
    float *xpb = snb + 2 * L.sin_f;  // two buffers of rotated pairs, 2 GN floats per item
    float *lob = xpb + 2 * L.xp_f;   // XO: two buffers of (cosine lo, sine lo)
    float4 *tabs = reinterpret_cast<float4 *>(lob + 2 * L.lo_f);
    uint64_t *bars = reinterpret_cast<uint64_t *>(tabs + (XO ? SinCosTable::kEntries : 0));
    if constexpr (XO) load_table(tabs, tab, tid, kBlockB);
    BlockRing br;
    br.init(bars, reinterpret_cast<int *>(bars + kNS), tid);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * lpw;
    const int nl = int(min64(lpw, H - head0));
    const int64_t nblk = (T + ts - 1) / ts;
    const int g_off = L.th_f + (has_a ? L.vec_f : 0), h_off = g_off + L.vec_f;
    const uint32_t stage_tx = uint32_t(L.th_f + nv * L.vec_f) * 4u;
    const uint64_t pol = policy_evict_first();
    const int lpw_log2 = __ffs(lpw) - 1;
    // Block j covers in-batch rows T-(j+1)*ts .. T-1-j*ts (rows below 0 are
    // skipped); the h box starts one row earlier and holds h_{t-1}.
    auto issue = [&](int s, int64_t j) {  // thread kBlockB-1 only
        float *st = ring + size_t(s) * L.stage_f;
        const int r = int(bi * T + T - (j + 1) * ts);
        mbar_arrive_expect_tx(&bars[s], stage_tx);
        tma_load_3d(st, &tmTh, 0, head0, r, &bars[s], pol);
        if (has_a) tma_load_3d(st + L.th_f, &tmA, 0, head0, r, &bars[s], pol);
        tma_load_3d(st + g_off, &tmG, 0, head0, r, &bars[s], pol);
        tma_load_3d(st + h_off, &tmH, 0, head0, r - 1, &bars[s], pol);
    };
    const int npro = int(min64(kNS, nblk));
    if (tid == kBlockB - 1) {
        prefetch_tmap(&tmTh);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmH);
        if (has_a) prefetch_tmap(&tmA);
        for (int s = 0; s < npro; ++s) issue(s, s);
    }
    if (producer)
        for (int s = 0; s < npro; ++s) br.rg.armed(s);
    auto first_row = [&](int64_t j) -> int {  // first valid box row of block j
        const int64_t tb = T - (j + 1) * ts;
        return int(tb < 0 ? -tb : 0);
    };

    const bool active = !producer && lane < nl;
    float h0v[GK], carry[GK], carryl[GK];  // carryl: XO lo parts
#pragma unroll
    for (int i = 0; i < GK; ++i) {
        h0v[i] = 0.f;
        carry[i] = 0.f;
        carryl[i] = 0.f;
    }
    if (active && h0 != nullptr) lds_vec<GK>(h0 + (bi * H + head0 + lane) * GK, h0v);

    for (int64_t it = 0; it <= nblk; ++it) {
        if (producer && it < nblk) {
            const int s = int(it % kNS);
            float *st = ring + size_t(s) * L.stage_f;
            float *sn = snb + (it & 1) * L.sin_f;
            if (br.rg.wait(s, ctl)) {
                if constexpr (XO) {
                    float *lo = lob + (it & 1) * L.lo_f;
                    angle_range_ff<kProdB>(st, sn, lo, lo + L.sin_f, first_row(it) * lpw * GN, ts * lpw * GN,
                                           tid - 32, tabs);
                } else {
                    angle_range<kProdB, true>(st, sn, first_row(it) * lpw * GN, ts * lpw * GN, tid - 32);
                }
            } else {
                if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
                *br.abort_word = 1;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kProdB) : "memory");  // angle warps only
            if (*br.abort_word == 0) {
                // the forward pass through the layers of every step of the
                // stage: x = a_t * h_{t-1}, each rotation's output pair kept
                const int64_t tb = T - (it + 1) * ts;
                float *xp = xpb + (it & 1) * L.xp_f;
                for (int q = first_row(it) * lpw + tid - 32; q < ts * lpw; q += kProdB) {
                    const int u = q >> lpw_log2, l = q & (lpw - 1);  // lpw is a power of two
                    float cs[GN], sv[GN], hv[GK], av[GK];
                    lds_vec<GN>(st + q * GN, cs);
                    lds_vec<GN>(sn + q * GN, sv);
                    if (tb + u >= 1) {
                        lds_vec<GK>(st + h_off + q * GK, hv);
                    } else if (h0 != nullptr && head0 + l < H) {
                        lds_vec<GK>(h0 + (bi * H + head0 + l) * GK, hv);
                    } else {
#pragma unroll
                        for (int i = 0; i < GK; ++i) hv[i] = 0.f;
                    }
                    if (has_a) {
                        lds_vec<GK>(st + L.th_f + q * GK, av);
                    } else {
#pragma unroll
                        for (int i = 0; i < GK; ++i) av[i] = 1.f;
                    }
                    float x[GK], pr[2 * GN];
#pragma unroll
                    for (int i = 0; i < GK; ++i) x[i] = av[i] * hv[i];
#pragma unroll
                    for (int ll = 0; ll < GK; ++ll)
#pragma unroll
                        for (int qq = 0; qq < layer_pairs(ll); ++qq) {
                            const int p = (ll & 1) + 2 * qq, n = layer_base(ll) + qq;
                            rot_fwd(x[p], x[p + 1], cs[n], sv[n]);
                            pr[2 * n] = x[p];
                            pr[2 * n + 1] = x[p + 1];
                        }
#pragma unroll
                    for (int c4 = 0; c4 < 2 * GN; c4 += 4)
                        *reinterpret_cast<float4 *>(xp + q * 2 * GN + c4) =
                            make_float4(pr[c4], pr[c4 + 1], pr[c4 + 2], pr[c4 + 3]);
                }
            }
        }
        if (active && it >= 1) {
            const int64_t j = it - 1;
            const int64_t tb = T - (j + 1) * ts;  // in-batch row of box row 0
            const float *st = ring + size_t(j % kNS) * L.stage_f;
            const float *sc = snb + (j & 1) * L.sin_f;
            const float *xp = xpb + (j & 1) * L.xp_f;
            if constexpr (XO) {
                const float *lo = lob + (j & 1) * L.lo_f;
                for (int u = ts - 1; u >= first_row(j); --u) {
                    const int64_t t = tb + u;
                    const int item = u * lpw + lane;
                    const float *cp = st + item * GN, *sp = sc + item * GN, *pp = xp + item * 2 * GN;
                    const float *clp = lo + item * GN, *slp = lo + L.sin_f + item * GN;
                    float gv[GK], lam[GK], laml[GK];
                    lds_vec<GK>(st + g_off + item * GK, gv);
#pragma unroll
                    for (int i = 0; i < GK; ++i) {
                        float s_, e_;
                        ff_two_sum(carry[i], gv[i], s_, e_);
                        ff_fast_two_sum(s_, e_ + carryl[i], lam[i], laml[i]);
                    }
                    const int64_t o = ((bi * T + t) * H + head0 + lane);
                    stg_vec_cs<GK>(db + o * GK, lam);
                    float dthv[GN];
#pragma unroll
                    for (int l = GK - 1; l >= 0; --l) {
#pragma unroll
                        for (int q = 0; q < layer_pairs(l); ++q) {
                            const int p = (l & 1) + 2 * q, n = layer_base(l) + q;
                            dthv[n] = fmaf(lam[p + 1], pp[2 * n], -lam[p] * pp[2 * n + 1]);
                            ff_rot_bwd(lam[p], laml[p], lam[p + 1], laml[p + 1], cp[n], clp[n], sp[n], slp[n]);
                        }
                    }
                    stg_vec_cs<GN>(dth + o * GN, dthv);
#pragma unroll
                    for (int i = 0; i < GK; ++i) {
                        carry[i] = lam[i];
                        carryl[i] = laml[i];
                    }
                }
            } else
            for (int u = ts - 1; u >= first_row(j); --u) {
                const int64_t t = tb + u;
                const int item = u * lpw + lane;
                float cs[GN], sv[GN], lam[GK], hp[GK], pr[2 * GN];
                lds_vec<GN>(st + item * GN, cs);
                lds_vec<GN>(sc + item * GN, sv);
                lds_vec<2 * GN>(xp + item * 2 * GN, pr);
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
                // adjoint back through the layers, with the rotated pairs the
                // angle warps kept
                float dthv[GN];
#pragma unroll
                for (int l = GK - 1; l >= 0; --l) {
#pragma unroll
                    for (int q = 0; q < layer_pairs(l); ++q) {
                        const int p = (l & 1) + 2 * q, n = layer_base(l) + q;
                        dthv[n] = fmaf(lam[p + 1], pr[2 * n], -lam[p] * pr[2 * n + 1]);
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
        __syncthreads();
        MGS_BLOCK_ABORT_CHECK(br, producer, lane);
        if (it >= 1 && it - 1 + kNS < nblk) {
            const int s = int((it - 1) % kNS);
            if (tid == kBlockB - 1) {
                fence_proxy_async_smem();
                issue(s, it - 1 + kNS);
            }
            if (producer) br.rg.armed(s);
        }
    }
    if (active && dh0 != nullptr) {
        float *p = dh0 + (bi * H + head0 + lane) * GK;
        *reinterpret_cast<float4 *>(p) = make_float4(carry[0], carry[1], carry[2], carry[3]);
        *reinterpret_cast<float4 *>(p + 4) = make_float4(carry[4], carry[5], carry[6], carry[7]);
    }
}

// ---------------------------------------------------------------- matrix forward
// Warp 0's thread j of a lane's 8-thread group carries column j of P_t.
__global__ void __launch_bounds__(kBlockF)
    gms_fwd_kernel(const __grid_constant__ CUtensorMap tmTh, float *__restrict__ P, int64_t B, int64_t T,
                   int64_t H, int64_t groups_per_b, DevCtl ctl) {
    constexpr int TS = kGmsFwdTS;
    constexpr int STAGEF = TS * kGmsLanes * GN;  // one theta box (a multiple of 32 floats)
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp != 0;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    float *ring = reinterpret_cast<float *>(smem_raw);
    float *snb = ring + kNS * STAGEF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(snb + 2 * STAGEF);
    BlockRing br;
    br.init(bars, reinterpret_cast<int *>(bars + kNS), tid);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * kGmsLanes;
    const int sub = lane >> 3, col = lane & 7;
    const bool active = !producer && head0 + sub < H;
    const int64_t nblk = (T + TS - 1) / TS;
    const int row0 = int(bi * T);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {  // thread kBlockF-1 only
        mbar_arrive_expect_tx(&bars[s], uint32_t(STAGEF * 4));
        tma_load_3d(ring + size_t(s) * STAGEF, &tmTh, 0, head0, row0 + int(j * TS), &bars[s], pol);
    };
    const int npro = int(min64(kNS, nblk));
    if (tid == kBlockF - 1) {
        prefetch_tmap(&tmTh);
        for (int s = 0; s < npro; ++s) issue(s, s);
    }
    if (producer)
        for (int s = 0; s < npro; ++s) br.rg.armed(s);

    float v[GK];
#pragma unroll
    for (int i = 0; i < GK; ++i) v[i] = (i == col) ? 1.f : 0.f;
    float *pp = P + ((bi * T) * H + head0 + sub) * (GK * GK) + col;

    for (int64_t it = 0; it <= nblk; ++it) {
        if (producer && it < nblk) {
            const int s = int(it % kNS);
            if (br.rg.wait(s, ctl)) {
                angle_range<kProdF>(ring + size_t(s) * STAGEF, snb + (it & 1) * STAGEF, 0,
                            int(min64(TS, T - it * TS)) * kGmsLanes * GN, tid - 32);
            } else {
                if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
                *br.abort_word = 1;
            }
        }
        if (!producer && it >= 1) {
            const int64_t j = it - 1;
            const float *st = ring + size_t(j % kNS) * STAGEF;
            const float *sc = snb + (j & 1) * STAGEF;
            const int n = int(min64(TS, T - j * TS));
            for (int u = 0; u < n; ++u) {
                const int item = u * kGmsLanes + sub;
                float cs[GN], sv[GN];
                lds_vec<GN>(st + item * GN, cs);
                lds_vec<GN>(sc + item * GN, sv);
                mesh_apply(v, cs, sv);
                if (active) {
#pragma unroll
                    for (int i = 0; i < GK; ++i) st_cs(pp + i * GK, v[i]);
                }
                pp += H * GK * GK;
            }
        }
        __syncthreads();
        MGS_BLOCK_ABORT_CHECK(br, producer, lane);
        if (it >= 1 && it - 1 + kNS < nblk) {
            const int s = int((it - 1) % kNS);
            if (tid == kBlockF - 1) {
                fence_proxy_async_smem();
                issue(s, it - 1 + kNS);
            }
            if (producer) br.rg.armed(s);
        }
    }
}

// ---------------------------------------------------------------- matrix backward
// Per step and column j (t downwards, warp 0): Lambda = G_t[:, j] + carry;
// x = P_t[:, j]; both go back through the layers by transposed rotations (x
// recovers the column before each layer, exact up to rounding since the mesh
// is orthogonal), each thread adding its column's share of every angle's
// gradient; the eight shares are summed by a butterfly reduce-scatter that
// leaves angles 4j .. 4j+3 with thread j.  carry = A_t^T Lambda[:, j].
__global__ void __launch_bounds__(kBlockB)
    gms_bwd_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmP,
                   const __grid_constant__ CUtensorMap tmG, float *__restrict__ dth, int64_t B, int64_t T,
                   int64_t H, int64_t groups_per_b, DevCtl ctl) {
    constexpr int TS = kGmsBwdTS;
    using TM = MatTile<GK, true>;  // swizzled: conflict-free column reads
    constexpr int MATF = TS * TM::MF, THF = TS * kGmsLanes * GN;
    constexpr int STAGEF = int(align_up(size_t(2 * MATF + THF), TM::kAlign / 4));
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp != 0;
    const int64_t g = blockIdx.x;
    if (g >= B * groups_per_b) return;
    unsigned char *sbase = align_smem(smem_raw, TM::kAlign);
    float *ring = reinterpret_cast<float *>(sbase);
    float *snb = ring + kNS * STAGEF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(snb + 2 * THF);
    BlockRing br;
    br.init(bars, reinterpret_cast<int *>(bars + kNS), tid);

    const int64_t bi = g / groups_per_b;
    const int head0 = int(g % groups_per_b) * kGmsLanes;
    const int sub = lane >> 3, col = lane & 7;
    const bool active = !producer && head0 + sub < H;
    const int64_t nblk = (T + TS - 1) / TS;
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {  // thread kBlockB-1 only
        float *st = ring + size_t(s) * STAGEF;
        const int r = int(bi * T + T - (j + 1) * TS);
        mbar_arrive_expect_tx(&bars[s], uint32_t((2 * MATF + THF) * 4));
        TM::load(st, &tmP, head0, r, &bars[s], pol);
        TM::load(st + MATF, &tmG, head0, r, &bars[s], pol);
        tma_load_3d(st + 2 * MATF, &tmTh, 0, head0, r, &bars[s], pol);
    };
    const int npro = int(min64(kNS, nblk));
    if (tid == kBlockB - 1) {
        prefetch_tmap(&tmTh);
        prefetch_tmap(&tmP);
        prefetch_tmap(&tmG);
        for (int s = 0; s < npro; ++s) issue(s, s);
    }
    if (producer)
        for (int s = 0; s < npro; ++s) br.rg.armed(s);
    auto first_row = [&](int64_t j) -> int {
        const int64_t tb = T - (j + 1) * TS;
        return int(tb < 0 ? -tb : 0);
    };

    float carry[GK];
#pragma unroll
    for (int i = 0; i < GK; ++i) carry[i] = 0.f;

    for (int64_t it = 0; it <= nblk; ++it) {
        if (producer && it < nblk) {
            const int s = int(it % kNS);
            if (br.rg.wait(s, ctl)) {
                angle_range<kProdB>(ring + size_t(s) * STAGEF + 2 * MATF, snb + (it & 1) * THF,
                            first_row(it) * kGmsLanes * GN, THF, tid - 32);
            } else {
                if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);
                *br.abort_word = 1;
            }
        }
        if (!producer && it >= 1) {
            const int64_t j = it - 1;
            const int64_t tb = T - (j + 1) * TS;
            const float *st = ring + size_t(j % kNS) * STAGEF;
            const float *sth = st + 2 * MATF;
            const float *sc = snb + (j & 1) * THF;
            for (int u = TS - 1; u >= first_row(j); --u) {
                const int64_t t = tb + u;
                const TileRef<GK, true> Pt{st, u, sub}, Gt{st + MATF, u, sub};
                const int item = u * kGmsLanes + sub;
                float cs[GN], sv[GN], lam[GK], x[GK];
                lds_vec<GN>(sth + item * GN, cs);
                lds_vec<GN>(sc + item * GN, sv);
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
                    st_cs4(dth + ((bi * T + t) * H + head0 + sub) * GN + 4 * col,
                           make_float4(d[0], d[1], d[2], d[3]));
#pragma unroll
                for (int i = 0; i < GK; ++i) carry[i] = lam[i];
            }
        }
        __syncthreads();
        MGS_BLOCK_ABORT_CHECK(br, producer, lane);
        if (it >= 1 && it - 1 + kNS < nblk) {
            const int s = int((it - 1) % kNS);
            if (tid == kBlockB - 1) {
                fence_proxy_async_smem();
                issue(s, it - 1 + kNS);
            }
            if (producer) br.rg.armed(s);
        }
    }
}

// ---------------------------------------------------------------- few lanes, long sequences
// With few (batch, head) lanes and a long sequence, each lane of the kernels
// above walks a long serial chain on one thread.  There T is split into
// chunks and the scan runs as the reduce-then-scan of mgs_chunk.cuh, still
// from the angles: one warp per (group of 4 lanes, chunk) item, thread j of a
// lane's 8-thread group holding column j of the chunk's aggregate (the mesh
// applied to the columns of the identity) and, where a vector recurrence is
// needed, the whole vector (every thread of the lane computes it, no
// shuffles).  Each stage's angles are converted to cosines and sines in
// shared memory by the whole warp.  Neither A_t nor dA_t is ever formed: the
// workspace holds only the per-chunk aggregates and carries.

constexpr int kGcLanes = 4;                    // lanes per warp (8 threads each)
constexpr int kGcTS = 4;                       // steps per stage
constexpr int kGcNSmax = 4;                    // stages in flight (at most)
constexpr int kGcThF = kGcTS * kGcLanes * GN;  // floats of one stage's angle box
constexpr int kGcVecF = kGcTS * kGcLanes * GK; // floats of one stage's vector box
using GcTile = MatTile<GK, true>;              // k x k boxes (swizzled), matrix scan backward
constexpr int kGcMatF = kGcTS * GcTile::MF;

// Stage layout: [angles -> cosines][sines][nv vector boxes][nm k x k boxes].
// Small stages, and fewer of them for the k x k boxes, keep a one-warp
// block's shared memory low enough for many blocks per SM (these kernels are
// latency bound; with 96 KB blocks only two fit on an SM).
template <int NV, int NM>
struct GcStage {
    static constexpr int NS = NM > 0 ? 2 : kGcNSmax;
    static constexpr int vec_off = 2 * kGcThF;
    static constexpr int mat_off = int(align_up(size_t(vec_off + NV * kGcVecF), 256));
    static constexpr int floats = int(align_up(size_t(mat_off + NM * kGcMatF), NM > 0 ? 256 : 32));
    static constexpr uint32_t tx_bytes(int nv, int nm) { return uint32_t(kGcThF + nv * kGcVecF + nm * kGcMatF) * 4u; }
    // dynamic shared memory: the ring, its barriers, slack to align the base to 1024 bytes
    static constexpr int smem = int(size_t(NS) * floats * 4 + NS * sizeof(uint64_t) + 1024);
};

// The whole warp converts a landed stage's angles: cosines in place, sines
// into the stage's sine area.
template <bool kFast>
__device__ __forceinline__ void gc_convert(float *st, int lane) {
    float *sn = st + kGcThF;
    for (int i = lane; i < kGcThF; i += 32) {
        float c, sv;
        unbiased_cos_sin<kFast>(st[i], c, sv);
        st[i] = c;
        sn[i] = sv;
    }
    __syncwarp();
}

// x <- G^T x (the transposed mesh: layer k first, each by its transposed rotations)
__device__ __forceinline__ void mesh_apply_t(float (&x)[GK], const float (&cs)[GN], const float (&sn)[GN]) {
#pragma unroll
    for (int l = GK - 1; l >= 0; --l)
#pragma unroll
        for (int q = 0; q < layer_pairs(l); ++q) {
            const int p = (l & 1) + 2 * q, n = layer_base(l) + q;
            rot_bwd(x[p], x[p + 1], cs[n], sn[n]);
        }
}

// Element j of a register vector, selected without dynamic indexing.
__device__ __forceinline__ float pick8(const float (&v)[GK], int j) {
    float r = v[0];
#pragma unroll
    for (int i = 1; i < GK; ++i) r = (i == j) ? v[i] : r;
    return r;
}

// Common per-item set-up of the chunked Givens kernels: the ring and the item.
struct GcItem {
    ChunkItem it;
    int sub, col, nl;
    int64_t tb, te, len, nb;
    __device__ GcItem(int64_t item, int64_t nper, int64_t cfirst, int64_t gpb, int64_t T, int64_t H, int64_t Lc)
        : it(item, nper, cfirst, gpb, kGcLanes) {
        sub = int(threadIdx.x) >> 3;
        col = int(threadIdx.x) & 7;
        nl = int(min64(kGcLanes, H - it.head0));
        tb = it.c * Lc;
        te = min64(T, tb + Lc);
        len = te - tb;
        nb = (len + kGcTS - 1) / kGcTS;
    }
};

#define MGS_GC_WAIT_OR_RETURN(rg, s)                          \
    if (!(rg).wait(s, ctl)) {                                 \
        if (lane == 0) record_error(ctl, ERR_MBAR_TIMEOUT);   \
        (rg).drain(ctl, lane);                                \
        return;                                               \
    }

// ---- affine scan, launch 1 forward: h_end = M h_in + c of chunks 0 .. C-2
__global__ void __launch_bounds__(32)
    gc_affine_fwd_agg_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, float *__restrict__ Ms, float *__restrict__ Cs,
                             int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc, DevCtl ctl) {
    using L = GcStage<2, 0>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C - 1, 0, gpb, T, H, Lc);
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L::floats;
        const int r = int(w.it.bi * T + w.tb + j * kGcTS);
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(2, 0));
        tma_load_3d(st, &tmTh, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off, &tmA, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off + kGcVecF, &tmB, 0, w.it.head0, r, &bars[s], pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mcol[GK], cv[GK];  // column col of M; the whole offset c
#pragma unroll
    for (int i = 0; i < GK; ++i) {
        mcol[i] = (i == w.col) ? 1.f : 0.f;
        cv[i] = 0.f;
    }
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<true>(st, lane);
        const int n = int(min64(kGcTS, w.len - j * kGcTS));
        for (int u = 0; u < n; ++u) {
            const int item = u * kGcLanes + w.sub;
            float cs[GN], sv[GN], av[GK], bv[GK];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
            lds_vec<GK>(st + L::vec_off + item * GK, av);
            lds_vec<GK>(st + L::vec_off + kGcVecF + item * GK, bv);
#pragma unroll
            for (int i = 0; i < GK; ++i) {
                mcol[i] *= av[i];
                cv[i] *= av[i];
            }
            mesh_apply(mcol, cs, sv);
            mesh_apply(cv, cs, sv);
#pragma unroll
            for (int i = 0; i < GK; ++i) cv[i] += bv[i];
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
    const int64_t itm = w.it.g * C + w.it.c;
    st_ws_col<GK>(Ms + itm * (kGcLanes * GK * GK) + w.sub * GK * GK, w.col, mcol);
    __stcg(Cs + itm * (kGcLanes * GK) + w.sub * GK + w.col, pick8(cv, w.col));
}

// ---- affine scan, launch 3 forward: h_t from each chunk's carry
__global__ void __launch_bounds__(32)
    gc_affine_fwd_out_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, float *__restrict__ h,
                             const float *__restrict__ Es, int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc,
                             DevCtl ctl) {
    using L = GcStage<2, 0>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C, 0, gpb, T, H, Lc);
    const bool active = w.sub < w.nl;
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L::floats;
        const int r = int(w.it.bi * T + w.tb + j * kGcTS);
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(2, 0));
        tma_load_3d(st, &tmTh, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off, &tmA, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off + kGcVecF, &tmB, 0, w.it.head0, r, &bars[s], pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    pdl_wait();  // the carries of launch 2
    float x[GK];
    lds_row_global<GK>(Es + (w.it.g * C + w.it.c) * (kGcLanes * GK) + w.sub * GK, x);
    float *hp = h + ((w.it.bi * T + w.tb) * H + w.it.head0 + w.sub) * GK + w.col;
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<true>(st, lane);
        const int n = int(min64(kGcTS, w.len - j * kGcTS));
        for (int u = 0; u < n; ++u) {
            const int item = u * kGcLanes + w.sub;
            float cs[GN], sv[GN], av[GK], bv[GK];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
            lds_vec<GK>(st + L::vec_off + item * GK, av);
            lds_vec<GK>(st + L::vec_off + kGcVecF + item * GK, bv);
#pragma unroll
            for (int i = 0; i < GK; ++i) x[i] *= av[i];
            mesh_apply(x, cs, sv);
#pragma unroll
            for (int i = 0; i < GK; ++i) x[i] += bv[i];
            if (active) st_cs(hp, pick8(x, w.col));
            hp += H * GK;
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
}

// ---- affine scan, launch 1 backward: mu_out = M mu_in + C of chunks 1 .. C-1
// (per step lambda = g + mu, mu <- A^T lambda = a * G^T lambda)
__global__ void __launch_bounds__(32)
    gc_affine_bwd_agg_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmG, float *__restrict__ Ms, float *__restrict__ Cs,
                             int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc, DevCtl ctl) {
    using L = GcStage<2, 0>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C - 1, 1, gpb, T, H, Lc);
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();
    // block j covers t = te-1-j*TS down to max(tb, te-(j+1)*TS); boxes start at
    // row te-(j+1)*TS, step u at box row TS-1-u
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L::floats;
        const int r = int(w.it.bi * T + w.te - (j + 1) * kGcTS);
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(2, 0));
        tma_load_3d(st, &tmTh, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off, &tmA, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off + kGcVecF, &tmG, 0, w.it.head0, r, &bars[s], pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mcol[GK], mu[GK];  // column col of M; the whole offset C
#pragma unroll
    for (int i = 0; i < GK; ++i) {
        mcol[i] = (i == w.col) ? 1.f : 0.f;
        mu[i] = 0.f;
    }
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<true>(st, lane);
        const int64_t tt = w.te - 1 - j * kGcTS;
        const int n = int(min64(kGcTS, tt - w.tb + 1));
        for (int u = 0; u < n; ++u) {
            const int item = (kGcTS - 1 - u) * kGcLanes + w.sub;
            float cs[GN], sv[GN], av[GK], gv[GK];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
            lds_vec<GK>(st + L::vec_off + item * GK, av);
            lds_vec<GK>(st + L::vec_off + kGcVecF + item * GK, gv);
#pragma unroll
            for (int i = 0; i < GK; ++i) mu[i] += gv[i];
            mesh_apply_t(mu, cs, sv);
            mesh_apply_t(mcol, cs, sv);
#pragma unroll
            for (int i = 0; i < GK; ++i) {
                mu[i] *= av[i];
                mcol[i] *= av[i];
            }
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
    const int64_t itm = w.it.g * C + w.it.c;
    st_ws_col<GK>(Ms + itm * (kGcLanes * GK * GK) + w.sub * GK * GK, w.col, mcol);
    __stcg(Cs + itm * (kGcLanes * GK) + w.sub * GK + w.col, pick8(mu, w.col));
}

// ---- affine scan, launch 3 backward: d theta, da, db (dh0 from chunk 0)
__global__ void __launch_bounds__(32)
    gc_affine_bwd_out_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmH,
                             const float *__restrict__ h0, float *__restrict__ dth, float *__restrict__ da,
                             float *__restrict__ db, float *__restrict__ dh0, const float *__restrict__ Es,
                             int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc, DevCtl ctl) {
    using L = GcStage<3, 0>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C, 0, gpb, T, H, Lc);
    const bool active = w.sub < w.nl;
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    // as in launch 1; the h box starts one row earlier and holds h_{t-1}
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L::floats;
        const int r = int(w.it.bi * T + w.te - (j + 1) * kGcTS);
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(3, 0));
        tma_load_3d(st, &tmTh, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off, &tmA, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off + kGcVecF, &tmG, 0, w.it.head0, r, &bars[s], pol);
        tma_load_3d(st + L::vec_off + 2 * kGcVecF, &tmH, 0, w.it.head0, r - 1, &bars[s], pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float h0v[GK];
#pragma unroll
    for (int i = 0; i < GK; ++i) h0v[i] = 0.f;
    if (h0 != nullptr && active) lds_row_global<GK>(h0 + (w.it.bi * H + w.it.head0 + w.sub) * GK, h0v);
    pdl_wait();  // the carries of launch 2
    float mu[GK];  // A_{t+1}^T lambda_{t+1} past the step, the whole vector
    lds_row_global<GK>(Es + (w.it.g * C + w.it.c) * (kGcLanes * GK) + w.sub * GK, mu);
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<true>(st, lane);
        const int64_t tt = w.te - 1 - j * kGcTS;
        const int n = int(min64(kGcTS, tt - w.tb + 1));
        for (int u = 0; u < n; ++u) {
            const int64_t t = tt - u;
            const int item = (kGcTS - 1 - u) * kGcLanes + w.sub;
            float cs[GN], sv[GN], av[GK], lam[GK], hp[GK];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
            lds_vec<GK>(st + L::vec_off + item * GK, av);
            lds_vec<GK>(st + L::vec_off + kGcVecF + item * GK, lam);
            if (t >= 1) {
                lds_vec<GK>(st + L::vec_off + 2 * kGcVecF + item * GK, hp);
            } else {
#pragma unroll
                for (int i = 0; i < GK; ++i) hp[i] = h0v[i];
            }
#pragma unroll
            for (int i = 0; i < GK; ++i) lam[i] += mu[i];
            const int64_t o = (w.it.bi * T + t) * H + w.it.head0 + w.sub;
            if (active) st_cs(db + o * GK + w.col, pick8(lam, w.col));
            // forward through the layers from a * h_{t-1}, keeping each rotation's output pair
            float x[GK], pr[2 * GN];
#pragma unroll
            for (int i = 0; i < GK; ++i) x[i] = av[i] * hp[i];
#pragma unroll
            for (int l = 0; l < GK; ++l)
#pragma unroll
                for (int q = 0; q < layer_pairs(l); ++q) {
                    const int p = (l & 1) + 2 * q, nn = layer_base(l) + q;
                    rot_fwd(x[p], x[p + 1], cs[nn], sv[nn]);
                    pr[2 * nn] = x[p];
                    pr[2 * nn + 1] = x[p + 1];
                }
            // lambda back through the layers; each angle's gradient on the way
            float dthv[GN];
#pragma unroll
            for (int l = GK - 1; l >= 0; --l)
#pragma unroll
                for (int q = 0; q < layer_pairs(l); ++q) {
                    const int p = (l & 1) + 2 * q, nn = layer_base(l) + q;
                    dthv[nn] = fmaf(lam[p + 1], pr[2 * nn], -lam[p] * pr[2 * nn + 1]);
                    rot_bwd(lam[p], lam[p + 1], cs[nn], sv[nn]);
                }
            if (active) {
                // thread col < 7 stores angles 4 col .. 4 col + 3
#pragma unroll
                for (int c4 = 0; c4 < GN / 4; ++c4)
                    if (c4 == w.col)
                        st_cs4(dth + o * GN + 4 * c4,
                               make_float4(dthv[4 * c4], dthv[4 * c4 + 1], dthv[4 * c4 + 2], dthv[4 * c4 + 3]));
                if (da != nullptr) st_cs(da + o * GK + w.col, pick8(lam, w.col) * pick8(hp, w.col));
            }
#pragma unroll
            for (int i = 0; i < GK; ++i) mu[i] = av[i] * lam[i];
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
    if (w.it.c == 0 && dh0 != nullptr && active)
        dh0[(w.it.bi * H + w.it.head0 + w.sub) * GK + w.col] = pick8(mu, w.col);
}

// ---- matrix scan, launch 1 forward: M = G_e ... G_s of chunks 0 .. C-2
__global__ void __launch_bounds__(32)
    gc_matrix_fwd_agg_kernel(const __grid_constant__ CUtensorMap tmTh, float *__restrict__ Ms, int64_t T, int64_t H,
                             int64_t gpb, int64_t C, int64_t Lc, DevCtl ctl) {
    using L = GcStage<0, 0>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C - 1, 0, gpb, T, H, Lc);
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(0, 0));
        tma_load_3d(ring + size_t(s) * L::floats, &tmTh, 0, w.it.head0, int(w.it.bi * T + w.tb + j * kGcTS), &bars[s],
                    pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float v[GK];
#pragma unroll
    for (int i = 0; i < GK; ++i) v[i] = (i == w.col) ? 1.f : 0.f;
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<false>(st, lane);
        const int n = int(min64(kGcTS, w.len - j * kGcTS));
        for (int u = 0; u < n; ++u) {
            const int item = u * kGcLanes + w.sub;
            float cs[GN], sv[GN];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
            mesh_apply(v, cs, sv);
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
    st_ws_col<GK>(Ms + (w.it.g * C + w.it.c) * GcTile::MF + w.sub * GK * GK, w.col, v);
}

// ---- matrix scan, launch 3 forward: P_t from each chunk's carry
__global__ void __launch_bounds__(32)
    gc_matrix_fwd_out_kernel(const __grid_constant__ CUtensorMap tmTh, float *__restrict__ P,
                             const float *__restrict__ Es, int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc,
                             DevCtl ctl) {
    using L = GcStage<0, 0>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C, 0, gpb, T, H, Lc);
    const bool active = w.sub < w.nl;
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(0, 0));
        tma_load_3d(ring + size_t(s) * L::floats, &tmTh, 0, w.it.head0, int(w.it.bi * T + w.tb + j * kGcTS), &bars[s],
                    pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    pdl_wait();  // the carries of launch 2
    float v[GK];
    ld_ws_col<GK>(Es + (w.it.g * C + w.it.c) * GcTile::MF + w.sub * GK * GK, w.col, v);
    float *pp = P + ((w.it.bi * T + w.tb) * H + w.it.head0 + w.sub) * (GK * GK) + w.col;
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<false>(st, lane);
        const int n = int(min64(kGcTS, w.len - j * kGcTS));
        for (int u = 0; u < n; ++u) {
            const int item = u * kGcLanes + w.sub;
            float cs[GN], sv[GN];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
            mesh_apply(v, cs, sv);
            if (active) {
#pragma unroll
                for (int i = 0; i < GK; ++i) st_cs(pp + i * GK, v[i]);
            }
            pp += H * GK * GK;
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
}

// ---- matrix scan, launch 1 backward: (M, C) of chunks 1 .. C-1, M = G_s^T ... G_e^T
__global__ void __launch_bounds__(32)
    gc_matrix_bwd_agg_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmG,
                             float *__restrict__ Ms, float *__restrict__ Cs, int64_t T, int64_t H, int64_t gpb,
                             int64_t C, int64_t Lc, DevCtl ctl) {
    using L = GcStage<0, 1>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C - 1, 1, gpb, T, H, Lc);
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_last();
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L::floats;
        const int r = int(w.it.bi * T + w.te - (j + 1) * kGcTS);
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(0, 1));
        tma_load_3d(st, &tmTh, 0, w.it.head0, r, &bars[s], pol);
        GcTile::load(st + L::mat_off, &tmG, w.it.head0, r, &bars[s], pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float mcol[GK], mu[GK];  // columns col of M and of C
#pragma unroll
    for (int i = 0; i < GK; ++i) {
        mcol[i] = (i == w.col) ? 1.f : 0.f;
        mu[i] = 0.f;
    }
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<false>(st, lane);
        const int64_t tt = w.te - 1 - j * kGcTS;
        const int n = int(min64(kGcTS, tt - w.tb + 1));
        for (int u = 0; u < n; ++u) {
            const int q = kGcTS - 1 - u;
            const int item = q * kGcLanes + w.sub;
            const TileRef<GK, true> Gt{st + L::mat_off, q, w.sub};
            float cs[GN], sv[GN];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
#pragma unroll
            for (int i = 0; i < GK; ++i) mu[i] += Gt.at(i, w.col);
            mesh_apply_t(mu, cs, sv);
            mesh_apply_t(mcol, cs, sv);
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
    const int64_t slot = (w.it.g * C + w.it.c) * GcTile::MF + w.sub * GK * GK;
    st_ws_col<GK>(Ms + slot, w.col, mcol);
    st_ws_col<GK>(Cs + slot, w.col, mu);
}

// ---- matrix scan, launch 3 backward: d theta from each chunk's carry; per
// step and column j: Lambda = G_t[:, j] + carry, x = P_t[:, j], both back
// through the layers (x recovers the pre-rotation columns), the eight
// columns' shares of each angle summed by a butterfly reduce-scatter
__global__ void __launch_bounds__(32)
    gc_matrix_bwd_out_kernel(const __grid_constant__ CUtensorMap tmTh, const __grid_constant__ CUtensorMap tmP,
                             const __grid_constant__ CUtensorMap tmG, float *__restrict__ dth,
                             const float *__restrict__ Es, int64_t T, int64_t H, int64_t gpb, int64_t C, int64_t Lc,
                             DevCtl ctl) {
    using L = GcStage<0, 2>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ring = reinterpret_cast<float *>(align_smem(smem_raw, 1024));
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + L::NS * L::floats);
    const int lane = threadIdx.x;
    const GcItem w(blockIdx.x, C, 0, gpb, T, H, Lc);
    const bool active = w.sub < w.nl;
    WarpRing<L::NS> rg;
    rg.init(bars, lane);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t j) {  // lane 0 only
        float *st = ring + size_t(s) * L::floats;
        const int r = int(w.it.bi * T + w.te - (j + 1) * kGcTS);
        mbar_arrive_expect_tx(&bars[s], L::tx_bytes(0, 2));
        tma_load_3d(st, &tmTh, 0, w.it.head0, r, &bars[s], pol);
        GcTile::load(st + L::mat_off, &tmP, w.it.head0, r, &bars[s], pol);
        GcTile::load(st + L::mat_off + kGcMatF, &tmG, w.it.head0, r, &bars[s], pol);
    };
    const int npro = int(min64(L::NS, w.nb));
    if (lane == 0)
        for (int s = 0; s < npro; ++s) issue(s, s);
    for (int s = 0; s < npro; ++s) rg.armed(s);

    pdl_wait();  // the carries of launch 2
    float carry[GK];
    ld_ws_col<GK>(Es + (w.it.g * C + w.it.c) * GcTile::MF + w.sub * GK * GK, w.col, carry);
    for (int64_t j = 0; j < w.nb; ++j) {
        const int s = int(j % L::NS);
        MGS_GC_WAIT_OR_RETURN(rg, s);
        float *st = ring + size_t(s) * L::floats;
        gc_convert<false>(st, lane);
        const int64_t tt = w.te - 1 - j * kGcTS;
        const int n = int(min64(kGcTS, tt - w.tb + 1));
        for (int u = 0; u < n; ++u) {
            const int64_t t = tt - u;
            const int q = kGcTS - 1 - u;
            const int item = q * kGcLanes + w.sub;
            const TileRef<GK, true> Pt{st + L::mat_off, q, w.sub}, Gt{st + L::mat_off + kGcMatF, q, w.sub};
            float cs[GN], sv[GN], lam[GK], x[GK];
            lds_vec<GN>(st + item * GN, cs);
            lds_vec<GN>(st + kGcThF + item * GN, sv);
#pragma unroll
            for (int i = 0; i < GK; ++i) {
                lam[i] = Gt.at(i, w.col) + carry[i];
                x[i] = Pt.at(i, w.col);
            }
            float d[32];
#pragma unroll
            for (int l = GK - 1; l >= 0; --l)
#pragma unroll
                for (int qq = 0; qq < layer_pairs(l); ++qq) {
                    const int p = (l & 1) + 2 * qq, nn = layer_base(l) + qq;
                    d[nn] = fmaf(lam[p + 1], x[p], -lam[p] * x[p + 1]);
                    rot_bwd(x[p], x[p + 1], cs[nn], sv[nn]);
                    rot_bwd(lam[p], lam[p + 1], cs[nn], sv[nn]);
                }
#pragma unroll
            for (int nn = GN; nn < 32; ++nn) d[nn] = 0.f;
#pragma unroll
            for (int o = 4, half = 16; o >= 1; o >>= 1, half >>= 1) {
                const bool up = (w.col & o) != 0;
#pragma unroll
                for (int c = 0; c < half; ++c) {
                    const float send = up ? d[c] : d[c + half];
                    const float keep = up ? d[c + half] : d[c];
                    d[c] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (active && w.col < GN / 4)
                st_cs4(dth + ((w.it.bi * T + t) * H + w.it.head0 + w.sub) * GN + 4 * w.col,
                       make_float4(d[0], d[1], d[2], d[3]));
#pragma unroll
            for (int i = 0; i < GK; ++i) carry[i] = lam[i];
        }
        __syncwarp();
        if (j + L::NS < w.nb) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(s, j + L::NS);
            }
            rg.armed(s);
        }
    }
}

// Lanes per recurrence warp for the affine scan: as many as keep at least
// one block per SM, at most kGasMaxLanes (beyond that the angle warps, which
// convert 28 angles per lane and step, fall behind the recurrence), and no
// more than the heads of one batch row.
int gas_lanes_per_block(int64_t B, int64_t H) {
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int lpw = 1;
    while (lpw < kGasMaxLanes && B * H / (2 * lpw) >= sms) lpw *= 2;
    while (lpw > 1 && lpw / 2 >= H) lpw /= 2;
    return lpw;
}

// The few-lane path is taken when the matrix kernels would split T into
// chunks (fewer than 256 groups of 4 lanes) and T is at least 256.
bool few_lane_path(int64_t B, int64_t T, int64_t H) { return T >= 256 && mas_workspace_bytes(B, T, H, GK) > 0; }


}  // namespace

size_t givens_workspace_bytes(int op, int64_t B, int64_t T, int64_t H) {
    if (!few_lane_path(B, T, H)) return 0;
    // the chunk aggregates and carries only, laid out as matrix_affine_scan's
    // (affine) and matrix_scan's (matrix) chunked paths lay out theirs
    switch (op) {
        case 0:
        case 1: return mas_workspace_bytes(B, T, H, GK);
        case 2: return ms_workspace_bytes(B, T, H, GK, false);
        default: return ms_workspace_bytes(B, T, H, GK, true);
    }
}

namespace {
// Tensor maps of the chunked Givens kernels: angle and vector boxes of
// kGcTS steps x kGcLanes heads.
cudaError_t gc_vec_map(CUtensorMap *m, const float *base, int64_t B, int64_t T, int64_t H, int E) {
    return make_head_map(m, base, B * T, H, E, kGcLanes, kGcTS);
}
}  // namespace

const SinCosTable &sincos_table() {
    static const SinCosTable t = SinCosTable::build();
    return t;
}

cudaError_t launch_gas_fwd(const float *theta, const float *a, const float *b, const float *h0, float *h,
                           int64_t B, int64_t T, int64_t H, void *ws, size_t ws_bytes, const DevCtl &ctl,
                           cudaStream_t s) {
    // without the gate the exact-orthogonal kernels run at every shape (the
    // few-lane path's fp32 matrix kernels cannot carry the extra precision)
    const bool xo = a == nullptr;
    if (!xo && few_lane_path(B, T, H)) {
        const ChunkPlan pl = plan_chunks(B, T, H, GK);
        const int64_t gpb = (H + kGcLanes - 1) / kGcLanes;
        const ScanWs w(static_cast<unsigned char *>(ws), pl, kGcLanes * GK * GK, kGcLanes * GK);
        CUtensorMap tTh, tA, tB;
        cudaError_t e;
        if ((e = gc_vec_map(&tTh, theta, B, T, H, GN)) != cudaSuccess) return e;
        if ((e = gc_vec_map(&tA, a, B, T, H, GK)) != cudaSuccess) return e;
        if ((e = gc_vec_map(&tB, b, B, T, H, GK)) != cudaSuccess) return e;
        constexpr int smem = GcStage<2, 0>::smem;
        if ((e = ensure_smem_attr((const void *)gc_affine_fwd_agg_kernel, smem)) != cudaSuccess) return e;
        if ((e = ensure_smem_attr((const void *)gc_affine_fwd_out_kernel, smem)) != cudaSuccess) return e;
        gc_affine_fwd_agg_kernel<<<dim3(unsigned(pl.G * (pl.C - 1))), 32, smem, s>>>(tTh, tA, tB, w.M, w.Cv, T, H, gpb,
                                                                                   pl.C, pl.L, ctl);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_chain<GK, false, true, +1>(w.M, w.Cv, w.E, h0, pl.G, pl.C, gpb, H, ctl, s)) != cudaSuccess)
            return e;
        return launch_pdl(gc_affine_fwd_out_kernel, dim3(unsigned(pl.G * pl.C)), smem, s, tTh, tA, tB, h, w.E, T, H,
                          gpb, pl.C, pl.L, ctl);
    }
    const int lpw = gas_lanes_per_block(B, H), ts = kItems / lpw;
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
    const int smem = int(GasSmem(lpw, ts, a ? 2 : 1, false, xo).bytes());
    const auto kern = xo ? gas_fwd_kernel<true> : gas_fwd_kernel<false>;
    if ((e = ensure_smem_attr((const void *)kern, smem)) != cudaSuccess) return e;
    kern<<<dim3(unsigned(blocks)), kBlockF, smem, s>>>(tTh, tA, tB, h0, h, B, T, H, gpb, lpw, ts, a != nullptr,
                                                       sincos_table(), ctl);
    return cudaGetLastError();
}

cudaError_t launch_gas_bwd(const float *theta, const float *a, const float *h0, const float *h, const float *gh,
                           float *dth, float *da, float *db, float *dh0, int64_t B, int64_t T, int64_t H,
                           void *ws, size_t ws_bytes, const DevCtl &ctl, cudaStream_t s) {
    const bool xo = a == nullptr;  // as in the forward
    if (!xo && few_lane_path(B, T, H)) {
        const ChunkPlan pl = plan_chunks(B, T, H, GK);
        const int64_t gpb = (H + kGcLanes - 1) / kGcLanes;
        const ScanWs w(static_cast<unsigned char *>(ws), pl, kGcLanes * GK * GK, kGcLanes * GK);
        CUtensorMap tTh, tA, tG, tH;
        cudaError_t e;
        if ((e = gc_vec_map(&tTh, theta, B, T, H, GN)) != cudaSuccess) return e;
        if ((e = gc_vec_map(&tA, a, B, T, H, GK)) != cudaSuccess) return e;
        if ((e = gc_vec_map(&tG, gh, B, T, H, GK)) != cudaSuccess) return e;
        if ((e = gc_vec_map(&tH, h, B, T, H, GK)) != cudaSuccess) return e;
        constexpr int sa = GcStage<2, 0>::smem, so = GcStage<3, 0>::smem;
        if ((e = ensure_smem_attr((const void *)gc_affine_bwd_agg_kernel, sa)) != cudaSuccess) return e;
        if ((e = ensure_smem_attr((const void *)gc_affine_bwd_out_kernel, so)) != cudaSuccess) return e;
        gc_affine_bwd_agg_kernel<<<dim3(unsigned(pl.G * (pl.C - 1))), 32, sa, s>>>(tTh, tA, tG, w.M, w.Cv, T, H, gpb,
                                                                                 pl.C, pl.L, ctl);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_chain<GK, false, true, -1>(w.M, w.Cv, w.E, nullptr, pl.G, pl.C, gpb, H, ctl, s)) != cudaSuccess)
            return e;
        return launch_pdl(gc_affine_bwd_out_kernel, dim3(unsigned(pl.G * pl.C)), so, s, tTh, tA, tG, tH, h0, dth, da,
                          db, dh0, w.E, T, H, gpb, pl.C, pl.L, ctl);
    }
    const int lpw = gas_lanes_per_block(B, H), ts = kItems / lpw;
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
    const int smem = int(GasSmem(lpw, ts, a ? 3 : 2, true, xo).bytes());
    const auto kern = xo ? gas_bwd_kernel<true> : gas_bwd_kernel<false>;
    if ((e = ensure_smem_attr((const void *)kern, smem)) != cudaSuccess) return e;
    kern<<<dim3(unsigned(blocks)), kBlockB, smem, s>>>(tTh, tA, tG, tH, h0, dth, da, db, dh0, B, T, H, gpb, lpw, ts,
                                                       a != nullptr, sincos_table(), ctl);
    return cudaGetLastError();
}

cudaError_t launch_gms_fwd(const float *theta, float *P, int64_t B, int64_t T, int64_t H, void *ws,
                           size_t ws_bytes, const DevCtl &ctl, cudaStream_t s) {
    if (few_lane_path(B, T, H)) {
        const ChunkPlan pl = plan_chunks(B, T, H, GK);
        const int64_t gpb = (H + kGcLanes - 1) / kGcLanes;
        const ScanWs w(static_cast<unsigned char *>(ws), pl, GcTile::MF, 0);
        CUtensorMap tTh;
        cudaError_t e;
        if ((e = gc_vec_map(&tTh, theta, B, T, H, GN)) != cudaSuccess) return e;
        constexpr int smem = GcStage<0, 0>::smem;
        if ((e = ensure_smem_attr((const void *)gc_matrix_fwd_agg_kernel, smem)) != cudaSuccess) return e;
        if ((e = ensure_smem_attr((const void *)gc_matrix_fwd_out_kernel, smem)) != cudaSuccess) return e;
        gc_matrix_fwd_agg_kernel<<<dim3(unsigned(pl.G * (pl.C - 1))), 32, smem, s>>>(tTh, w.M, T, H, gpb, pl.C, pl.L,
                                                                                   ctl);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_chain<GK, true, false, +1>(w.M, nullptr, w.E, nullptr, pl.G, pl.C, gpb, H, ctl, s)) !=
            cudaSuccess)
            return e;
        return launch_pdl(gc_matrix_fwd_out_kernel, dim3(unsigned(pl.G * pl.C)), smem, s, tTh, P, w.E, T, H, gpb, pl.C,
                          pl.L, ctl);
    }
    CUtensorMap tTh;
    cudaError_t e;
    if ((e = make_head_map(&tTh, theta, B * T, H, GN, kGmsLanes, kGmsFwdTS)) != cudaSuccess) return e;
    const int64_t gpb = (H + kGmsLanes - 1) / kGmsLanes, blocks = B * gpb;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    constexpr int STAGEF = kGmsFwdTS * kGmsLanes * GN;
    const int smem = int((kNS + 2) * STAGEF * 4 + kNS * sizeof(uint64_t) + 16);
    if ((e = ensure_smem_attr((const void *)gms_fwd_kernel, smem)) != cudaSuccess) return e;
    gms_fwd_kernel<<<dim3(unsigned(blocks)), kBlockF, smem, s>>>(tTh, P, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

cudaError_t launch_gms_bwd(const float *theta, const float *P, const float *G, float *dth, int64_t B, int64_t T,
                           int64_t H, void *ws, size_t ws_bytes, const DevCtl &ctl, cudaStream_t s) {
    if (few_lane_path(B, T, H)) {
        const ChunkPlan pl = plan_chunks(B, T, H, GK);
        const int64_t gpb = (H + kGcLanes - 1) / kGcLanes;
        const ScanWs w(static_cast<unsigned char *>(ws), pl, GcTile::MF, GcTile::MF);
        CUtensorMap tTh, tP, tG;
        cudaError_t e;
        if ((e = gc_vec_map(&tTh, theta, B, T, H, GN)) != cudaSuccess) return e;
        if ((e = GcTile::make(&tP, P, B * T, H, kGcTS)) != cudaSuccess) return e;
        if ((e = GcTile::make(&tG, G, B * T, H, kGcTS)) != cudaSuccess) return e;
        constexpr int sa = GcStage<0, 1>::smem, so = GcStage<0, 2>::smem;
        if ((e = ensure_smem_attr((const void *)gc_matrix_bwd_agg_kernel, sa)) != cudaSuccess) return e;
        if ((e = ensure_smem_attr((const void *)gc_matrix_bwd_out_kernel, so)) != cudaSuccess) return e;
        gc_matrix_bwd_agg_kernel<<<dim3(unsigned(pl.G * (pl.C - 1))), 32, sa, s>>>(tTh, tG, w.M, w.Cv, T, H, gpb, pl.C,
                                                                                 pl.L, ctl);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_chain<GK, true, true, -1>(w.M, w.Cv, w.E, nullptr, pl.G, pl.C, gpb, H, ctl, s)) !=
            cudaSuccess)
            return e;
        return launch_pdl(gc_matrix_bwd_out_kernel, dim3(unsigned(pl.G * pl.C)), so, s, tTh, tP, tG, dth, w.E, T, H,
                          gpb, pl.C, pl.L, ctl);
    }
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
    const int smem = int(size_t(kNS * STAGEF + 2 * THF) * 4 + kNS * sizeof(uint64_t) + 16 + TM::kAlign);
    if ((e = ensure_smem_attr((const void *)gms_bwd_kernel, smem)) != cudaSuccess) return e;
    gms_bwd_kernel<<<dim3(unsigned(blocks)), kBlockB, smem, s>>>(tTh, tP, tG, dth, B, T, H, gpb, ctl);
    return cudaGetLastError();
}

}  // namespace mgs
