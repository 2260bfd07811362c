// Delta rule (DeltaNet), forward, in the chunked WY form ("mingru-scans" home
// page, lineage paragraph: DeltaMinGRU reimplements DeltaNet, Yang et al.
// 2024, arXiv:2406.06484, using its chunked WY representation as the
// parallel forward).  Per (batch, head) lane, state S (d_v x d_k, here D x D):
//   S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T,   o_t = S_t q_t.
//
// A chunk of C = 64 steps with state S on entry is, in matrix form (rows are
// time steps, K, V, Q are C x D):
//   A   = strict_tril(diag(beta) K K^T)
//   (I + A) [W | U] = diag(beta) [K | V],   P = tril(Q K^T)
//   U'  = U - W S^T
//   O   = Q S^T + P U'
//   S  <- S + U'^T K
// which is the recurrence exactly (the WY representation of the product of
// the chunk's rank-one updates).  Substituting U' into the last two lines
// gives the chunk as an affine map of the state,
//   S^T <- M S^T + N,   O = R S^T + O_c,
//   M = I - K^T W,  N = K^T U,  R = Q - P W,  O_c = P U,
// whose four matrices depend on the chunk's inputs only.  They are formed for
// every chunk at once (delta_wy_kernel, one block per chunk); the state pass
// (delta_state_kernel) then carries S^T through a lane's chunks in order with
// one stacked product per chunk, [R; M] S^T.  Its columns (the value index i)
// are independent, so a lane is split into blocks of 16, 32 or 64 value
// columns (narrower when lanes are few, so that more blocks run).
//
// The 64 x 64 products run on the fifth-generation tensor cores
// (tcgen05.mma kind::tf32, M = 128: two 64-row products stacked in one), with
// fp32 accuracy from a three-term split: x = xb + xs with xb = x rounded to
// tf32 and xs = x - xb, a b ~ as bb + ab bs + ab bb (the as bs term is below
// fp32 resolution).  The stacked A operands sit in tensor memory, split by the
// threads that hold their rows; the B operands are 128-byte-swizzled K-major
// tiles in shared memory; the accumulators are in tensor memory.  Where the B
// operand is stored as [B_small; B_big] row blocks, one N = 2n instruction
// gives ab [bs | bb] and one N = n instruction adds as bb onto the second half
// (two instructions per k step instead of three; the result is the sum of the
// two halves).
//   WY pass:    [K; Q] K^T           -> A (masked, scaled) and P
//               [K^T; V^T] T'^T      -> W^T and U^T
//               [K^T; P] [W | U]     -> K^T W, N, P W, O_c
//   state pass: [R; M] S^T           -> R S^T (+ O_c: the output), M S^T (+ N: the state)
// T' = (I + A)^{-1} diag(beta) (lower triangular, so [W | U] = T' [K | V]) is
// formed on the fp32 pipes by 16 x 16 blocks: the diagonal blocks
// D_b = (I + A_bb)^{-1} by forward substitution (one warp each),
// T'_bb = D_b diag(beta_b), then E_bm = D_b A_bm for the six blocks below the
// diagonal, then the blocks of T' below the diagonal one subdiagonal at a time,
//   T'_bc = -sum_{c <= m < b} E_bm T'_mc,
// which is (I + A) T' = diag(beta) solved by blocks.
#include "mgs_tiles.cuh"
#include "mgs_umma.cuh"

namespace mgs {
namespace {

constexpr int DD = 64;               // head dimension (d_k = d_v)
constexpr int CH = 64;               // chunk length
constexpr int MATB = CH * DD * 4;    // bytes of a 64 x 64 fp32 matrix
constexpr int PANEL = CH * 128;      // bytes of one swizzled panel of 64 rows (32 floats each)
constexpr int LD = 68;               // row stride (floats) of the plain matrices of the solve
constexpr int DLD = 20;              // row stride of the 16 x 16 blocks (D_b, E_bm)
constexpr int WS_ROWS = 4 * CH;      // workspace rows (of 64 floats) per chunk: R, M, O_c^T, N^T
constexpr int kWyThreads = 256;      // eight warps: TMEM lane quarter w % 4, column half w / 4
constexpr int kStateThreads = 288;   // the same eight warps and one copy warp

// Shared memory of delta_wy_kernel (bytes from a 1024-byte aligned base).
//   [0, 32K)    K as a stacked B operand: panel p (16 KB) = [K residuals; K]
//               rows, for k = 32p .. 32p+31 (the TMA writes K into the second
//               half, the split writes the residuals beside it);
//   [32K, 48K)  Q;  [48K, 64K) V (swizzled 64 x 64);
//   [64K, ..)   A (plain, stride LD), D_b, E_bm, beta, barriers.
// Reused once dead: T' (plain) over K; T' as the stacked B operand of the
// second product over V and A; the third product's B operand [W^T; U^T]
// (128 rows, tf32 parts and residuals in two separate operands) over K and
// over V and A.  Q lives to the end (R = Q - P W).
struct WyLayout {
    static constexpr int kst = 0, q = 2 * MATB, v = 3 * MATB;
    static constexpr int a = 4 * MATB;
    static constexpr int dinv = a + CH * LD * 4;
    static constexpr int xs = dinv + CH * DLD * 4;
    static constexpr int beta = xs + 6 * 16 * DLD * 4;
    static constexpr int bars = beta + CH * 4;
    static constexpr int tplain = 0, t2 = v, b3b = 0, b3s = v;
    static constexpr int om = 0, oo = MATB, on = v;  // staged outputs M, O_c^T, N^T (R over Q)
    static constexpr size_t bytes = size_t(bars) + 64 + 1024;
};
static_assert(CH * LD * 4 <= 2 * MATB, "plain T' fits over K");
static_assert(WyLayout::t2 + 2 * MATB <= WyLayout::dinv, "stacked T' stays clear of D_b");
static_assert(WyLayout::b3s + 2 * MATB <= WyLayout::dinv, "third B operand stays clear of D_b");
static_assert(WyLayout::bars % 8 == 0, "barrier alignment");

// TMEM columns of delta_wy_kernel (256 allocated): the stacked products need
// 128 columns; the A operand's tf32 parts and residuals 64 each.
constexpr uint32_t kWyD = 0, kWyAB = 128, kWyAS = 192, kWyCols = 256;

// Shared memory of delta_state_kernel<NI>: NS stages of [R; M] (two swizzled
// panels of 128 rows) and the block's rows of O_c^T and N^T (NI x 64 each,
// swizzled, panels of NI rows); the B operand S as [S residuals; S] rows (two
// panels of 2 NI rows); then full[NS], empty[NS], the product barrier, the
// TMEM address and the abort word.
template <int NI>
struct StLayout {
    static constexpr int NS = NI == 64 ? 3 : NI == 32 ? 4 : 5;
    static constexpr int apanel = 2 * CH * 128;
    static constexpr int osl = 2 * apanel, nsl = osl + NI * DD * 4;
    static constexpr int stage = nsl + NI * DD * 4;
    static constexpr int bpanel = 2 * NI * 128, spanel = NI * 128;
    static constexpr int sb = NS * stage;
    static constexpr int bars = sb + 2 * bpanel;
    static constexpr size_t bytes = size_t(bars) + 8 * (2 * NS + 1) + 16 + 1024;
};

// TMEM columns of delta_state_kernel (all 512): two A operand buffers ([R; M]
// of consecutive chunks; tf32 parts and residuals), then the product (2 NI).
constexpr uint32_t kStCols = 512, kStD = 256;
__device__ __forceinline__ uint32_t st_abig(int b) { return uint32_t(128 * b); }
__device__ __forceinline__ uint32_t st_asmall(int b) { return uint32_t(128 * b + 64); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier among the eight compute warps only (the copy warp runs on its own).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// x = big + small, big = x rounded to tf32, small = x - big (exact)
__device__ __forceinline__ void split_tf32(float x, float &big, float &small) {
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(x));
    big = __uint_as_float(u);
    small = x - big;
}

// Columns 32h .. 32h+31 of row r of a swizzled tile whose panels (32 columns
// each) are `panel` bytes apart.
__device__ __forceinline__ void sw_row32(const unsigned char *m, int r, int h, int panel, float (&v)[32]) {
    const unsigned char *row = m + h * panel + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 x = *reinterpret_cast<const float4 *>(row + ((c ^ (r & 7)) << 4));
        v[4 * c] = x.x;
        v[4 * c + 1] = x.y;
        v[4 * c + 2] = x.z;
        v[4 * c + 3] = x.w;
    }
}

// Byte offset of element (row n, k) of a swizzled K-major operand whose two
// panels (k 0..31, 32..63) are `panel` bytes apart.
__device__ __forceinline__ uint32_t bop_off(int n, int k, int panel) {
    return uint32_t(k >> 5) * uint32_t(panel) + sw128_off(n, k & 31);
}

// 32 consecutive columns of this thread's TMEM lane: the tf32 parts at column
// cb, the residuals at cs (addresses relative to the warp's lanes); both
// stores in flight together, one wait.
__device__ __forceinline__ void tmem_put_split32(uint32_t tlanes, uint32_t cb, uint32_t cs, const float (&v)[32]) {
    float bg[32], rs[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) split_tf32(v[i], bg[i], rs[i]);
    tmem_st32x2(tlanes + cb, bg, tlanes + cs, rs);
}

// D (128 x N) = A B^T over k = 0..63 in three tf32 terms per multiply: A in
// TMEM (tf32 parts from column a_big, residuals from a_small, one column per
// k), B in shared memory as two swizzled K-major operands (parts at b_big,
// residuals at b_small, panels `panel` bytes apart).  Issued by one thread.
__device__ __forceinline__ void mma_split3(uint32_t d, uint32_t a_big, uint32_t a_small, uint32_t b_big,
                                           uint32_t b_small, uint32_t panel, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = uint32_t(kk >> 2) * panel + uint32_t(kk & 3) * 32u;
        const uint64_t db = umma_desc_sw128(b_big + off, 16u, 1024u);
        const uint64_t ds = umma_desc_sw128(b_small + off, 16u, 1024u);
        umma_tf32_ts(d, a_small + 8u * kk, db, idesc, kk > 0);
        umma_tf32_ts(d, a_big + 8u * kk, ds, idesc, true);
        umma_tf32_ts(d, a_big + 8u * kk, db, idesc, true);
    }
}

// As mma_split3 with B stored as [B_small; B_big] row blocks of n rows each
// (panels of 2n rows at b): D[:, 0:n) = A_big B_small^T and
// D[:, n:2n) = (A_big + A_small) B_big^T; the product is the sum of the two.
template <int n>
__device__ __forceinline__ void mma_split3_stacked(uint32_t d, uint32_t a_big, uint32_t a_small, uint32_t b) {
    constexpr uint32_t panel = 2 * n * 128;
    constexpr uint32_t id2 = umma_idesc_tf32(128, 2 * n), id1 = umma_idesc_tf32(128, n);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = uint32_t(kk >> 2) * panel + uint32_t(kk & 3) * 32u;
        umma_tf32_ts(d, a_big + 8u * kk, umma_desc_sw128(b + off, 16u, 1024u), id2, kk > 0);
        umma_tf32_ts(d + n, a_small + 8u * kk, umma_desc_sw128(b + off + n * 128u, 16u, 1024u), id1, true);
    }
}

// Sum of the two halves of a stacked product: columns c0 .. c0+NC-1 of the
// result (TMEM columns d + c0 .. and d + n + c0 ..).
template <int NC>
__device__ __forceinline__ void tmem_ld_stacked(uint32_t d, int n, int c0, float (&v)[NC]) {
    float w[NC];
    tmem_ld_pair<NC>(d + uint32_t(c0), v, d + uint32_t(n + c0), w);
#pragma unroll
    for (int i = 0; i < NC; ++i) v[i] += w[i];
}

// One block per chunk (chunks of a lane consecutive): R, M (row-major, rows t
// and j), O_c^T and N^T (rows i) of the chunk into the workspace, 256 rows of
// 64 floats per chunk, stored through the tensor map tmO.  Rows past the
// sequence end contribute nothing.
__global__ void __launch_bounds__(kWyThreads, 2)
    delta_wy_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const float *__restrict__ beta, int64_t B, int64_t T, int64_t H, DevCtl ctl) {
    using L = WyLayout;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = align_smem(smem_raw, 1024);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::bars);  // TMA, then the three products
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar + 4);
    volatile int *abort_word = reinterpret_cast<volatile int *>(slot + 1);
    float *Am = reinterpret_cast<float *>(sm + L::a), *Dv = reinterpret_cast<float *>(sm + L::dinv);
    float *Xs = reinterpret_cast<float *>(sm + L::xs), *sb = reinterpret_cast<float *>(sm + L::beta);
    float *Tm = reinterpret_cast<float *>(sm + L::tplain);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hh = warp >> 2, r = 32 * q4 + lane;  // TMEM lane (row of the stacked operands)
    const int64_t nch = (T + CH - 1) / CH;
    if (int64_t(blockIdx.x) >= B * H * nch) return;
    // 32-bit divisions (the grid, the chunk count and H are below 2^31)
    const int lane32 = int(blockIdx.x) / int(nch);
    const int64_t c = int64_t(blockIdx.x) - int64_t(lane32) * nch;
    const int bi = lane32 / int(H), hd = lane32 - bi * int(H);
    const int n = int(min64(CH, T - c * CH));
    const int row0 = int(int64_t(bi) * T + c * CH);

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        fence_barrier_init();
        *abort_word = 0;
    }
    if (warp == 0) {
        tmem_alloc(slot, kWyCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the state pass may be scheduled as soon as every block of this one has
    // started (it waits for this grid's completion before reading its output)
    pdl_trigger();
    const uint32_t tm = *slot;
    const uint32_t tq = tm + (uint32_t(32 * q4) << 16);
    if (tid == 0) {
        const uint64_t once = policy_evict_first();
        mbar_arrive_expect_tx(&bar[0], uint32_t(3 * MATB));
        for (int p = 0; p < 2; ++p) {
            tma_load_3d(sm + L::kst + p * 2 * PANEL + PANEL, &tmK, 32 * p, hd, row0, &bar[0], once);
            tma_load_3d(sm + L::q + p * PANEL, &tmQ, 32 * p, hd, row0, &bar[0], once);
            tma_load_3d(sm + L::v + p * PANEL, &tmV, 32 * p, hd, row0, &bar[0], once);
        }
    }
    if (tid < CH) sb[tid] = tid < n ? beta[(int64_t(row0) + tid) * H + hd] : 0.f;
    int issued = 0;  // products issued (thread 0)
    do {
        bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar[0], 0, ctl.timeout_ns));
        if (!ok && lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        __syncthreads();
        if (*abort_word != 0) break;
        // rows past the sequence end (the next sequence's, or fill) contribute nothing
        if (n < CH) {
            const int per = (CH - n) * 32;
            for (int e = tid; e < 2 * per; e += kWyThreads) {
                const int p = e / per, rowoff = n * 128 + (e - p * per) * 4;
                *reinterpret_cast<float *>(sm + L::kst + p * 2 * PANEL + PANEL + rowoff) = 0.f;
                *reinterpret_cast<float *>(sm + L::q + p * PANEL + rowoff) = 0.f;
                *reinterpret_cast<float *>(sm + L::v + p * PANEL + rowoff) = 0.f;
            }
            __syncthreads();
        }
        // [K; Q] into TMEM (thread: row r, columns 32 hh ..); K as the first
        // product's stacked B operand: tf32 parts in place, residuals in the
        // panel's first half (each thread rewrites exactly the elements it read)
        {
            float v[32];
            if (r < 64)
                sw_row32(sm + L::kst + PANEL, r, hh, 2 * PANEL, v);
            else
                sw_row32(sm + L::q, r - 64, hh, PANEL, v);
            tmem_put_split32(tq, kWyAB + 32 * hh, kWyAS + 32 * hh, v);
            if (r < 64) {
                unsigned char *ks = sm + L::kst + hh * 2 * PANEL + r * 128, *kb = ks + PANEL;
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    float4 b4, s4;
                    split_tf32(v[4 * c4], b4.x, s4.x);
                    split_tf32(v[4 * c4 + 1], b4.y, s4.y);
                    split_tf32(v[4 * c4 + 2], b4.z, s4.z);
                    split_tf32(v[4 * c4 + 3], b4.w, s4.w);
                    const int o = (c4 ^ (r & 7)) << 4;
                    *reinterpret_cast<float4 *>(kb + o) = b4;
                    *reinterpret_cast<float4 *>(ks + o) = s4;
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            mma_split3_stacked<CH>(tm + kWyD, tm + kWyAB, tm + kWyAS, smem_addr(sm + L::kst));
            umma_commit(&bar[1]);
            ++issued;
        }
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar[1], 0, ctl.timeout_ns));
        tc_fence_after();
        float prow[32];  // rows 64..: P = tril(Q K^T), row t = r - 64, columns 32 hh .. (kept for the third product)
        if (ok) {
            // rows 0..63: A = strict_tril(diag(beta) K K^T) (plain, for the solve)
            float d[32];
            tmem_ld_stacked<32>(tq + kWyD, CH, 32 * hh, d);
            const int t = r & 63;
            if (r < 64) {
                const float bt = sb[t];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    float4 a4;
                    const int s0 = 32 * hh + 4 * c4;
                    a4.x = s0 < t ? bt * d[4 * c4] : 0.f;
                    a4.y = s0 + 1 < t ? bt * d[4 * c4 + 1] : 0.f;
                    a4.z = s0 + 2 < t ? bt * d[4 * c4 + 2] : 0.f;
                    a4.w = s0 + 3 < t ? bt * d[4 * c4 + 3] : 0.f;
                    *reinterpret_cast<float4 *>(Am + t * LD + s0) = a4;
                }
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) prow[u] = 32 * hh + u <= t ? d[u] : 0.f;
            }
            // [K^T; V^T] into TMEM over the first product's operand (complete):
            // row r < 64 is column r of K (parts + residuals = K exactly), row
            // 64 + j column j of V
            float v[32];
            if (r < 64) {
                const unsigned char *ps = sm + L::kst + (r >> 5) * 2 * PANEL, *pk = ps + PANEL;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const uint32_t off = sw128_off(32 * hh + u, r & 31);
                    v[u] = *reinterpret_cast<const float *>(pk + off) + *reinterpret_cast<const float *>(ps + off);
                }
            } else {
                const unsigned char *pv = sm + L::v + ((r - 64) >> 5) * PANEL;
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    v[u] = *reinterpret_cast<const float *>(pv + sw128_off(32 * hh + u, (r - 64) & 31));
            }
            tmem_put_split32(tq, kWyAB + 32 * hh, kWyAS + 32 * hh, v);
        } else if (lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        tc_fence_before();
        __syncthreads();
        if (*abort_word != 0) break;
        // Solve, phase 1.  Warps 0-3: D_b = (I + A_bb)^{-1}, b = warp, lane j < 16
        // builds column j by forward substitution; T'_bb = D_b diag(beta_b).  The
        // column is kept in registers and stored after it is complete, so that no
        // shared store sits between the loads of the chain.
        if (warp < 4 && lane < 16) {
            const int b0 = 16 * warp;
            float dcol[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                float arow[16];
#pragma unroll
                for (int qq = 0; qq < rr; qq += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Am + (b0 + rr) * LD + b0 + qq);
                    arow[qq] = a4.x;
                    arow[qq + 1] = a4.y;
                    arow[qq + 2] = a4.z;
                    arow[qq + 3] = a4.w;
                }
                float acc = (rr == lane) ? 1.f : 0.f;
#pragma unroll
                for (int qq = 0; qq < rr; ++qq) acc = fmaf(-arow[qq], dcol[qq], acc);
                dcol[rr] = acc;
            }
            const float bj = sb[b0 + lane];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                Dv[(b0 + rr) * DLD + lane] = dcol[rr];
                Tm[(b0 + rr) * LD + b0 + lane] = dcol[rr] * bj;
            }
        }
        __syncthreads();
        // Solve, phase 2.  E_bm = D_b A_bm for the six blocks below the diagonal
        // (pair j = b(b-1)/2 + m), then T'_bc = -sum_{c <= m < b} E_bm T'_mc one
        // subdiagonal d = b - c at a time.  Thread: element (tid / 16, tid % 16)
        // of every block of the step.
        const int er = tid >> 4, ec = tid & 15;
        {
            float acc[6];
#pragma unroll
            for (int j = 0; j < 6; ++j) acc[j] = 0.f;
#pragma unroll
            for (int qq = 0; qq < 16; qq += 4) {
#pragma unroll
                for (int j = 0; j < 6; ++j) {
                    const int b = j < 1 ? 1 : j < 3 ? 2 : 3, m = j - b * (b - 1) / 2;
                    const float4 d4 = *reinterpret_cast<const float4 *>(Dv + (16 * b + er) * DLD + qq);
                    const float *a = Am + (16 * b + qq) * LD + 16 * m + ec;
                    acc[j] = fmaf(d4.x, a[0], acc[j]);
                    acc[j] = fmaf(d4.y, a[LD], acc[j]);
                    acc[j] = fmaf(d4.z, a[2 * LD], acc[j]);
                    acc[j] = fmaf(d4.w, a[3 * LD], acc[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 6; ++j) Xs[(16 * j + er) * DLD + ec] = acc[j];
        }
        __syncthreads();
#pragma unroll
        for (int dg = 1; dg < 4; ++dg) {
            float acc[3];
#pragma unroll
            for (int cb = 0; cb < 3; ++cb) acc[cb] = 0.f;
#pragma unroll
            for (int cb = 0; cb < 4 - dg; ++cb) {
                const int b = cb + dg;
#pragma unroll
                for (int m = cb; m < b; ++m) {
                    const float *e = Xs + (16 * (b * (b - 1) / 2 + m) + er) * DLD;
                    const float *tt = Tm + 16 * m * LD + 16 * cb + ec;
#pragma unroll
                    for (int qq = 0; qq < 16; qq += 4) {
                        const float4 e4 = *reinterpret_cast<const float4 *>(e + qq);
                        acc[cb] = fmaf(e4.x, tt[(qq + 0) * LD], acc[cb]);
                        acc[cb] = fmaf(e4.y, tt[(qq + 1) * LD], acc[cb]);
                        acc[cb] = fmaf(e4.z, tt[(qq + 2) * LD], acc[cb]);
                        acc[cb] = fmaf(e4.w, tt[(qq + 3) * LD], acc[cb]);
                    }
                }
            }
#pragma unroll
            for (int cb = 0; cb < 4 - dg; ++cb) Tm[(16 * (cb + dg) + er) * LD + 16 * cb + ec] = -acc[cb];
            __syncthreads();
        }
        // T' as the second product's stacked B operand (rows t, k = s; zero
        // above the diagonal): panel p = [T' residuals; T'] rows
        {
            const int t = tid >> 2, s0 = 16 * (tid & 3);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int s = s0 + 4 * c4;
                const float4 x = *reinterpret_cast<const float4 *>(Tm + t * LD + s);
                float4 bg, rs;
                split_tf32(s <= t ? x.x : 0.f, bg.x, rs.x);
                split_tf32(s + 1 <= t ? x.y : 0.f, bg.y, rs.y);
                split_tf32(s + 2 <= t ? x.z : 0.f, bg.z, rs.z);
                split_tf32(s + 3 <= t ? x.w : 0.f, bg.w, rs.w);
                const uint32_t off = bop_off(t, s, 2 * PANEL);
                *reinterpret_cast<float4 *>(sm + L::t2 + off) = rs;
                *reinterpret_cast<float4 *>(sm + L::t2 + PANEL + off) = bg;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            mma_split3_stacked<CH>(tm + kWyD, tm + kWyAB, tm + kWyAS, smem_addr(sm + L::t2));
            umma_commit(&bar[2]);
            ++issued;
        }
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar[2], 0, ctl.timeout_ns));
        tc_fence_after();
        if (ok) {
            // [W^T; U^T] (row r: W^T row r, or U^T row r - 64; k = t) as the
            // third product's B operand, tf32 parts and residuals apart
            float d[32];
            tmem_ld_stacked<32>(tq + kWyD, CH, 32 * hh, d);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                float4 bg, rs;
                split_tf32(d[4 * c4], bg.x, rs.x);
                split_tf32(d[4 * c4 + 1], bg.y, rs.y);
                split_tf32(d[4 * c4 + 2], bg.z, rs.z);
                split_tf32(d[4 * c4 + 3], bg.w, rs.w);
                const uint32_t off = bop_off(r, 32 * hh + 4 * c4, 2 * PANEL);
                *reinterpret_cast<float4 *>(sm + L::b3b + off) = bg;
                *reinterpret_cast<float4 *>(sm + L::b3s + off) = rs;
            }
            // [K^T; P]: rows 64.. take P in place of V^T (the second product is done)
            if (r >= 64) tmem_put_split32(tq, kWyAB + 32 * hh, kWyAS + 32 * hh, prow);
        } else if (lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*abort_word != 0) break;
        if (tid == 0) {
            tc_fence_after();
            mma_split3(tm + kWyD, tm + kWyAB, tm + kWyAS, smem_addr(sm + L::b3b), smem_addr(sm + L::b3s), 2 * PANEL,
                       umma_idesc_tf32(128, 2 * CH));
            umma_commit(&bar[3]);
            ++issued;
        }
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar[3], 0, ctl.timeout_ns));
        tc_fence_after();
        if (ok) {
            // columns 0..63: rows j: M = I - K^T W; rows t: R = Q - P W.
            // columns 64..127: rows j: N = K^T U (kept as N^T); rows t: O_c = P U (as O_c^T).
            // Staged in shared memory as swizzled 64 x 64 tiles (R in place of Q),
            // then stored by TMA.
            float d1[32], d2[32];
            tmem_ld_pair<32>(tq + kWyD + 32 * hh, d1, tq + kWyD + CH + 32 * hh, d2);
            const int rr = r & 63;
            if (r < 64) {
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const int k0 = 32 * hh + 4 * c4;
                    *reinterpret_cast<float4 *>(sm + L::om + bop_off(rr, k0, PANEL)) =
                        make_float4((k0 == rr ? 1.f : 0.f) - d1[4 * c4], (k0 + 1 == rr ? 1.f : 0.f) - d1[4 * c4 + 1],
                                    (k0 + 2 == rr ? 1.f : 0.f) - d1[4 * c4 + 2],
                                    (k0 + 3 == rr ? 1.f : 0.f) - d1[4 * c4 + 3]);
                }
            } else {
                float qv[32];
                sw_row32(sm + L::q, rr, hh, PANEL, qv);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4)
                    *reinterpret_cast<float4 *>(sm + L::q + bop_off(rr, 32 * hh + 4 * c4, PANEL)) =
                        make_float4(qv[4 * c4] - d1[4 * c4], qv[4 * c4 + 1] - d1[4 * c4 + 1],
                                    qv[4 * c4 + 2] - d1[4 * c4 + 2], qv[4 * c4 + 3] - d1[4 * c4 + 3]);
            }
            // N^T[i][j] (rows j) or O_c^T[i][t] (rows t): the warp's 32 lanes fill
            // 32 consecutive floats of each row i
            unsigned char *tb = sm + (r < 64 ? L::on : L::oo);
#pragma unroll
            for (int u = 0; u < 32; ++u) *reinterpret_cast<float *>(tb + bop_off(32 * hh + u, rr, PANEL)) = d2[u];
        } else if (lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (*abort_word != 0) break;
        if (tid == 0) {
            const int row = int(blockIdx.x) * WS_ROWS;
            for (int p = 0; p < 2; ++p) {
                tma_store_2d(&tmO, 32 * p, row, sm + L::q + p * PANEL);
                tma_store_2d(&tmO, 32 * p, row + CH, sm + L::om + p * PANEL);
                tma_store_2d(&tmO, 32 * p, row + 2 * CH, sm + L::oo + p * PANEL);
                tma_store_2d(&tmO, 32 * p, row + 3 * CH, sm + L::on + p * PANEL);
            }
            bulk_commit();
            bulk_wait_read();
        }
    } while (false);
    // copies and products this block started are complete before its shared
    // memory and TMEM are released (at once, unless a wait above gave up)
    if (tid == 0) {
        bool d = mbar_wait_bounded(&bar[0], 0, ctl.timeout_ns);
        for (int i = 0; i < issued; ++i) d = mbar_wait_bounded(&bar[1 + i], 0, ctl.timeout_ns) && d;
        if (!d) record_error(ctl, ERR_DRAIN_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, kWyCols);
    }
}

// Column j of the stacked B operand S (rows i = c0 .. c0 + HC - 1 of the
// block's NI: residuals in rows i, tf32 parts in rows NI + i).
template <int NI, int HC>
__device__ __forceinline__ void put_state(unsigned char *Sst, const float (&s)[HC], int j, int c0) {
#pragma unroll
    for (int u = 0; u < HC; ++u) {
        float bg, rs;
        split_tf32(s[u], bg, rs);
        const uint32_t off = bop_off(c0 + u, j, 2 * NI * 128);
        *reinterpret_cast<float *>(Sst + off) = rs;
        *reinterpret_cast<float *>(Sst + NI * 128 + off) = bg;
    }
}

// One block per (lane, NI value columns i0..): walks the lane's chunks in
// order holding S^T[:, i0..] in registers (thread: one row j, NI / 2 columns)
// and S[i0.., :] as the product's B operand.  Per chunk c:
//   1. [R; M] of chunk c + 1 into TMEM (the other buffer) while the product
//      of chunk c runs;
//   2. product done: O = R S^T + O_c (rows t) to memory, S^T = M S^T + N
//      (rows j) and the B operand;
//   3. the product of chunk c + 1 issued.
// Warp 8 is the copy warp: it refills a stage by TMA once all eight compute
// warps have arrived on its "empty" barrier (after their last read of it).
template <int NI>
__global__ void __launch_bounds__(kStateThreads, 1)
    delta_state_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmS,
                       const float *__restrict__ S0, float *__restrict__ o, float *__restrict__ ST_out, int64_t B,
                       int64_t T, int64_t H, DevCtl ctl) {
    using L = StLayout<NI>;
    constexpr int NS = L::NS, NVB = DD / NI, HC = NI / 2;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = align_smem(smem_raw, 1024);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::bars), *empty = full + NS, *bar_m = full + 2 * NS;
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar_m + 1);
    volatile int *abort_word = reinterpret_cast<volatile int *>(slot + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t blk = blockIdx.x;
    if (blk >= B * H * NVB) return;
    const int lane_id = int(blk / NVB), i0 = int(blk % NVB) * NI;  // 32-bit: lanes < 2^31
    const int bi = lane_id / int(H), hd = lane_id - bi * int(H);
    const int64_t nch = (T + CH - 1) / CH;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWyThreads / 32);
        }
        mbar_init(bar_m, 1);
        fence_barrier_init();
        *abort_word = 0;
    }
    if (warp == 0) {
        tmem_alloc(slot, kStCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *slot;

    if (warp == kWyThreads / 32) {  // the copy warp
        if (lane == 0) {
            // the lane's state blocks read the same [R; M]
            const uint64_t pol = policy_evict_normal();
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmS);
            // launched as a programmatic dependent of the WY pass: its output is
            // complete and visible after this wait
            pdl_wait();
            int64_t last = -1;
            for (int64_t c = 0; c < nch; ++c) {
                const int s = int(c % NS);
                if (c >= NS) {
                    // The abort word is written only by compute warps, before a
                    // barrier of theirs, so that all eight read the same value
                    // after it; this warp just stops issuing, and their bounded
                    // waits for the missing stage give up together.
                    const bool ok = mbar_wait_bounded(&empty[s], uint32_t(((c - NS) / NS) & 1), ctl.timeout_ns);
                    if (!ok) record_error(ctl, ERR_MBAR_TIMEOUT);
                    if (!ok || *abort_word != 0) break;
                }
                unsigned char *st = sm + s * L::stage;
                const int wr = int((int64_t(lane_id) * nch + c) * WS_ROWS);  // workspace row of the chunk's R
                mbar_arrive_expect_tx(&full[s], uint32_t(L::stage));
                tma_load_2d(st, &tmA, 0, wr, &full[s], pol);
                tma_load_2d(st + L::apanel, &tmA, 32, wr, &full[s], pol);
                for (int p = 0; p < 2; ++p) {
                    tma_load_2d(st + L::osl + p * L::spanel, &tmS, 32 * p, wr + 2 * CH + i0, &full[s], pol);
                    tma_load_2d(st + L::nsl + p * L::spanel, &tmS, 32 * p, wr + 3 * CH + i0, &full[s], pol);
                }
                last = c;
            }
            // the block's shared memory outlives every copy this warp started
            bool ok = true;
            for (int64_t c = last - NS + 1; c <= last; ++c)
                if (c >= 0 && !mbar_wait_bounded(&full[c % NS], uint32_t((c / NS) & 1), ctl.timeout_ns)) ok = false;
            if (!ok) record_error(ctl, ERR_DRAIN_TIMEOUT);
        }
        return;
    }

    const int q4 = warp & 3, hh = warp >> 2, r = 32 * q4 + lane;  // TMEM lane (row of [R; M])
    const uint32_t tq = tm + (uint32_t(32 * q4) << 16);
    const bool lower = q4 >= 2;  // rows 64..: M S^T (the state); else R S^T (the output)
    const int c0 = hh * HC;      // this thread's first column of the block's NI
    unsigned char *Sst = sm + L::sb;
    const uint32_t aS = smem_addr(Sst);
    float hold[HC];  // lower: S^T[j][i0 + c0 + u], j = r - 64
    if (lower) {
        const int j = r - 64;
#pragma unroll
        for (int u = 0; u < HC; ++u)
            hold[u] = S0 != nullptr ? S0[int64_t(lane_id) * DD * DD + int64_t(i0 + c0 + u) * DD + j] : 0.f;
        put_state<NI, HC>(Sst, hold, j, c0);
    }
    fence_proxy_async_smem();
    // [R; M] row r of the stage's chunk into TMEM buffer b
    auto put_a = [&](const unsigned char *st, int b) {
        float v[32];
        sw_row32(st, r, hh, L::apanel, v);
        tmem_put_split32(tq, st_abig(b) + 32 * hh, st_asmall(b) + 32 * hh, v);
    };
    int nm = 0;  // products issued (thread 0)
    {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[0], 0, ctl.timeout_ns));
        if (ok)
            put_a(sm, 0);
        else if (lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        tc_fence_before();
        compute_sync();
    }
    if (*abort_word == 0 && tid == 0) {
        tc_fence_after();
        mma_split3_stacked<NI>(tm + kStD, tm + st_abig(0), tm + st_asmall(0), aS);
        umma_commit(bar_m);
        ++nm;
    }
    for (int64_t c = 0; c < nch && *abort_word == 0; ++c) {
        const int s = int(c % NS), b = int(c & 1);
        const unsigned char *st = sm + s * L::stage;
        const int n = int(min64(CH, T - c * CH));
        // 1. the next chunk's [R; M] into the other buffer (its reader, the
        // product of chunk c - 1, is done)
        bool ok1 = true;
        if (c + 1 < nch) {
            const int s1 = int((c + 1) % NS);
            ok1 = __all_sync(0xffffffffu,
                             mbar_wait_bounded(&full[s1], uint32_t(((c + 1) / NS) & 1), ctl.timeout_ns));
            if (ok1) put_a(sm + s1 * L::stage, b ^ 1);
        }
        // 2. the product of chunk c: O = R S^T + O_c (rows t = r < n), S^T = M S^T + N
        const bool ok2 = __all_sync(0xffffffffu, mbar_wait_bounded(bar_m, uint32_t(c & 1), ctl.timeout_ns));
        tc_fence_after();
        if (ok2) {
            float x[HC];
            tmem_ld_stacked<HC>(tq + kStD, NI, c0, x);
            if (lower) {
                const int j = r - 64;
                const unsigned char *nt = st + L::nsl;
#pragma unroll
                for (int u = 0; u < HC; ++u)
                    hold[u] = x[u] + *reinterpret_cast<const float *>(nt + bop_off(c0 + u, j, L::spanel));
                put_state<NI, HC>(Sst, hold, j, c0);
            } else if (r < n) {
                const unsigned char *ot = st + L::osl;
                float *dst = o + ((int64_t(bi) * T + c * CH + r) * H + hd) * DD + i0 + c0;
                auto oc = [&](int u) { return *reinterpret_cast<const float *>(ot + bop_off(c0 + u, r, L::spanel)); };
#pragma unroll
                for (int u = 0; u < HC; u += 4)
                    *reinterpret_cast<float4 *>(dst + u) =
                        make_float4(x[u] + oc(u), x[u + 1] + oc(u + 1), x[u + 2] + oc(u + 2), x[u + 3] + oc(u + 3));
            }
        }
        if ((!ok1 || !ok2) && lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp's last read of the stage is done
        compute_sync();
        if (*abort_word != 0) break;
        // 3. the next chunk's product (its operands: the buffer written in 1,
        // the state written in 2, both ordered by the barrier)
        if (c + 1 < nch && tid == 0) {
            tc_fence_after();
            mma_split3_stacked<NI>(tm + kStD, tm + st_abig(b ^ 1), tm + st_asmall(b ^ 1), aS);
            umma_commit(bar_m);
            ++nm;
        }
    }
    if (*abort_word == 0 && ST_out != nullptr && lower) {
        const int j = r - 64;
#pragma unroll
        for (int u = 0; u < HC; ++u) ST_out[int64_t(lane_id) * DD * DD + int64_t(i0 + c0 + u) * DD + j] = hold[u];
    }
    // a product still in flight after a failed wait completes before TMEM is freed
    if (tid == 0 && nm > 0 && !mbar_wait_bounded(bar_m, uint32_t((nm - 1) & 1), ctl.timeout_ns))
        record_error(ctl, ERR_DRAIN_TIMEOUT);
    tc_fence_before();
    compute_sync();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, kStCols);
    }
}

// [rows][H][64] floats, boxes of 32 x 1 x 64 with 128-byte swizzle (two boxes
// per 64-row chunk: columns 0..31 and 32..63).
cudaError_t make_chunk_map(CUtensorMap *m, const float *base, int64_t rows, int64_t H) {
    const uint64_t dims[3] = {uint64_t(DD), uint64_t(H), uint64_t(rows)};
    const uint64_t str[2] = {uint64_t(DD) * 4u, uint64_t(H) * DD * 4u};
    const uint32_t box[3] = {32u, 1u, uint32_t(CH)};
    return make_tmap(m, base, 3, dims, str, box, true);
}

// The workspace as rows of 64 floats (R, M, O_c^T, N^T of every chunk),
// boxes of box_x x box_y floats.
cudaError_t make_ws_map(CUtensorMap *m, const float *ws, int64_t rows, int box_x, int box_y, bool swizzle) {
    const uint64_t dims[2] = {uint64_t(DD), uint64_t(rows)};
    const uint64_t str[1] = {uint64_t(DD) * 4u};
    const uint32_t box[2] = {uint32_t(box_x), uint32_t(box_y)};
    return make_tmap(m, ws, 2, dims, str, box, swizzle);
}

template <int NI>
cudaError_t launch_state(float *w, int64_t chunks, const float *S0, float *o, float *ST, int64_t B, int64_t T,
                         int64_t H, const DevCtl &ctl, cudaStream_t s) {
    constexpr int NVB = DD / NI;
    CUtensorMap tA, tS;
    cudaError_t e;
    if ((e = make_ws_map(&tA, w, chunks * WS_ROWS, 32, 2 * CH, true)) != cudaSuccess) return e;
    if ((e = make_ws_map(&tS, w, chunks * WS_ROWS, 32, NI, true)) != cudaSuccess) return e;
    const int smem = int(StLayout<NI>::bytes);
    if ((e = ensure_smem_attr((const void *)delta_state_kernel<NI>, smem)) != cudaSuccess) return e;
    // programmatic dependent launch: the blocks set up (barriers, TMEM, the
    // initial state) while the WY pass finishes; the copy warp waits for it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(B * H * NVB));
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, delta_state_kernel<NI>, tA, tS, S0, o, ST, B, T, H, ctl);
}

}  // namespace

size_t delta_workspace_bytes(int64_t B, int64_t T, int64_t H) {
    return size_t(B) * size_t(H) * size_t((T + CH - 1) / CH) * WS_ROWS * DD * sizeof(float);
}

cudaError_t launch_delta_fwd(const float *q, const float *k, const float *v, const float *beta, const float *S0,
                             float *o, float *ST, int64_t B, int64_t T, int64_t H, void *ws, const DevCtl &ctl,
                             cudaStream_t s) {
    const int64_t nch = (T + CH - 1) / CH, chunks = B * H * nch, lanes = B * H;
    if (chunks > 0x7fffffff / WS_ROWS || lanes * 4 > 0x7fffffff) return cudaErrorInvalidConfiguration;
    if (chunks == 0) return cudaSuccess;
    float *w = static_cast<float *>(ws);
    CUtensorMap tQ, tK, tV;
    cudaError_t e;
    if ((e = make_chunk_map(&tQ, q, B * T, H)) != cudaSuccess) return e;
    if ((e = make_chunk_map(&tK, k, B * T, H)) != cudaSuccess) return e;
    if ((e = make_chunk_map(&tV, v, B * T, H)) != cudaSuccess) return e;
    const int smem_a = int(WyLayout::bytes);
    if ((e = ensure_smem_attr((const void *)delta_wy_kernel, smem_a)) != cudaSuccess) return e;
    CUtensorMap tO;
    if ((e = make_ws_map(&tO, w, chunks * WS_ROWS, 32, CH, true)) != cudaSuccess) return e;
    delta_wy_kernel<<<dim3(unsigned(chunks)), kWyThreads, smem_a, s>>>(tQ, tK, tV, tO, beta, B, T, H, ctl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // State blocks as wide as the lane count allows while still giving about
    // one block per SM (each block splits the lane's whole [R; M] into TMEM,
    // so wide blocks do the least of that per column; narrow ones give more
    // blocks when lanes are few).
    if (lanes >= 152) return launch_state<64>(w, chunks, S0, o, ST, B, T, H, ctl, s);
    if (lanes >= 76) return launch_state<32>(w, chunks, S0, o, ST, B, T, H, ctl, s);
    return launch_state<16>(w, chunks, S0, o, ST, B, T, H, ctl, s);
}

}  // namespace mgs
