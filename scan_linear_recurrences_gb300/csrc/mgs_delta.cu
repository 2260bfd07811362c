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
// the chunk's rank-one updates).  W, U and P depend on the chunk's inputs
// only, so they are formed for every chunk at once (delta_wy_kernel, one
// block per chunk); only the last three lines carry the state from chunk to
// chunk.  Those lines act on each value index i (row i of S, column i of U',
// O) separately, so the state pass (delta_state_kernel) splits every lane
// into blocks of 8, 16, 32 or 64 value columns (narrower when lanes are few,
// so that more blocks run) that walk the lane's chunks in order, each holding
// its slice of S^T.
//
// [W | U] = T' [K | V] with T' = (I + A)^{-1} diag(beta), lower triangular.
// T' is formed by 16 x 16 blocks: the diagonal blocks D_b = (I + A_bb)^{-1}
// by forward substitution (one warp each), T'_bb = D_b diag(beta_b), then
// E_bm = D_b A_bm for the six blocks below the diagonal, then the blocks of
// T' below the diagonal one subdiagonal at a time,
//   T'_bc = -sum_{c <= m < b} E_bm T'_mc,
// which is (I + A) T' = diag(beta) solved by blocks.  Q, K, V (and in the
// state pass W, P and the slice of U) arrive by tiled TMA loads; a box
// wider than the 64-float rows leaves the last floats of every shared row as
// the tensor map's zero fill, a padded layout that keeps the products' shared
// reads free of bank conflicts.  The 64 x 64 products run on the tensor cores
// (mma.sync tf32 with a three-term split for fp32 accuracy); the small
// triangular blocks on the fp32 pipes.
#include "mgs_tiles.cuh"

namespace mgs {
namespace {

constexpr int DD = 64;         // head dimension (d_k = d_v)
constexpr int CH = 64;         // chunk length
constexpr int LD = 68;         // padded row stride (floats)
constexpr int MATF = CH * LD;  // floats per padded 64 x 64 matrix
constexpr int kThreads = 256;
constexpr int kStages = 3;      // at most this many chunks in flight in the state pass
constexpr int DLD = 20;         // row stride of the 16 x 16 blocks (D_b, level sums)
constexpr int WSM = CH * DD;    // floats of one stored 64 x 64 matrix (W, U or P)

// State blocks of NT n-tiles (8 NT value columns); the shared stride of their
// 64 x 8 NT operands is 8 mod 32 floats, so that a fragment's reads
// (rows k0 + q, columns g) fall in 32 different banks.
template <int NT>
struct StateCols {
    static constexpr int VS = 8 * NT;
    static constexpr int LDB = NT == 1 ? 8 : VS + 8;
};

// Shared memory of delta_wy_kernel (floats): Q, K, V, A, T' (padded
// 64 x 68), D (64 x DLD: rows 16b..16b+15, columns 0..15), E (6 blocks of
// 16 x DLD, block b(b-1)/2 + m holding E_bm), beta (64), the barrier and the
// abort word.
struct WySmem {
    static constexpr int q = 0;
    static constexpr int k = MATF;
    static constexpr int v = 2 * MATF;
    static constexpr int a = 3 * MATF;
    static constexpr int t = 4 * MATF;
    static constexpr int dinv = 5 * MATF;
    static constexpr int xs = dinv + CH * DLD;
    static constexpr int beta = xs + 6 * 16 * DLD;
    static constexpr int bars = beta + CH;  // 8-byte aligned (all offsets are multiples of 4 floats)
    static constexpr size_t bytes = size_t(bars) * 4 + sizeof(uint64_t) + 16;
};

// Shared memory of delta_state_kernel (floats): nst stages of [W P Q K]
// (padded 64 x 68) and the block's columns of U (64 x LDB); the block's slice
// of S^T (64 x LDB, key-major), U' (64 x LDB), then kStages "full" and
// kStages "empty" barriers and the abort word.
struct StateSmem {
    int stage, st, up, bars;
    size_t bytes;
    __host__ __device__ StateSmem(int nst, int ldb) {
        stage = 4 * MATF + CH * ldb;
        st = nst * stage;
        up = st + DD * ldb;
        bars = up + CH * ldb;
        bytes = size_t(bars) * 4 + 2 * kStages * sizeof(uint64_t) + 16;
    }
};

constexpr int kStateThreads = kThreads + 32;  // eight compute warps and one copy warp

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier among the eight compute warps only (the copy warp runs on its own).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kThreads) : "memory"); }

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- 64 x 64 x 64 products on the tensor cores (mma.sync m16n8k8, tf32).
// fp32 accuracy from three tf32 products per multiply: with x = xb + xs
// (xb = x rounded to tf32, xs = the rest rounded to tf32),
// a b ~ as bb + ab bs + ab bb (the as bs term is below fp32 resolution).
// Fragment layout of m16n8k8 (g = lane / 4, q = lane % 4):
//   A (16 x 8, row):  a0 (g, q)  a1 (g+8, q)  a2 (g, q+4)  a3 (g+8, q+4)
//   B (8 x 8, col):   b0 (q, g)  b1 (q+4, g)
//   C (16 x 8):       c0 (g, 2q) c1 (g, 2q+1) c2 (g+8, 2q) c3 (g+8, 2q+1)
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void split_tf32(float x, uint32_t &big, uint32_t &small) {
    big = to_tf32(x);
    small = to_tf32(x - __uint_as_float(big));
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc[nt] += op(A)[m0.., :] op(B)[:, n0 + 8 nt ..] over k = 0..63 for one
// warp's 16 x (8 NT) block of the result.  AT = false: A row-major [m][k];
// AT = true: A stored [k][m].  BT = false: B row-major [k][n]; BT = true: B
// stored [n][k].  Stride LD.  Only k < kend and n-tiles nt < ntl take part
// (the zero triangles of the masked products are skipped; both limits are
// warp-uniform).
template <bool AT, int NT, bool BT = false>
__device__ __forceinline__ void mma64(const float *__restrict__ A, const float *__restrict__ B, float (&acc)[NT][4],
                                      int m0, int n0, int lane, int kend = DD, int ntl = NT) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll 2
    for (int k0 = 0; k0 < kend; k0 += 8) {
        float av[4];
        if constexpr (AT) {
            av[0] = A[(k0 + q) * LD + m0 + g];
            av[1] = A[(k0 + q) * LD + m0 + g + 8];
            av[2] = A[(k0 + q + 4) * LD + m0 + g];
            av[3] = A[(k0 + q + 4) * LD + m0 + g + 8];
        } else {
            av[0] = A[(m0 + g) * LD + k0 + q];
            av[1] = A[(m0 + g + 8) * LD + k0 + q];
            av[2] = A[(m0 + g) * LD + k0 + q + 4];
            av[3] = A[(m0 + g + 8) * LD + k0 + q + 4];
        }
        uint32_t ab[4], as[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_tf32(av[i], ab[i], as[i]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (nt >= ntl) break;
            const int n = n0 + 8 * nt + g;
            uint32_t bb[2], bs[2];
            if constexpr (BT) {
                split_tf32(B[n * LD + k0 + q], bb[0], bs[0]);
                split_tf32(B[n * LD + k0 + q + 4], bb[1], bs[1]);
            } else {
                split_tf32(B[(k0 + q) * LD + n], bb[0], bs[0]);
                split_tf32(B[(k0 + q + 4) * LD + n], bb[1], bs[1]);
            }
            mma_tf32(acc[nt], as, bb);
            mma_tf32(acc[nt], ab, bs);
            mma_tf32(acc[nt], ab, bb);
        }
    }
}

// acc[nt] += op(A)[m0.., 0..kend) B[0..kend, 8 nt..] for one warp's
// 16 x 8 NT block, A as in mma64 (stride LD), B row-major [k][n] of stride
// LDB.  With a single n-tile the three terms of the split go to three
// accumulators (shorter dependency chains), summed at the end.
template <bool AT, int NT, int LDB>
__device__ __forceinline__ void mma_tile(const float *__restrict__ A, const float *__restrict__ B,
                                         float (&acc)[NT][4], int m0, int lane, int kend = DD) {
    const int g = lane >> 2, q = lane & 3;
    constexpr int NA = NT == 1 ? 3 : 1;
    float c[NA][NT][4];
#pragma unroll
    for (int t = 0; t < NA; ++t)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) c[t][nt][e] = 0.f;
#pragma unroll(NT > 2 ? 2 : 8)
    for (int k0 = 0; k0 < DD; k0 += 8) {
        if (k0 >= kend) break;
        float av[4];
        if constexpr (AT) {
            av[0] = A[(k0 + q) * LD + m0 + g];
            av[1] = A[(k0 + q) * LD + m0 + g + 8];
            av[2] = A[(k0 + q + 4) * LD + m0 + g];
            av[3] = A[(k0 + q + 4) * LD + m0 + g + 8];
        } else {
            av[0] = A[(m0 + g) * LD + k0 + q];
            av[1] = A[(m0 + g + 8) * LD + k0 + q];
            av[2] = A[(m0 + g) * LD + k0 + q + 4];
            av[3] = A[(m0 + g + 8) * LD + k0 + q + 4];
        }
        uint32_t ab[4], as[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_tf32(av[i], ab[i], as[i]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint32_t bb[2], bs[2];
            split_tf32(B[(k0 + q) * LDB + 8 * nt + g], bb[0], bs[0]);
            split_tf32(B[(k0 + q + 4) * LDB + 8 * nt + g], bb[1], bs[1]);
            mma_tf32(c[0][nt], as, bb);
            mma_tf32(c[NA > 1 ? 1 : 0][nt], ab, bs);
            mma_tf32(c[NA > 2 ? 2 : 0][nt], ab, bb);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float sum = c[0][nt][e];
#pragma unroll
            for (int t = 1; t < NA; ++t) sum += c[t][nt][e];
            acc[nt][e] += sum;
        }
}

template <int NT>
__device__ __forceinline__ void zero_frag(float (&acc)[NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
}

// Row and column of accumulator element e of n-tile nt.
__device__ __forceinline__ int frag_row(int m0, int lane, int e) { return m0 + (lane >> 2) + 8 * (e >> 1); }
__device__ __forceinline__ int frag_col(int n0, int lane, int nt, int e) {
    return n0 + 8 * nt + 2 * (lane & 3) + (e & 1);
}

template <int NT>
__device__ __forceinline__ void store_frag(float *C, const float (&acc)[NT][4], int m0, int n0, int lane) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *reinterpret_cast<float2 *>(C + frag_row(m0, lane, 2 * h) * LD + frag_col(n0, lane, nt, 0)) =
                make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
}

// Stores a warp's 16 x 64 accumulator block (rows m0..) as rows of 64 floats.
__device__ __forceinline__ void store_frag_global(float *__restrict__ C, const float (&acc)[8][4], int m0, int lane) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *reinterpret_cast<float2 *>(C + frag_row(m0, lane, 2 * h) * DD + frag_col(0, lane, nt, 0)) =
                make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
}

// One block per chunk (chunks of a lane consecutive): W, U and P of the chunk
// into the workspace, each 64 x 64 row-major (rows past the sequence end are
// zero).
__global__ void __launch_bounds__(kThreads, 2)
    delta_wy_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const float *__restrict__ beta, float *__restrict__ ws,
                    int64_t B, int64_t T, int64_t H, DevCtl ctl) {
    using L = WySmem;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *sm = reinterpret_cast<float *>(smem_raw);
    float *Q = sm + L::q, *K = sm + L::k, *V = sm + L::v, *Am = sm + L::a, *Tm = sm + L::t;
    float *Dv = sm + L::dinv, *Xs = sm + L::xs, *sb = sm + L::beta;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::bars);
    int *abort_word = reinterpret_cast<int *>(bar + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nch = (T + CH - 1) / CH;
    const int64_t ci = blockIdx.x;
    if (ci >= B * H * nch) return;
    // 32-bit divisions (the grid, the chunk count and H are below 2^31)
    const int lane32 = int(blockIdx.x) / int(nch);
    const int64_t lane_id = lane32, c = int64_t(blockIdx.x) - int64_t(lane32) * nch;
    const int64_t bi = lane32 / int(H), hd = lane32 - int(bi) * int(H);
    const int n = int(min64(CH, T - c * CH));
    const int r = int(bi * T + c * CH);
    float *Wg = ws + ci * 3 * WSM, *Ug = Wg + WSM, *Pg = Wg + 2 * WSM;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
        *abort_word = 0;
    }
    __syncthreads();
    WarpRing<1> rg;
    rg.bar = bar;
    rg.inflight = 0;
    rg.phase = 0;
    if (tid == 0) {
        // Q and K are read again by the state pass: kept in L2 at normal priority
        const uint64_t keep = policy_evict_normal(), once = policy_evict_first();
        mbar_arrive_expect_tx(bar, uint32_t(3 * MATF * 4));
        tma_load_3d(Q, &tmQ, 0, int(hd), r, bar, keep);
        tma_load_3d(K, &tmK, 0, int(hd), r, bar, keep);
        tma_load_3d(V, &tmV, 0, int(hd), r, bar, once);
    }
    rg.armed(0);
    if (tid < CH) sb[tid] = tid < n ? beta[(int64_t(r) + tid) * H + hd] : 0.f;
    if (!rg.wait(0, ctl) && lane == 0) {
        record_error(ctl, ERR_MBAR_TIMEOUT);
        *abort_word = 1;
    }
    __syncthreads();
    if (*abort_word != 0) {
        rg.drain(ctl, lane);
        return;
    }
    // rows past the sequence end (the next sequence's, or fill) contribute nothing
    if (n < CH)
        for (int e = tid; e < (CH - n) * LD; e += kThreads) {
            Q[n * LD + e] = 0.f;
            K[n * LD + e] = 0.f;
            V[n * LD + e] = 0.f;
        }
    __syncthreads();
    // Row blocks 16w (warps 0-3) and 16(7-w) (warps 4-7) in the triangular
    // products, so that the two warps of each SM sub-partition share out the
    // same number of tiles.
    const bool lo = warp < 4;
    const int mt = lo ? 16 * warp : 48 - 16 * (warp - 4);
    // Phase 1.  Warps 0-3: A = strict_tril(diag(beta) K K^T); warps 4-7:
    // P = tril(Q K^T), straight to the workspace.
    {
        float acc[8][4];
        zero_frag(acc);
        // only columns up to the diagonal: n-tiles below mt/8 + 2
        mma64<false, 8, true>(lo ? K : Q, K, acc, mt, 0, lane, DD, mt / 8 + 2);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = frag_row(mt, lane, e), s2 = frag_col(0, lane, nt, e);
                acc[nt][e] = lo ? ((s2 < t) ? sb[t] * acc[nt][e] : 0.f) : ((s2 <= t) ? acc[nt][e] : 0.f);
            }
        if (lo)
            store_frag(Am, acc, mt, 0, lane);
        else
            store_frag_global(Pg, acc, mt, lane);
    }
    __syncthreads();
    // Phase 2.  Warps 0-3: D_b = (I + A_bb)^{-1}, b = warp, lane j < 16 builds
    // column j by forward substitution; T'_bb = D_b diag(beta_b).  The column
    // is kept in registers and stored after it is complete, so that no shared
    // store sits between the loads of the chain.
    if (lo && lane < 16) {
        const int b0 = 16 * warp;
        float dcol[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            float arow[16];
#pragma unroll
            for (int q4 = 0; q4 < rr; q4 += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(Am + (b0 + rr) * LD + b0 + q4);
                arow[q4] = a4.x;
                arow[q4 + 1] = a4.y;
                arow[q4 + 2] = a4.z;
                arow[q4 + 3] = a4.w;
            }
            float acc = (rr == lane) ? 1.f : 0.f;
#pragma unroll
            for (int q = 0; q < rr; ++q) acc = fmaf(-arow[q], dcol[q], acc);
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
    // Phase 3.  E_bm = D_b A_bm for the six blocks below the diagonal (pair
    // j = b(b-1)/2 + m), then T'_bc = -sum_{c <= m < b} E_bm T'_mc one
    // subdiagonal d = b - c at a time.  Thread: element (tid / 16, tid % 16)
    // of every block of the step.
    const int er = tid >> 4, ec = tid & 15;
    {
        float acc[6];
#pragma unroll
        for (int j = 0; j < 6; ++j) acc[j] = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 16; q4 += 4) {
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                const int b = j < 1 ? 1 : j < 3 ? 2 : 3, m = j - b * (b - 1) / 2;
                const float4 d4 = *reinterpret_cast<const float4 *>(Dv + (16 * b + er) * DLD + q4);
                const float *a = Am + (16 * b + q4) * LD + 16 * m + ec;
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
    for (int d = 1; d < 4; ++d) {
        constexpr int kMaxB = 3;
        float acc[kMaxB];
#pragma unroll
        for (int cb = 0; cb < kMaxB; ++cb) acc[cb] = 0.f;
#pragma unroll
        for (int cb = 0; cb < 4 - d; ++cb) {
            const int b = cb + d;
#pragma unroll
            for (int m = cb; m < b; ++m) {
                const float *e = Xs + (16 * (b * (b - 1) / 2 + m) + er) * DLD;
                const float *t = Tm + 16 * m * LD + 16 * cb + ec;
#pragma unroll
                for (int q4 = 0; q4 < 16; q4 += 4) {
                    const float4 e4 = *reinterpret_cast<const float4 *>(e + q4);
                    acc[cb] = fmaf(e4.x, t[(q4 + 0) * LD], acc[cb]);
                    acc[cb] = fmaf(e4.y, t[(q4 + 1) * LD], acc[cb]);
                    acc[cb] = fmaf(e4.z, t[(q4 + 2) * LD], acc[cb]);
                    acc[cb] = fmaf(e4.w, t[(q4 + 3) * LD], acc[cb]);
                }
            }
        }
#pragma unroll
        for (int cb = 0; cb < 4 - d; ++cb) Tm[(16 * (cb + d) + er) * LD + 16 * cb + ec] = -acc[cb];
        __syncthreads();
    }
    // Phase 4.  Warps 0-3: W = T' K; warps 4-7: U = T' V (k only up to the
    // diagonal block), straight to the workspace.
    {
        float acc[8][4];
        zero_frag(acc);
        mma64<false, 8>(Tm, lo ? K : V, acc, mt, 0, lane, mt + 16);
        store_frag_global(lo ? Wg : Ug, acc, mt, lane);
    }
}

// One block per (lane, 8 NT value columns i0..): walks the lane's chunks in
// order with the slice S^T[:, i0..] in shared memory.  Per chunk:
//   warps 0-3: U'[16w..] = U[16w.., i] - W[16w..] S^T[:, i]
//   warps 4-7: O = Q[16(w-4)..] S^T[:, i], then O += P U' (k up to the diagonal)
//   warps 0-3: S^T[16w.., i] += K^T U'
// Warp 8 is the copy warp: it refills a stage by TMA once all eight compute
// warps have arrived on its "empty" barrier (after their last read of it),
// so issuing the copies never holds up the compute warps.  Only the copy
// warp issues copies, so only it drains them when the block gives up.
template <int NT>
__global__ void __launch_bounds__(kStateThreads)
    delta_state_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmU,
                       const float *__restrict__ S0, float *__restrict__ o, float *__restrict__ ST_out, int64_t B,
                       int64_t T, int64_t H, int nst, DevCtl ctl) {
    constexpr int VS = StateCols<NT>::VS, LDB = StateCols<NT>::LDB, NVB = DD / VS;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const StateSmem L(nst, LDB);
    float *sm = reinterpret_cast<float *>(smem_raw);
    float *STc = sm + L.st, *Up = sm + L.up;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.bars), *empty = full + kStages;
    volatile int *abort_word = reinterpret_cast<volatile int *>(empty + kStages);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t blk = blockIdx.x;
    if (blk >= B * H * NVB) return;
    const int64_t lane_id = blk / NVB;
    const int i0 = int(blk % NVB) * VS;
    const int64_t bi = int(lane_id) / int(H), hd = int(lane_id) - int(bi) * int(H);  // 32-bit: lanes < 2^31
    const int64_t nch = (T + CH - 1) / CH;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kThreads / 32);
        }
        fence_barrier_init();
        *abort_word = 0;
    }
    __syncthreads();

    if (warp == kThreads / 32) {  // the copy warp
        if (lane == 0) {
            // the lane's state blocks read the same W, P, Q, K (and U rows)
            const uint64_t pol = policy_evict_normal();
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmU);
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            // stage s and the parity of its "empty" phase to wait for, kept as
            // counters (no 64-bit division by the run-time stage count)
            int s = 0;
            uint32_t eph = 0;
            int64_t last = -1;
            for (int64_t c = 0; c < nch; ++c, s = (s + 1 == nst) ? 0 : s + 1) {
                if (c >= nst) {
                    // The abort word is written only by compute warps, before a
                    // barrier of theirs, so that all eight read the same value
                    // after it; this warp just stops issuing, and their bounded
                    // waits for the missing stage give up together.
                    const bool ok = mbar_wait_bounded(&empty[s], eph, ctl.timeout_ns);
                    if (!ok) record_error(ctl, ERR_MBAR_TIMEOUT);
                    if (!ok || *abort_word != 0) break;
                    if (s + 1 == nst) eph ^= 1u;
                }
                float *st = sm + s * L.stage;
                const int r = int(bi * T + c * CH);
                const int wr = int((lane_id * nch + c) * 3 * CH);  // workspace row of the chunk's W
                mbar_arrive_expect_tx(&full[s], uint32_t(L.stage * 4));
                tma_load_2d(st, &tmW, 0, wr, &full[s], pol);
                tma_load_2d(st + MATF, &tmW, 0, wr + 2 * CH, &full[s], pol);
                tma_load_3d(st + 2 * MATF, &tmQ, 0, int(hd), r, &full[s], pol);
                tma_load_3d(st + 3 * MATF, &tmK, 0, int(hd), r, &full[s], pol);
                tma_load_2d(st + 4 * MATF, &tmU, i0, wr + CH, &full[s], pol);
                last = c;
            }
            // the block's shared memory outlives every copy this warp started
            bool ok = true;
            for (int64_t c = last - nst + 1; c <= last; ++c)
                if (c >= 0 && !mbar_wait_bounded(&full[c % nst], uint32_t((c / nst) & 1), ctl.timeout_ns)) ok = false;
            if (!ok) record_error(ctl, ERR_DRAIN_TIMEOUT);
        }
        return;
    }

    // the slice of the initial state, key-major: STc[j][i] = S0[i0 + i][j]
    for (int e = tid; e < DD * VS; e += kThreads) {
        const int i = e >> 6, j = e & 63;
        STc[j * LDB + i] = S0 != nullptr ? S0[lane_id * DD * DD + (i0 + i) * DD + j] : 0.f;
    }

    const bool lo = warp < 4;
    const int m0 = 16 * (warp & 3);
    int s = 0;          // stage of chunk c
    uint32_t fph = 0;   // parity of its "full" phase
    for (int64_t c = 0; c < nch; ++c) {
        const int n = c + 1 < nch ? CH : int(T - c * CH);
        bool ok = mbar_wait_bounded(&full[s], fph, ctl.timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        compute_sync();  // also orders the previous chunk's state update before this chunk's reads
        if (*abort_word != 0) return;
        float *st = sm + s * L.stage;
        const float *W = st, *P = st + MATF, *Q = st + 2 * MATF, *Uc = st + 4 * MATF;
        float *K = st + 3 * MATF;
        // rows of K past the sequence end meet rows of U' that are exactly zero;
        // zeroed so that whatever they hold contributes nothing (only the last
        // chunk is short, and its stage is not refilled)
        if (n < CH)
            for (int e = tid; e < (CH - n) * LD; e += kThreads) K[n * LD + e] = 0.f;
        float acc[NT][4];
        zero_frag(acc);
        mma_tile<false, NT, LDB>(lo ? W : Q, STc, acc, m0, lane);
        if (lo) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = frag_row(m0, lane, 2 * h), i = frag_col(0, lane, nt, 0);
                    const float2 u2 = *reinterpret_cast<const float2 *>(Uc + t * LDB + i);
                    *reinterpret_cast<float2 *>(Up + t * LDB + i) =
                        make_float2(u2.x - acc[nt][2 * h], u2.y - acc[nt][2 * h + 1]);
                }
        }
        compute_sync();
        if (lo) {
            float dS[NT][4];
            zero_frag(dS);
            mma_tile<true, NT, LDB>(K, Up, dS, m0, lane);  // dS[j][i] = sum_t K[t][j] U'[t][i]
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // this warp's reads of the stage are done
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float2 *pp = reinterpret_cast<float2 *>(STc + frag_row(m0, lane, 2 * h) * LDB +
                                                            frag_col(0, lane, nt, 0));
                    const float2 v = *pp;
                    *pp = make_float2(v.x + dS[nt][2 * h], v.y + dS[nt][2 * h + 1]);
                }
        } else {
            mma_tile<false, NT, LDB>(P, Up, acc, m0, lane, m0 + 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = frag_row(m0, lane, 2 * h);
                    if (t < n)
                        *reinterpret_cast<float2 *>(o + ((bi * T + c * CH + t) * H + hd) * DD + i0 +
                                                    frag_col(0, lane, nt, 0)) =
                            make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
                }
        }
        // U' is rewritten in the next chunk's first phase: every read of it
        // here must be done first
        compute_sync();
        if (++s == nst) {
            s = 0;
            fph ^= 1u;
        }
    }
    if (ST_out != nullptr) {
        for (int e = tid; e < DD * VS; e += kThreads) {
            const int i = e >> 6, j = e & 63;
            ST_out[lane_id * DD * DD + (i0 + i) * DD + j] = STc[j * LDB + i];
        }
    }
}

// [rows][H][64] floats, boxes of 68 x 1 x 64: the 4 floats past each row are
// out of the tensor and arrive as zeros (the padded shared layout).
cudaError_t make_chunk_map(CUtensorMap *m, const float *base, int64_t rows, int64_t H) {
    const uint64_t dims[3] = {uint64_t(DD), uint64_t(H), uint64_t(rows)};
    const uint64_t str[2] = {uint64_t(DD) * 4u, uint64_t(H) * DD * 4u};
    const uint32_t box[3] = {uint32_t(LD), 1u, uint32_t(CH)};
    return make_tmap(m, base, 3, dims, str, box);
}

// The workspace as rows of 64 floats (W, U, P of every chunk): boxes of
// box_x x 64 floats; a box wider than the columns left in the row ends in the
// tensor map's zero fill (the padded layouts above).
cudaError_t make_ws_map(CUtensorMap *m, const float *ws, int64_t rows, int box_x) {
    const uint64_t dims[2] = {uint64_t(DD), uint64_t(rows)};
    const uint64_t str[1] = {uint64_t(DD) * 4u};
    const uint32_t box[2] = {uint32_t(box_x), uint32_t(CH)};
    return make_tmap(m, ws, 2, dims, str, box);
}

template <int NT>
cudaError_t launch_state(const CUtensorMap &tQ, const CUtensorMap &tK, const CUtensorMap &tW, float *w,
                         int64_t chunks, const float *S0, float *o, float *ST, int64_t B, int64_t T, int64_t H,
                         int nst, const DevCtl &ctl, cudaStream_t s) {
    constexpr int LDB = StateCols<NT>::LDB, NVB = DD / StateCols<NT>::VS;
    if (nst == 2 && (T + CH - 1) / CH > 2 && StateSmem(3, LDB).bytes <= 227 * 1024) nst = 3;
    CUtensorMap tU;
    cudaError_t e;
    if ((e = make_ws_map(&tU, w, chunks * 3 * CH, LDB)) != cudaSuccess) return e;
    const int smem = int(StateSmem(nst, LDB).bytes);
    if ((e = ensure_smem_attr((const void *)delta_state_kernel<NT>, smem)) != cudaSuccess) return e;
    delta_state_kernel<NT><<<dim3(unsigned(B * H * NVB)), kStateThreads, smem, s>>>(tQ, tK, tW, tU, S0, o, ST, B,
                                                                                    T, H, nst, ctl);
    return cudaGetLastError();
}

}  // namespace

size_t delta_workspace_bytes(int64_t B, int64_t T, int64_t H) {
    return size_t(B) * size_t(H) * size_t((T + CH - 1) / CH) * 3 * WSM * sizeof(float);
}

cudaError_t launch_delta_fwd(const float *q, const float *k, const float *v, const float *beta, const float *S0,
                             float *o, float *ST, int64_t B, int64_t T, int64_t H, void *ws, const DevCtl &ctl,
                             cudaStream_t s) {
    const int64_t nch = (T + CH - 1) / CH, chunks = B * H * nch, lanes = B * H;
    if (chunks > 0x7fffffff / (3 * CH) || lanes * 8 > 0x7fffffff) return cudaErrorInvalidConfiguration;
    float *w = static_cast<float *>(ws);
    CUtensorMap tQ, tK, tV, tW;
    cudaError_t e;
    if ((e = make_chunk_map(&tQ, q, B * T, H)) != cudaSuccess) return e;
    if ((e = make_chunk_map(&tK, k, B * T, H)) != cudaSuccess) return e;
    if ((e = make_chunk_map(&tV, v, B * T, H)) != cudaSuccess) return e;
    if ((e = make_ws_map(&tW, w, chunks * 3 * CH, LD)) != cudaSuccess) return e;
    const int smem_a = int(WySmem::bytes);
    if ((e = ensure_smem_attr((const void *)delta_wy_kernel, smem_a)) != cudaSuccess) return e;
    delta_wy_kernel<<<dim3(unsigned(chunks)), kThreads, smem_a, s>>>(tQ, tK, tV, beta, w, B, T, H, ctl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // State blocks as wide as the lane count allows while still giving about
    // one block per SM (the per-chunk products are cheapest per column in the
    // widest blocks; narrow ones shorten the chain when lanes are few).  As
    // many stages in flight as the chunks and shared memory allow.
    const int nst = int(min64(nch, 2));
    if (lanes >= 152) return launch_state<8>(tQ, tK, tW, w, chunks, S0, o, ST, B, T, H, nst, ctl, s);
    if (lanes >= 76) return launch_state<4>(tQ, tK, tW, w, chunks, S0, o, ST, B, T, H, nst, ctl, s);
    if (lanes >= 38) return launch_state<2>(tQ, tK, tW, w, chunks, S0, o, ST, B, T, H, nst, ctl, s);
    return launch_state<1>(tQ, tK, tW, w, chunks, S0, o, ST, B, T, H, nst, ctl, s);
}

}  // namespace mgs
