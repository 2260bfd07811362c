// Delta rule (DeltaNet), forward, in the chunked WY form ("mingru-scans" home
// page, lineage paragraph: DeltaMinGRU reimplements DeltaNet, Yang et al.
// 2024, arXiv:2406.06484, using its chunked WY representation as the
// parallel forward).  Per (batch, head) lane, state S (d_v x d_k, here D x D):
//   S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T,   o_t = S_t q_t.
//
// A chunk of C = 64 steps with state S on entry is, in matrix form (rows are
// time steps, K, V, Q are C x D):
//   A   = strict_tril(diag(beta) K K^T)
//   (I + A) [W | U] = diag(beta) [K | V],   U' = U - W S^T
//   O   = Q S^T + tril(Q K^T) U'
//   S  <- S + U'^T K
// which is the recurrence exactly (the WY representation of the product of
// the chunk's rank-one updates).  Since (I + A) is the same for W and U, U'
// is obtained from one solve, (I + A) U' = diag(beta) (V - K S^T), and W is
// never formed.  The solve is blocked by 16 rows: the four 16 x 16 diagonal
// blocks of (I + A) are inverted by forward substitution (one warp each), then
// U'_b = D_b (R_b - A_{b,<b} U'_{<b}) block after block.  The state is kept
// key-major (S^T) in shared memory so that every product reads its operands
// by rows.
//
// One 256-thread block per lane walks its chunks in order; each chunk's Q, K
// and V arrive by tiled TMA loads (a 68-float box over 64-float rows, so the
// last 4 floats of every shared row are the tensor map's zero fill: a padded
// layout that keeps the products' shared reads free of bank conflicts), two
// chunks in flight.  The 64 x 64 x 64 products run on the tensor cores
// (mma.sync tf32 with a three-term split for fp32 accuracy), each warp owning a
// 16 x 32 block of the result; the forward substitution runs on the fp32 pipes.
#include "mgs_tiles.cuh"

namespace mgs {
namespace {

constexpr int DD = 64;         // head dimension (d_k = d_v)
constexpr int CH = 64;         // chunk length
constexpr int LD = 68;         // padded row stride (floats)
constexpr int MATF = CH * LD;  // floats per padded 64 x 64 matrix
constexpr int kThreads = 256;
constexpr int kStages = 2;

// Shared memory layout (floats): stages [Q K V] x kStages, then ST, KT, A, QK,
// D (the inverted diagonal blocks, rows 16b..16b+15, columns 0..15), U (R,
// then U' in place; also the 16-row panel of the blocked solve), beta (64),
// barriers.
struct DeltaSmem {
    static constexpr int stage = 3 * MATF;
    static constexpr int st = kStages * stage;
    static constexpr int kt = st + MATF;
    static constexpr int a = kt + MATF;
    static constexpr int qk = a + MATF;
    static constexpr int w = qk + MATF;
    static constexpr int u = w + MATF;
    static constexpr int beta = u + MATF;
    static constexpr int bars = beta + CH;  // 8-byte aligned (all offsets are multiples of 4 floats)
    static constexpr size_t bytes = size_t(bars) * 4 + kStages * sizeof(uint64_t) + 16;  // + abort word
};

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

// acc[nt] += op(A)[m0.., :] B[:, n0 + 8 nt ..] over k = 0..63 for one warp's
// 16 x (8 NT) block of the result.  AT = false: A row-major [m][k];
// AT = true: A stored [k][m].  B row-major [k][n].  Stride LD.
// Only k < kend and n-tiles nt < ntl take part (the zero triangles of the
// masked products are skipped; both limits are warp-uniform).
template <bool AT, int NT>
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
            split_tf32(B[(k0 + q) * LD + n], bb[0], bs[0]);
            split_tf32(B[(k0 + q + 4) * LD + n], bb[1], bs[1]);
            mma_tf32(acc[nt], as, bb);
            mma_tf32(acc[nt], ab, bs);
            mma_tf32(acc[nt], ab, bb);
        }
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

__global__ void __launch_bounds__(kThreads)
    delta_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const float *__restrict__ beta,
                     const float *__restrict__ S0, float *__restrict__ o, float *__restrict__ ST_out, int64_t B,
                     int64_t T, int64_t H, DevCtl ctl) {
    using L = DeltaSmem;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *sm = reinterpret_cast<float *>(smem_raw);
    float *ST = sm + L::st, *KT = sm + L::kt, *Am = sm + L::a, *QK = sm + L::qk, *U = sm + L::u;
    float *Wd = sm + L::w;           // inverted diagonal blocks D_b
    float *Pn = KT;                  // 16-row panel of the blocked solve (KT is free by then)
    float *sb = sm + L::beta;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::bars);
    int *abort_word = reinterpret_cast<int *>(bars + kStages);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t lane_id = blockIdx.x;  // (batch, head)
    if (lane_id >= B * H) return;
    const int64_t bi = lane_id / H, hd = lane_id % H;
    const int64_t nch = (T + CH - 1) / CH;
    const int row0 = int(bi * T);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        *abort_word = 0;
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int s, int64_t c) {  // thread 0 only
        float *st = sm + s * L::stage;
        const int r = row0 + int(c * CH);
        mbar_arrive_expect_tx(&bars[s], uint32_t(3 * MATF * 4));
        tma_load_3d(st, &tmQ, 0, int(hd), r, &bars[s], pol);
        tma_load_3d(st + MATF, &tmK, 0, int(hd), r, &bars[s], pol);
        tma_load_3d(st + 2 * MATF, &tmV, 0, int(hd), r, &bars[s], pol);
    };
    // Every thread tracks the ring (all wait on the same barriers).
    WarpRing<kStages> rg;
    rg.bar = bars;
    rg.inflight = 0;
    rg.phase = 0;
    const int npro = int(min64(kStages, nch));
    if (tid == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        for (int s = 0; s < npro; ++s) issue(s, s);
    }
    for (int s = 0; s < npro; ++s) rg.armed(s);

    float beta_next = (tid < CH && tid < T) ? beta[(bi * T + tid) * H + hd] : 0.f;
    // initial state, key-major: ST[j][i] = S0[i][j]
    for (int e = tid; e < DD * DD; e += kThreads) {
        const int i = e >> 6, j = e & 63;
        ST[j * LD + i] = S0 != nullptr ? S0[lane_id * DD * DD + e] : 0.f;
    }

    for (int64_t c = 0; c < nch; ++c) {
        const int s = int(c % kStages);
        const int n = int(min64(CH, T - c * CH));
        // a wait that gives up in any warp makes the whole block leave at the
        // next barrier, after each warp has drained the copies it still counts
        if (!rg.wait(s, ctl) && lane == 0) {
            record_error(ctl, ERR_MBAR_TIMEOUT);
            *abort_word = 1;
        }
        __syncthreads();
        if (*abort_word != 0) {
            rg.drain(ctl, lane);
            return;
        }
        float *Q = sm + s * L::stage, *K = Q + MATF, *V = K + MATF;
        // beta of the chunk (0 past the sequence end; loaded one chunk ahead);
        // the rows of Q, K and V past the end (the next sequence's, or fill)
        // are zeroed so that they contribute exactly nothing
        if (tid < CH) {
            sb[tid] = beta_next;
            const int64_t tn = (c + 1) * CH + tid;
            beta_next = tn < T ? beta[(bi * T + tn) * H + hd] : 0.f;
        }
        if (n < CH)
            for (int e = tid; e < (CH - n) * LD; e += kThreads) {
                Q[n * LD + e] = 0.f;
                K[n * LD + e] = 0.f;
                V[n * LD + e] = 0.f;
            }
        __syncthreads();
        // KT[j][t] = K[t][j]
        for (int e = tid; e < CH * DD; e += kThreads) {
            const int t = e & 63, j = e >> 6;
            KT[j * LD + t] = K[t * LD + j];
        }
        __syncthreads();
        // Phase 1.  Warps 0-3 (rows 16w..): A = strict_tril(diag(beta) K K^T)
        // and R = diag(beta) (V - K S^T).  Warps 4-7 (rows 16(w-4)..):
        // QK = tril(Q K^T) and Q S^T, the latter kept in registers as the
        // start of O.
        const bool lo = warp < 4;
        const int mr = 16 * (warp & 3);  // this warp's 16 rows in phases 1 and 4
        float oacc[8][4];                // warps 4-7: Q S^T, then O; warps 0-3: K^T U'
        zero_frag(oacc);
        {
            // the triangular products take rows 16w (warps 0-3) and 16(7-w)
            // (warps 4-7), so that the two warps of each SM sub-partition
            // (w and w+4) share out the same number of tiles
            const int mt = lo ? mr : 48 - mr;
            float acc[8][4];
            zero_frag(acc);
            // only columns up to the diagonal: n-tiles below mt/8 + 2
            mma64<false>(lo ? K : Q, KT, acc, mt, 0, lane, DD, mt / 8 + 2);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = frag_row(mt, lane, e), s2 = frag_col(0, lane, nt, e);
                    acc[nt][e] = lo ? ((s2 < t) ? sb[t] * acc[nt][e] : 0.f) : ((s2 <= t) ? acc[nt][e] : 0.f);
                }
            store_frag(lo ? Am : QK, acc, mt, 0, lane);
            mma64<false>(lo ? K : Q, ST, oacc, mr, 0, lane);
            if (lo) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t = frag_row(mr, lane, 2 * h), i = frag_col(0, lane, nt, 0);
                        const float2 v2 = *reinterpret_cast<const float2 *>(V + t * LD + i);
                        *reinterpret_cast<float2 *>(U + t * LD + i) =
                            make_float2(sb[t] * (v2.x - oacc[nt][2 * h]), sb[t] * (v2.y - oacc[nt][2 * h + 1]));
                    }
                zero_frag(oacc);
            }
        }
        __syncthreads();
        // Phase 2.  D_b = (I + A_bb)^{-1}, b = warp (0-3), lane j < 16 builds
        // column j by forward substitution.
        if (warp < 4 && lane < 16) {
            const int b0 = 16 * warp;
            float dcol[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = (r == lane) ? 1.f : 0.f;
#pragma unroll
                for (int q = 0; q < r; ++q) acc = fmaf(-Am[(b0 + r) * LD + b0 + q], dcol[q], acc);
                dcol[r] = acc;
                Wd[(b0 + r) * LD + lane] = acc;
            }
        }
        __syncthreads();
        // Phase 3.  Blocked solve, U' in place of R: for b = 0..3,
        // P = R_b - A_{b,<b} U'_{<b};  U'_b = D_b P.  Thread: column tid % 64,
        // rows 4 (tid / 64) .. +3 of the block.
        {
            const int col = tid & 63, r0 = 4 * (tid >> 6);
            for (int b = 0; b < 4; ++b) {
                const int b0 = 16 * b;
                float p[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) p[r] = U[(b0 + r0 + r) * LD + col];
                for (int s4 = 0; s4 < b0; s4 += 4) {
                    const float u0 = U[(s4 + 0) * LD + col], u1 = U[(s4 + 1) * LD + col];
                    const float u2 = U[(s4 + 2) * LD + col], u3 = U[(s4 + 3) * LD + col];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(Am + (b0 + r0 + r) * LD + s4);
                        p[r] = fmaf(-a4.x, u0, p[r]);
                        p[r] = fmaf(-a4.y, u1, p[r]);
                        p[r] = fmaf(-a4.z, u2, p[r]);
                        p[r] = fmaf(-a4.w, u3, p[r]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) Pn[(r0 + r) * LD + col] = p[r];
                __syncthreads();
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int q4 = 0; q4 < 16; q4 += 4) {
                        const float4 d4 = *reinterpret_cast<const float4 *>(Wd + (b0 + r0 + r) * LD + q4);
                        acc = fmaf(d4.x, Pn[(q4 + 0) * LD + col], acc);
                        acc = fmaf(d4.y, Pn[(q4 + 1) * LD + col], acc);
                        acc = fmaf(d4.z, Pn[(q4 + 2) * LD + col], acc);
                        acc = fmaf(d4.w, Pn[(q4 + 3) * LD + col], acc);
                    }
                    U[(b0 + r0 + r) * LD + col] = acc;
                }
                __syncthreads();
            }
        }
        // Phase 4.  Warps 4-7: O = Q S^T + tril(Q K^T) U' (k only up to the
        // diagonal); warps 0-3: rows 16w.. of K^T U' (the state update).
        if (lo) {
            mma64<true>(K, U, oacc, mr, 0, lane);  // oacc[j][i] = sum_t K[t][j] U'[t][i]
        } else {
            mma64<false>(QK, U, oacc, mr, 0, lane, mr + 16);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = frag_row(mr, lane, 2 * h);
                    if (t < n)
                        *reinterpret_cast<float2 *>(o + ((bi * T + c * CH + t) * H + hd) * DD +
                                                    frag_col(0, lane, nt, 0)) =
                            make_float2(oacc[nt][2 * h], oacc[nt][2 * h + 1]);
                }
        }
        __syncthreads();  // every read of ST and of this stage is done
        if (lo) {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float2 *pp =
                        reinterpret_cast<float2 *>(ST + frag_row(mr, lane, 2 * h) * LD + frag_col(0, lane, nt, 0));
                    const float2 v = *pp;
                    *pp = make_float2(v.x + oacc[nt][2 * h], v.y + oacc[nt][2 * h + 1]);
                }
        }
        if (c + kStages < nch) {
            if (tid == 0) {
                fence_proxy_async_smem();
                issue(s, c + kStages);
            }
            rg.armed(s);
        }
        __syncthreads();
    }
    if (ST_out != nullptr) {
        for (int e = tid; e < DD * DD; e += kThreads) {
            const int i = e >> 6, j = e & 63;
            ST_out[lane_id * DD * DD + e] = ST[j * LD + i];
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

}  // namespace

cudaError_t launch_delta_fwd(const float *q, const float *k, const float *v, const float *beta, const float *S0,
                             float *o, float *ST, int64_t B, int64_t T, int64_t H, const DevCtl &ctl,
                             cudaStream_t s) {
    CUtensorMap tQ, tK, tV;
    cudaError_t e;
    if ((e = make_chunk_map(&tQ, q, B * T, H)) != cudaSuccess) return e;
    if ((e = make_chunk_map(&tK, k, B * T, H)) != cudaSuccess) return e;
    if ((e = make_chunk_map(&tV, v, B * T, H)) != cudaSuccess) return e;
    const int64_t blocks = B * H;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int smem = int(DeltaSmem::bytes);
    if ((e = ensure_smem_attr((const void *)delta_fwd_kernel, smem)) != cudaSuccess) return e;
    delta_fwd_kernel<<<dim3(unsigned(blocks)), kThreads, smem, s>>>(tQ, tK, tV, beta, S0, o, ST, B, T, H, ctl);
    return cudaGetLastError();
}

}  // namespace mgs
