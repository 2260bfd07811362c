// Tensor-map tiling shared by the block-matrix kernels: a tensor laid out as
// [B*T rows][H heads][E floats per head] is streamed in boxes of TS rows x LPW
// heads, one TMA instruction per box.  When LPW*E fits in one box row (at most
// 256 elements) the map is 2-D (H*E, B*T); otherwise 3-D (E, H, B*T).
#pragma once

#include "mgs_launch.h"

namespace mgs {

template <int E, int LPW>
struct HeadTile {
    static constexpr bool kThreeD = (LPW * E > 256);

    // Host: encode the map for `base` with TS rows per box.
    static cudaError_t make(CUtensorMap *map, const float *base, int64_t rows, int64_t H, int TS) {
        if constexpr (kThreeD) {
            const uint64_t dims[3] = {uint64_t(E), uint64_t(H), uint64_t(rows)};
            const uint64_t str[2] = {uint64_t(E) * 4u, uint64_t(H) * E * 4u};
            const uint32_t box[3] = {uint32_t(E), uint32_t(LPW), uint32_t(TS)};
            return make_tmap(map, base, 3, dims, str, box);
        } else {
            const uint64_t dims[2] = {uint64_t(H) * E, uint64_t(rows)};
            const uint64_t str[1] = {uint64_t(H) * E * 4u};
            const uint32_t box[2] = {uint32_t(LPW * E), uint32_t(TS)};
            return make_tmap(map, base, 2, dims, str, box);
        }
    }

    // Device: load the box whose first row is `row` (may be negative or past
    // the end: zero-filled) for heads head0 .. head0+LPW-1.
    static __device__ __forceinline__ void load(void *dst, const CUtensorMap *map, int head0, int row,
                                                uint64_t *bar, uint64_t pol) {
        if constexpr (kThreeD)
            tma_load_3d(dst, map, 0, head0, row, bar, pol);
        else
            tma_load_2d(dst, map, head0 * E, row, bar, pol);
    }
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// k x k blocks [B*T rows][H heads][k][k] staged TS rows x LPW heads per box.
// For k >= 8 the box is loaded with the TMA 128-byte swizzle over 32-float
// (128-byte) lines: within every 1024-byte group of 8 lines, 16-byte chunk c of
// line l lands at chunk c ^ l.  The 4 (k = 8) or 2 (k = 16) lanes of a warp
// then read their blocks from different banks, which makes row reads,
// broadcast matrix-vector reads and column reads conflict-free.  Boxes must
// start on 1024-byte boundaries.  For k < 8, or with SWZ = false, the layout
// is plain row-major (the single-pass kernels read one row per thread, where
// the swizzle's address arithmetic costs more than the 2-way conflicts it
// removes; the chunked kernels' broadcast reads gain from it).
template <int K, bool SWZ = (K >= 8)>
struct MatTile {
    static constexpr int LPW = 32 / K;
    static constexpr int MF = LPW * K * K;  // floats per step (one box row)
    static constexpr bool kSwz = SWZ && K >= 8;
    static constexpr size_t kAlign = kSwz ? 1024 : 128;

    static cudaError_t make(CUtensorMap *map, const float *base, int64_t rows, int64_t H, int TS) {
        if constexpr (kSwz) {
            const uint64_t lines = uint64_t(H) * K * K / 32;
            const uint64_t dims[3] = {32u, lines, uint64_t(rows)};
            const uint64_t str[2] = {128u, uint64_t(H) * K * K * 4u};
            const uint32_t box[3] = {32u, uint32_t(LPW * K * K / 32), uint32_t(TS)};
            return make_tmap(map, base, 3, dims, str, box, /*swizzle128=*/true);
        } else {
            return HeadTile<K * K, LPW>::make(map, base, rows, H, TS);
        }
    }

    static __device__ __forceinline__ void load(void *dst, const CUtensorMap *map, int head0, int row,
                                                uint64_t *bar, uint64_t pol) {
        if constexpr (kSwz)
            tma_load_3d(dst, map, 0, head0 * K * K / 32, row, bar, pol);
        else
            HeadTile<K * K, LPW>::load(dst, map, head0, row, bar, pol);
    }

    // Float index, relative to the box, of elements (i, j0..j0+3) of lane sub's
    // block at box row u (j0 a multiple of 4 when k >= 4).
    static __device__ __forceinline__ int idx4(int u, int sub, int i, int j0) {
        const int flat = sub * K * K + i * K + j0;
        if constexpr (kSwz) {
            const int line = flat >> 5;
            return (u * K + line) * 32 + ((((flat >> 2) & 7) ^ (line & 7)) << 2);
        } else {
            return u * MF + flat;
        }
    }
    static __device__ __forceinline__ int idx1(int u, int sub, int i, int j) {
        if constexpr (kSwz)
            return idx4(u, sub, i, j & ~3) + (j & 3);
        else
            return u * MF + sub * K * K + i * K + j;
    }
};

// One lane's k x k block inside a staged box.
template <int K, bool SWZ = (K >= 8)>
struct TileRef {
    using Tile = MatTile<K, SWZ>;
    const float *box;
    int u, sub;
    __device__ __forceinline__ float at(int i, int j) const { return box[Tile::idx1(u, sub, i, j)]; }
    // row i into registers
    __device__ __forceinline__ void row(int i, float (&r)[K]) const {
        if constexpr (K >= 4) {
#pragma unroll
            for (int c = 0; c < K / 4; ++c) {
                const float4 q = *reinterpret_cast<const float4 *>(box + Tile::idx4(u, sub, i, 4 * c));
                r[4 * c] = q.x; r[4 * c + 1] = q.y; r[4 * c + 2] = q.z; r[4 * c + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < K; ++c) r[c] = at(i, c);
        }
    }
};

// Per-thread offsets (floats, from the start of a box row) of the 16-byte
// quads of lane sub's k x k block.  The swizzle's XOR depends only on the
// lane and the quad, so it is computed once per thread instead of at every
// load of a step.
template <int K>
struct QuadOffsets {
    int o[K][(K + 3) / 4];
    int oc[K];  // element (i, col) of the thread's own column
    __device__ __forceinline__ QuadOffsets(int sub, int col) {
#pragma unroll
        for (int i = 0; i < K; ++i) {
#pragma unroll
            for (int c = 0; c < (K + 3) / 4; ++c) o[i][c] = MatTile<K>::idx4(0, sub, i, 4 * c);
            oc[i] = MatTile<K>::idx1(0, sub, i, col);
        }
    }
};

// One lane's k x k block inside a staged box, addressed through QuadOffsets
// (for k < 4 the box is unswizzled and a row is K consecutive floats).
template <int K>
struct TileRefQ {
    const float *box;  // the box row of this step
    const QuadOffsets<K> &q;
    // element (i, col) of the thread's own column
    __device__ __forceinline__ float at_col(int i) const { return box[q.oc[i]]; }
    __device__ __forceinline__ void row(int i, float (&r)[K]) const {
        if constexpr (K >= 4) {
#pragma unroll
            for (int c = 0; c < K / 4; ++c) {
                const float4 v = *reinterpret_cast<const float4 *>(box + q.o[i][c]);
                r[4 * c] = v.x; r[4 * c + 1] = v.y; r[4 * c + 2] = v.z; r[4 * c + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < K; ++c) r[c] = box[q.o[i][0] + c];
        }
    }
};

// y = M x for a staged block.
template <int K, bool SWZ>
__device__ __forceinline__ void tile_matvec(const TileRef<K, SWZ> &M, const float (&x)[K], float (&y)[K]) {
#pragma unroll
    for (int i = 0; i < K; ++i) {
        float r[K];
        M.row(i, r);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int m = 0; m < K; ++m) {
            if (m & 1) s1 = fmaf(r[m], x[m], s1);
            else s0 = fmaf(r[m], x[m], s0);
        }
        y[i] = s0 + s1;
    }
}

// y = M^T x for a staged block: y[m] = sum_i M[i][m] x[i].
template <int K, bool SWZ>
__device__ __forceinline__ void tile_matvec_t(const TileRef<K, SWZ> &M, const float (&x)[K], float (&y)[K]) {
#pragma unroll
    for (int m = 0; m < K; ++m) y[m] = 0.f;
#pragma unroll
    for (int i = 0; i < K; ++i) {
        float r[K];
        M.row(i, r);
#pragma unroll
        for (int m = 0; m < K; ++m) y[m] = fmaf(r[m], x[i], y[m]);
    }
}

// The whole k x k block of one step into registers, row-major (every load
// issued before any use, so a step's latency is one shared-memory round trip).
template <int K>
__device__ __forceinline__ void tile_load(const TileRefQ<K> &M, float (&a)[K][K]) {
#pragma unroll
    for (int i = 0; i < K; ++i) M.row(i, a[i]);
}

// y = A x, y = A^T x, and two of the latter, from a block in registers: the
// arithmetic and order of tile_matvec / tile_matvec_t below (the even and odd
// partial sums of a row, or adjacent outputs, paired in one two-wide FMA that
// rounds each half as fmaf; sm_100 and later).
template <int K>
__device__ __forceinline__ void reg_matvec(const float (&a)[K][K], const float (&x)[K], float (&y)[K]) {
    if constexpr (K >= 2) {
#pragma unroll
        for (int i = 0; i < K; ++i) {
            float2 s = make_float2(0.f, 0.f);  // (even m, odd m)
#pragma unroll
            for (int m = 0; m < K; m += 2)
                s = __ffma2_rn(make_float2(a[i][m], a[i][m + 1]), make_float2(x[m], x[m + 1]), s);
            y[i] = s.x + s.y;
        }
    } else {
        y[0] = fmaf(a[0][0], x[0], 0.f) + 0.f;
    }
}
template <int K>
__device__ __forceinline__ void reg_matvec_t(const float (&a)[K][K], const float (&x)[K], float (&y)[K]) {
    if constexpr (K >= 2) {
        float2 acc[K / 2];
#pragma unroll
        for (int m = 0; m < K / 2; ++m) acc[m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const float2 xi = make_float2(x[i], x[i]);
#pragma unroll
            for (int m = 0; m < K; m += 2) acc[m / 2] = __ffma2_rn(make_float2(a[i][m], a[i][m + 1]), xi, acc[m / 2]);
        }
#pragma unroll
        for (int m = 0; m < K; m += 2) {
            y[m] = acc[m / 2].x;
            y[m + 1] = acc[m / 2].y;
        }
    } else {
        y[0] = fmaf(a[0][0], x[0], 0.f);
    }
}
template <int K>
__device__ __forceinline__ void reg_matvec_t2(const float (&a)[K][K], const float (&x1)[K], const float (&x2)[K],
                                              float (&y1)[K], float (&y2)[K]) {
    if constexpr (K >= 2) {
        float2 a1[K / 2], a2[K / 2];
#pragma unroll
        for (int m = 0; m < K / 2; ++m) a1[m] = a2[m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const float2 u1 = make_float2(x1[i], x1[i]), u2 = make_float2(x2[i], x2[i]);
#pragma unroll
            for (int m = 0; m < K; m += 2) {
                const float2 rm = make_float2(a[i][m], a[i][m + 1]);
                a1[m / 2] = __ffma2_rn(rm, u1, a1[m / 2]);
                a2[m / 2] = __ffma2_rn(rm, u2, a2[m / 2]);
            }
        }
#pragma unroll
        for (int m = 0; m < K; m += 2) {
            y1[m] = a1[m / 2].x;
            y1[m + 1] = a1[m / 2].y;
            y2[m] = a2[m / 2].x;
            y2[m + 1] = a2[m / 2].y;
        }
    } else {
        y1[0] = fmaf(a[0][0], x1[0], 0.f);
        y2[0] = fmaf(a[0][0], x2[0], 0.f);
    }
}

// y = M x and y = M^T x through TileRefQ: the same arithmetic, in the same
// order, as above, with the even- and odd-indexed accumulators of a row (M x)
// or adjacent outputs (M^T x) paired in one two-wide FMA (sm_100 and later;
// each half rounds as fmaf), so the results are identical.
template <int K>
__device__ __forceinline__ void tile_matvec(const TileRefQ<K> &M, const float (&x)[K], float (&y)[K]) {
    if constexpr (K >= 2) {
#pragma unroll
        for (int i = 0; i < K; ++i) {
            float r[K];
            M.row(i, r);
            float2 s = make_float2(0.f, 0.f);  // (even m, odd m)
#pragma unroll
            for (int m = 0; m < K; m += 2)
                s = __ffma2_rn(make_float2(r[m], r[m + 1]), make_float2(x[m], x[m + 1]), s);
            y[i] = s.x + s.y;
        }
    } else {
        float r[1];
        M.row(0, r);
        y[0] = fmaf(r[0], x[0], 0.f) + 0.f;
    }
}
template <int K>
__device__ __forceinline__ void tile_matvec_t(const TileRefQ<K> &M, const float (&x)[K], float (&y)[K]) {
    if constexpr (K >= 2) {
        float2 acc[K / 2];
#pragma unroll
        for (int m = 0; m < K / 2; ++m) acc[m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < K; ++i) {
            float r[K];
            M.row(i, r);
            const float2 xi = make_float2(x[i], x[i]);
#pragma unroll
            for (int m = 0; m < K; m += 2) acc[m / 2] = __ffma2_rn(make_float2(r[m], r[m + 1]), xi, acc[m / 2]);
        }
#pragma unroll
        for (int m = 0; m < K; m += 2) {
            y[m] = acc[m / 2].x;
            y[m + 1] = acc[m / 2].y;
        }
    } else {
        float r[1];
        M.row(0, r);
        y[0] = fmaf(r[0], x[0], 0.f);
    }
}

// y1 = M^T x1 and y2 = M^T x2 in one pass over M's rows (each row read once;
// per output the same arithmetic and order as two tile_matvec_t calls).
template <int K>
__device__ __forceinline__ void tile_matvec_t2(const TileRefQ<K> &M, const float (&x1)[K], const float (&x2)[K],
                                               float (&y1)[K], float (&y2)[K]) {
    if constexpr (K >= 2) {
        float2 a1[K / 2], a2[K / 2];
#pragma unroll
        for (int m = 0; m < K / 2; ++m) a1[m] = a2[m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < K; ++i) {
            float r[K];
            M.row(i, r);
            const float2 u1 = make_float2(x1[i], x1[i]), u2 = make_float2(x2[i], x2[i]);
#pragma unroll
            for (int m = 0; m < K; m += 2) {
                const float2 rm = make_float2(r[m], r[m + 1]);
                a1[m / 2] = __ffma2_rn(rm, u1, a1[m / 2]);
                a2[m / 2] = __ffma2_rn(rm, u2, a2[m / 2]);
            }
        }
#pragma unroll
        for (int m = 0; m < K; m += 2) {
            y1[m] = a1[m / 2].x;
            y1[m + 1] = a1[m / 2].y;
            y2[m] = a2[m / 2].x;
            y2[m + 1] = a2[m / 2].y;
        }
    } else {
        tile_matvec_t(M, x1, y1);
        tile_matvec_t(M, x2, y2);
    }
}

// Rounds a shared-memory pointer up to `a` bytes (dynamic shared memory is
// allocated with that much slack).
__device__ __forceinline__ unsigned char *align_smem(unsigned char *p, size_t a) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    return p + ((a - (s & (a - 1))) & (a - 1));
}

}  // namespace mgs
