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

// Rounds a shared-memory pointer up to `a` bytes (dynamic shared memory is
// allocated with that much slack).
__device__ __forceinline__ unsigned char *align_smem(unsigned char *p, size_t a) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    return p + ((a - (s & (a - 1))) & (a - 1));
}

}  // namespace mgs
