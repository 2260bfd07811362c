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

}  // namespace mgs
