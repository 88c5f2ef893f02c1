// gemm_common.cuh - pieces shared by the tcgen05 grouped GEMM kernels.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"

namespace moe {

struct Tile {
    int m, g, nt, row0, row_end;
};

// Tile order: expert g outermost, then micro m (when `per_micro` is set), then
// the n-tile, with the m-tiles (row blocks) of one (g, m, n-tile) adjacent.
// Consecutive CTAs therefore share a weight tile through L2, and all micros
// of an expert run back to back so its activation rows are still in L2.
// seg/tiles are the group row offsets and the prefix of row blocks per group.
__device__ __forceinline__ Tile decode_group_tile(int tile, const int* seg, const int* tiles, int G, int n_tiles,
                                                  int n_micro, bool per_micro, int block_rows) {
    Tile t;
    const int per_row_tile = n_tiles * (per_micro ? n_micro : 1);
    int lo = 0, hi = G - 1;  // largest g with tiles[g] * per_row_tile <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tiles[mid] * per_row_tile <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    t.g = lo;
    const int mtiles = tiles[lo + 1] - tiles[lo];
    int local = tile - tiles[lo] * per_row_tile;
    t.m = 0;
    if (per_micro) {
        t.m = local / (mtiles * n_tiles);
        local -= t.m * mtiles * n_tiles;
    }
    t.nt = local / mtiles;
    const int mt = local - t.nt * mtiles;
    t.row0 = seg[lo] + mt * block_rows;
    t.row_end = seg[lo + 1];
    return t;
}

__device__ __forceinline__ const CUtensorMap* pick_map(int m, const CUtensorMap& b0, const CUtensorMap& b1,
                                                       const CUtensorMap& b2, const CUtensorMap& b3) {
    return m == 0 ? &b0 : m == 1 ? &b1 : m == 2 ? &b2 : &b3;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

}  // namespace moe
