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

// MXFP8 of activations (OCP Microscaling, the rule of the weights' quantiser):
// per 32-element block, shared exponent floor(log2(max |v|)) - 8 clamped to
// [-127, 127] (0 for an all-zero block), codes E4M3 of v / 2^shared (nearest,
// ties to even, saturating at +-448), scale byte shared + 127.

// 2^k as an fp32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(1u << (k + 149));
}

// The block's shared exponent from its largest magnitude.
__device__ __forceinline__ int mx_shared_exp(float amax) {
    if (!(amax > 0.f)) return 0;
    int ex;
    frexpf(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1
    return min(max(ex - 1 - 8, -127), 127);
}

// E4M3 codes of (lo, hi) in bytes 0 and 1 (the instruction converts its
// first source into the upper byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
    return pair;
}

// MXFP8 form of 128 consecutive bf16 values, four per lane (lane l holds
// elements 4l .. 4l+3): the E4M3 codes of this lane's four (returned, element
// order in the bytes) and, in every lane, the scale word of the four 32-blocks
// (byte b: block b), by the MX rule (shared exponent floor(log2 amax) - 8,
// codes nearest-even, saturating).
__device__ __forceinline__ uint32_t mx_quantize128(uint2 raw, int lane, uint32_t& word) {
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const float2 f0 = __bfloat1622float2(v[0]), f1 = __bfloat1622float2(v[1]);
    float a = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));  // the block's 8 lanes
    const int shared = mx_shared_exp(a);
    const float sc = pow2f(-shared);  // exact: a power of two
    const uint32_t codes = e4m3x2(f0.x * sc, f0.y * sc) | (e4m3x2(f1.x * sc, f1.y * sc) << 16);
    const uint32_t b = (lane & 7) == 0 ? (uint32_t)(shared + 127) << (8 * (lane >> 3)) : 0u;
    word = __reduce_or_sync(0xffffffffu, b);
    return codes;
}

}  // namespace moe
