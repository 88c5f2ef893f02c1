// mx_act.cu - MXFP8 activations for the block-scaled FP8 expert GEMMs.
//
// The routed experts of a batch run on the tensor cores' block-scaled FP8 MMA
// when their weights are MXFP8 (OCP Microscaling): the activations are then
// MXFP8 as well, with the same rule as the weights (mxfp8.cu): per 32
// consecutive elements along K, shared exponent floor(log2(max |v|)) - 8
// clamped to [-127, 127] (0 for an all-zero block), codes E4M3 of
// v / 2^shared, nearest with ties to even, saturating at +-448.
//
// Layouts, for GEMMs that take 128 K per stage: codes [rows][K] (uint8, the
// row order of the GEMM), scales stage-major [K/128][rows_pad][4] (uint8:
// the four 32-blocks of a stage of a row form one 32-bit word, byte i = block
// i), so the words of consecutive rows of one stage are consecutive. This
// file quantises the gathered token rows; h is quantised in the epilogue of
// the SwiGLU GEMM (gemm_pair.cu) into the same layout.
//
// One warp per token row (below): sixteen 16-byte loads per lane in flight,
// four lanes per 32-block.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// One warp per token: lane l loads elements 8l .. 8l+7 of each 256-element
// unit (one 16-byte load; a 32-block spans four lanes), sixteen units in
// flight (a whole 8 KB row of a 4096-wide layer), quantises them and writes
// the codes to the token's k route rows (8 bytes per lane and route; the rows
// are taken from the route lanes once per token) and each stage's scale word
// (lanes 0-15 hold the unit's first stage, 16-31 its second). The earlier form (a warp per 8 stages of a token, 8-byte loads
// four stages ahead) ran at 0.42 of the HBM bandwidth, bound by the latency of
// its loads and of the quantisation's dependent shuffles.
constexpr int kUnits = 16;  // 256-element units in flight per warp

// MXFP8 of this lane's eight elements of a 256-element unit: the eight codes
// (element order in the bytes) and, in every lane of the half-warp, the scale
// word of the half-warp's stage (byte b: 32-block b of the stage).
__device__ __forceinline__ uint2 quantize_unit(uint4 raw, int lane, uint32_t& word) {
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __bfloat1622float2(v[i]);
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));  // the block's four lanes
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const int shared = mx_shared_exp(a);
    const float sc = pow2f(-shared);  // exact: a power of two
    const uint2 codes = make_uint2(e4m3x2(f[0] * sc, f[1] * sc) | (e4m3x2(f[2] * sc, f[3] * sc) << 16),
                                   e4m3x2(f[4] * sc, f[5] * sc) | (e4m3x2(f[6] * sc, f[7] * sc) << 16));
    // every lane of a block holds its exponent: byte (lane / 4) % 4, then the
    // stage's four blocks (16 lanes) combined in every lane
    uint32_t w = (uint32_t)(shared + 127) << (8 * ((lane >> 2) & 3));
    w |= __shfl_xor_sync(0xffffffffu, w, 4);
    w |= __shfl_xor_sync(0xffffffffu, w, 8);
    word = w;
    return codes;
}

// Token t's row of x, quantised once, written to its k routes' rows
// inv[t*k + j] (the gather of the routes and the quantisation in one pass).
__global__ void __launch_bounds__(kThreads) gather_mx_kernel(MxActArgs a) {
    ptx::griddep_wait();  // launched early: the permutation is complete past here
    const int lane = threadIdx.x & 31;
    const int64_t T = a.rows / a.k;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int units = a.K / 256;
    const uint4* __restrict__ src = static_cast<const uint4*>(a.src);
    unsigned char* __restrict__ codes = static_cast<unsigned char*>(a.codes);
    uint32_t* __restrict__ scales = static_cast<uint32_t*>(a.scales);
    const int half = lane >> 4, l16 = lane & 15;
    for (int64_t t = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5; t < T; t += nwarps) {
        // lane j < k holds the row of route t*k + j; lanes 16 + j the same
        const int mine = l16 < a.k ? a.inv[t * a.k + l16] : 0;
        if (__any_sync(0xffffffffu, mine < 0 || mine >= a.rows)) {
            if (lane == 0) atomicOr(a.err, kErrCheck);
            continue;
        }
        int rows[kMaxTopK];  // the token's route rows, in every lane (j >= k: unused)
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) rows[j] = __shfl_sync(0xffffffffu, mine, j);
        for (int u0 = 0; u0 < units; u0 += kUnits) {
            uint4 raw[kUnits];
#pragma unroll
            for (int u = 0; u < kUnits; ++u)
                if (u0 + u < units) raw[u] = __ldg(src + (t * a.K + (int64_t)(u0 + u) * 256) / 8 + lane);
#pragma unroll
            for (int u = 0; u < kUnits; ++u) {
                if (u0 + u >= units) break;
                uint32_t word;
                const uint2 c = quantize_unit(raw[u], lane, word);
                const int s = 2 * (u0 + u) + half;  // this half-warp's stage
                const int col = s * 128 + 8 * l16;
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (j < a.k) *reinterpret_cast<uint2*>(codes + (int64_t)rows[j] * a.K + col) = c;
                if (l16 < a.k) scales[(int64_t)s * a.rows_pad + mine] = word;
            }
        }
    }
    ptx::griddep_launch_dependents();
}

int grid_for(int64_t warps_needed, int num_sms) {
    const int64_t want = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t cap = (int64_t)num_sms * 8;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_gather_mx(const MxActArgs& a, cudaStream_t s) {
    if (a.rows == 0) return cudaSuccess;
    if (a.K % 256 != 0) return cudaErrorInvalidValue;  // whole 256-element units (bf16 layers: H % 256 == 0)
    return launch_kernel(gather_mx_kernel, dim3(grid_for(a.rows / a.k, a.num_sms)), dim3(kThreads), 0, s,
                         a.early != 0, a);
}

}  // namespace moe
