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
// One warp per row part: lane l holds elements 4l .. 4l+3 of each
// 128-element stage (one 8-byte load), 8 lanes per 32-block. A warp loads
// kBatch stages before it quantises them, so that several loads per lane are
// in flight.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 4;  // stages loaded ahead per warp


// MXFP8 of this lane's four elements of one 128-element stage: returns the
// four codes (byte i = element 4l + i) and, in `word`, the stage's scale word
// (identical in every lane).
__device__ __forceinline__ uint32_t quantize_stage(uint2 raw, int lane, uint32_t& word) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
    float a = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));  // the 8 lanes of a block
    const int shared = mx_shared_exp(a);
    const float s = pow2f(-shared);  // exact: a power-of-two scaling
    const uint32_t codes = e4m3x2(f0.x * s, f0.y * s) | (e4m3x2(f1.x * s, f1.y * s) << 16);
    // byte b of the word: the scale of block b, from the first lane of its 8
    const uint32_t sc = (lane & 7) == 0 ? (uint32_t)(shared + 127) << (8 * (lane >> 3)) : 0u;
    word = __reduce_or_sync(0xffffffffu, sc);
    return codes;
}

// The gather splits a token's stages into parts of kPartStages, one warp per
// (token, part): one warp per token (4096 at the denoise size) left too few
// warps in flight to cover the latency of the quantisation's dependent
// shuffles and conversions (78 -> 61 us).
constexpr int kPartStages = 8;

__device__ __forceinline__ int parts_of(int stages) { return (stages + kPartStages - 1) / kPartStages; }

// Token t's row of x, quantised once, written to its k routes' rows
// inv[t*k + j] (the gather of the routes and the quantisation in one pass).
__global__ void __launch_bounds__(kThreads) gather_mx_kernel(MxActArgs a) {
    ptx::griddep_wait();  // launched early: the permutation is complete past here
    const int lane = threadIdx.x & 31;
    const int64_t T = a.rows / a.k;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int stages = a.K / 128, P = parts_of(stages);
    const uint2* __restrict__ src = static_cast<const uint2*>(a.src);
    uint32_t* __restrict__ codes = static_cast<uint32_t*>(a.codes);
    uint32_t* __restrict__ scales = static_cast<uint32_t*>(a.scales);
    for (int64_t item = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5; item < T * P; item += nwarps) {
        const int64_t t = item / P;
        const int s_lo = (int)(item % P) * kPartStages;
        const int s_hi = s_lo + kPartStages < stages ? s_lo + kPartStages : stages;
        const int dst = lane < a.k ? a.inv[t * a.k + lane] : 0;
        if (__any_sync(0xffffffffu, dst < 0 || dst >= a.rows)) {
            if (lane == 0) atomicOr(a.err, kErrCheck);
            continue;
        }
        int64_t rows[kMaxTopK];  // the token's route rows, in every lane
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) rows[j] = __shfl_sync(0xffffffffu, dst, j);
        for (int s0 = s_lo; s0 < s_hi; s0 += kBatch) {
            uint2 raw[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (s0 + u < s_hi) raw[u] = __ldg(src + (t * a.K + (s0 + u) * 128) / 4 + lane);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int s = s0 + u;
                if (s >= s_hi) break;
                uint32_t word;
                const uint32_t c = quantize_stage(raw[u], lane, word);
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j) {
                    if (j >= a.k) break;
                    codes[(rows[j] * a.K + s * 128) / 4 + lane] = c;
                    if (lane == j) scales[(int64_t)s * a.rows_pad + rows[j]] = word;
                }
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
    if (a.K % 128 != 0) return cudaErrorInvalidValue;
    const int64_t parts = (a.K / 128 + kPartStages - 1) / kPartStages;
    return launch_kernel(gather_mx_kernel, dim3(grid_for(a.rows / a.k * parts, a.num_sms)), dim3(kThreads), 0, s,
                         a.early != 0, a);
}

}  // namespace moe
