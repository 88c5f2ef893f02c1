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
                const uint32_t c = mx_quantize128(raw[u], lane, word);
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
