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
// i), so the words of consecutive rows of one stage are consecutive.
//
// One warp per row: lane l holds elements 4l .. 4l+3 of each 128-element
// stage (one 8-byte load), 8 lanes per 32-block.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// 2^k as an fp32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(1u << (k + 149));
}

__device__ __forceinline__ uint32_t e4m3(float u) {
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(pair) : "f"(u));
    return pair & 0xFFu;
}

// MXFP8 of this lane's four elements of one 128-element stage: returns the
// four codes (byte i = element 4l + i) and, in `word`, the stage's scale word
// (identical in every lane).
__device__ __forceinline__ uint32_t quantize_stage(uint2 raw, int lane, uint32_t& word) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
    float a = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));  // the 8 lanes of a block
    int shared = 0;
    if (a > 0.f) {
        int ex;
        frexpf(a, &ex);  // a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
        shared = min(max(ex - 1 - 8, -127), 127);
    }
    const float s = pow2f(-shared);  // exact: a power-of-two scaling
    const uint32_t codes = e4m3(f0.x * s) | (e4m3(f0.y * s) << 8) | (e4m3(f1.x * s) << 16) | (e4m3(f1.y * s) << 24);
    const uint32_t sc = (uint32_t)(shared + 127);
    word = __shfl_sync(0xffffffffu, sc, 0) | (__shfl_sync(0xffffffffu, sc, 8) << 8) |
           (__shfl_sync(0xffffffffu, sc, 16) << 16) | (__shfl_sync(0xffffffffu, sc, 24) << 24);
    return codes;
}

// Token t's row of x, quantised once, written to its k routes' rows
// inv[t*k + j] (the gather of the routes and the quantisation in one pass).
__global__ void __launch_bounds__(kThreads) gather_mx_kernel(MxActArgs a) {
    ptx::griddep_wait();  // launched early: the permutation is complete past here
    const int lane = threadIdx.x & 31;
    const int64_t T = a.rows / a.k;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int stages = a.K / 128;
    const uint2* __restrict__ src = static_cast<const uint2*>(a.src);
    uint32_t* __restrict__ codes = static_cast<uint32_t*>(a.codes);
    uint32_t* __restrict__ scales = static_cast<uint32_t*>(a.scales);
    for (int64_t t = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5; t < T; t += nwarps) {
        const int dst = lane < a.k ? a.inv[t * a.k + lane] : 0;
        if (__any_sync(0xffffffffu, dst < 0 || dst >= a.rows)) {
            if (lane == 0) atomicOr(a.err, kErrCheck);
            continue;
        }
        for (int s = 0; s < stages; ++s) {
            uint32_t word;
            const uint32_t c = quantize_stage(__ldg(src + (t * a.K + s * 128) / 4 + lane), lane, word);
            for (int j = 0; j < a.k; ++j) {
                const int64_t r = __shfl_sync(0xffffffffu, dst, j);
                codes[(r * a.K + s * 128) / 4 + lane] = c;
                if (lane == 0) scales[(int64_t)s * a.rows_pad + r] = word;
            }
        }
    }
    ptx::griddep_launch_dependents();
}

// Every row of a [rows][K] matrix quantised in place order.
__global__ void __launch_bounds__(kThreads) quantize_rows_mx_kernel(MxActArgs a) {
    ptx::griddep_wait();  // launched early: the rows are complete past here
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int stages = a.K / 128;
    const uint2* __restrict__ src = static_cast<const uint2*>(a.src);
    uint32_t* __restrict__ codes = static_cast<uint32_t*>(a.codes);
    uint32_t* __restrict__ scales = static_cast<uint32_t*>(a.scales);
    for (int64_t r = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5; r < a.rows; r += nwarps) {
        for (int s = 0; s < stages; ++s) {
            uint32_t word;
            const uint32_t c = quantize_stage(src[(r * a.K + s * 128) / 4 + lane], lane, word);
            codes[(r * a.K + s * 128) / 4 + lane] = c;
            if (lane == 0) scales[(int64_t)s * a.rows_pad + r] = word;
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
    return launch_kernel(gather_mx_kernel, dim3(grid_for(a.rows / a.k, a.num_sms)), dim3(kThreads), 0, s,
                         a.early != 0, a);
}

cudaError_t launch_quantize_rows_mx(const MxActArgs& a, cudaStream_t s) {
    if (a.rows == 0) return cudaSuccess;
    if (a.K % 128 != 0) return cudaErrorInvalidValue;
    return launch_kernel(quantize_rows_mx_kernel, dim3(grid_for(a.rows, a.num_sms)), dim3(kThreads), 0, s,
                         a.early != 0, a);
}

}  // namespace moe
