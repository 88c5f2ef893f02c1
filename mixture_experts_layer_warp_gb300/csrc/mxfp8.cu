// mxfp8.cu - block-scaled FP8 (MXFP8) quantisation of bf16 expert weights.
//
// The experts' block-scaled FP8 variant reads its weights in the OCP
// Microscaling MXFP8 format: E4M3 codes and one E8M0 power-of-two scale per
// 32 consecutive elements along K. For each block: shared exponent =
// floor(log2(max |v|)) - 8 (8 is the largest exponent of E4M3), clamped to
// [-127, 127] (an all-zero block gets 0); code = E4M3 of v / 2^shared,
// nearest with ties to even, saturating at +-448; scale code = shared + 127.
// One warp quantises one block (lane i holds element i).
#include <cuda_bf16.h>

#include "kernels.h"

namespace moe {
namespace {

// 2^k as an fp32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(1u << (k + 149));
}

__global__ void __launch_bounds__(256) mx_quantize_kernel(const __nv_bfloat16* __restrict__ w, int64_t blocks,
                                                          int rows, int nb, uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; blk < blocks; blk += warps) {
        const int64_t gr = blk / nb, b = blk % nb;  // (group, row) and the block along K
        const int64_t at = gr * (int64_t)nb * 32 + b * 32 + lane;
        const float v = __bfloat162float(w[at]);
        float a = fabsf(v);
#pragma unroll
        for (int d = 16; d; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
        int shared = 0;
        if (a > 0.f) {
            int ex;
            frexpf(a, &ex);  // a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
            shared = min(max(ex - 1 - 8, -127), 127);
        }
        const float u = v * pow2f(-shared);  // exact: a power-of-two scaling below 512
        uint16_t pair;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(pair) : "f"(u));
        codes[at] = (uint8_t)(pair & 0xFFu);
        if (lane == 0) {
            const int64_t g = gr / rows, r = gr % rows;
            scales[(g * nb + b) * rows + r] = (uint8_t)(shared + 127);
        }
    }
}

}  // namespace

cudaError_t launch_mx_quantize(const void* w, int64_t groups, int rows, int cols, void* codes, void* scales,
                               int num_sms, cudaStream_t s) {
    const int nb = cols / 32;
    const int64_t blocks = groups * (int64_t)rows * nb;
    if (blocks <= 0) return cudaSuccess;
    const int64_t want = (blocks + 7) / 8;  // eight warps per CTA
    const int grid = (int)(want < (int64_t)num_sms * 16 ? want : (int64_t)num_sms * 16);
    mx_quantize_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w), blocks, rows, nb,
                                            static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales));
    return cudaGetLastError();
}

}  // namespace moe
