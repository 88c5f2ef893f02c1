// finalize.cu - the single unpermute, routing-scale and top-k reduction.
//
// "HunyuanImage3 Hybrid Parallelism", section 6.1: the finalize reads the
// expert outputs by original token and top-k slot and forms
//     output[token] = sum over routes of routing_scale[token, route] * partial,
// adding in fp32, applying the scale once and reducing over top-k once. Here
// the per-micro partials were already summed in the GEMM2 accumulator, so
// each route contributes one row o[inv[t*k + j]]. The shared expert's output
// (Ascend Hunyuan Image 3.0 guide, section 3.1) is added unscaled, and with
// output accumulation on, the previous content of y as well.
//
// HBM-bound: one block per (token, 1024-column chunk), 16-byte vector loads
// of the k expert rows, two rows in flight per thread with the streaming hint
// (each o row is read once). One row at a time left the kernel at 0.81-0.86
// of the HBM bandwidth (55.2 -> 46.9 us at T = 4096, 457 -> 421 us at the CFG
// size); all eight rows at once took 60-80 registers, cut the resident
// threads per SM and ran slower.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// acc += s * row for the bf16 rows of two routes (j0, j0 + 1 when both < k),
// both loads issued before the arithmetic; fp32 in route order.
__device__ __forceinline__ void add_rows(const __nv_bfloat16* o, const int64_t* rows, const float* scale, int j0, int k,
                                         int64_t H, int v, float (&acc)[8]) {
    uint4 raw[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
        if (j0 + j < k) raw[j] = __ldcs(reinterpret_cast<const uint4*>(o + rows[j0 + j] * H + v * 8));
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        if (j0 + j < k) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
            const float s = scale[j0 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                acc[2 * i] = fmaf(s, f.x, acc[2 * i]);
                acc[2 * i + 1] = fmaf(s, f.y, acc[2 * i + 1]);
            }
        }
    }
}

// fp32 rows (the exact-fp32 layer): one route at a time.
__device__ __forceinline__ void add_rows(const float* o, const int64_t* rows, const float* scale, int j0, int k,
                                         int64_t H, int v, float (&acc)[8]) {
    for (int j = j0; j < j0 + 2 && j < k; ++j) {
        float val[8];
        load8(o + rows[j] * H + v * 8, val);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(scale[j], val[i], acc[i]);
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) finalize_kernel(FinalizeArgs a) {
    __shared__ int64_t rows[kMaxTopK];
    __shared__ float scale[kMaxTopK];
    ptx::griddep_wait();  // launched early: the expert outputs are complete past here
    const int t = blockIdx.x;
    const int64_t R = (int64_t)a.T * a.k;
    if (threadIdx.x < a.k) {
        int64_t r = a.inv[(int64_t)t * a.k + threadIdx.x];
        if (r < 0 || r >= R) {  // unreachable for a valid permutation: reported, never dereferenced
            if (a.err != nullptr) atomicOr(a.err, kErrCheck);
            r = 0;
        }
        rows[threadIdx.x] = r;
        scale[threadIdx.x] = a.w[(int64_t)t * a.k + threadIdx.x];
    }
    __syncthreads();
    const T* o = static_cast<const T*>(a.o);
    const T* sh = static_cast<const T*>(a.shared);
    T* y = static_cast<T*>(a.y);
    const int nv = a.H / 8;
    const int v = blockIdx.y * kThreads + threadIdx.x;  // one 8-element vector per thread
    if (v < nv) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < a.k; j0 += 2) add_rows(o, rows, scale, j0, a.k, a.H, v, acc);
        if (sh != nullptr) {
            float val[8];
            load8(sh + (int64_t)t * a.H + v * 8, val);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += val[i];
        }
        if (a.accumulate) {
            float val[8];
            load8(y + (int64_t)t * a.H + v * 8, val);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += val[i];
        }
        store8(y + (int64_t)t * a.H + v * 8, acc);
    }
    ptx::griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    const dim3 grid(a.T, (a.H / 8 + kThreads - 1) / kThreads);
    return a.bf16 ? launch_kernel(finalize_kernel<__nv_bfloat16>, grid, dim3(kThreads), 0, s, a.early != 0, a)
                  : launch_kernel(finalize_kernel<float>, grid, dim3(kThreads), 0, s, a.early != 0, a);
}

}  // namespace moe
