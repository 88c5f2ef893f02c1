// router.cu - the gate: fp32 router logits, softmax top-k with renormalised
// routing scales, and the per-block expert histogram that seeds the route sort.
//
// "HunyuanImage3 Hybrid Parallelism", section 6.1: the router yields expert ids
// and routing scores of shape [num_tokens, top_k]. Ascend Hunyuan Image 3.0
// guide, section 5.2: the gate runs in fp32. Softmax over all experts, top-k,
// then renormalisation of the k scales is the reading this layer takes.
//
// One block scores kRouterTokens tokens against all E <= 64 experts: a tiled
// fp32 SIMT product (x and Wr tiles staged in shared memory, 4 tokens x 4
// experts per thread), then one warp per token selects the top-k.
#include <cuda_bf16.h>

#include <cfloat>
#include <climits>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 128;  // 16 expert groups x 8 token groups
constexpr int kBK = 32;        // K chunk staged per iteration

template <typename TIn>
__device__ __forceinline__ void load8(const TIn* p, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// (v, e) ranks above (v2, e2): larger logit, then lower expert index.
__device__ __forceinline__ bool ranks_above(float v, int e, float v2, int e2) {
    return v > v2 || (v == v2 && e < e2);
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads) router_kernel(RouterArgs a) {
    __shared__ __align__(16) float xs[kBK][kRouterTokens];     // [k][token]
    __shared__ __align__(16) float ws[kBK][kMaxExperts];       // [k][expert]
    __shared__ float lg[kRouterTokens][kMaxExperts + 1];
    __shared__ int hist[kMaxExperts];

    const TIn* x = static_cast<const TIn*>(a.x);
    const TIn* wr = static_cast<const TIn*>(a.wr);
    const int tid = threadIdx.x;
    const int tx = tid % 16;  // experts 4tx..4tx+3
    const int ty = tid / 16;  // tokens 4ty..4ty+3
    const int t0 = blockIdx.x * kRouterTokens;
    const int H = a.H, E = a.E;

    if (tid < kMaxExperts) hist[tid] = 0;

    // Each 32-wide K chunk is summed in fp32, and chunk sums are combined with
    // compensated (Kahan) addition, so a logit lands within a few ulps of the
    // exact dot product and near-ties between experts stay rare.
    float sum[4][4], comp[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sum[i][j] = comp[i][j] = 0.f;

    for (int k0 = 0; k0 < H; k0 += kBK) {
        // x tile: 32 tokens x 32 k = 128 loads of 8 elements
        {
            const int tok = tid / 4, kk = (tid % 4) * 8;
            float v[8];
            const int t = t0 + tok;
            if (t < a.T) {
                load8<TIn>(x + (int64_t)t * H + k0 + kk, v);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) xs[kk + i][tok] = v[i];
        }
        // Wr tile: 64 experts x 32 k = 256 loads of 8 elements
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
            const int idx = tid + rep * kThreads;
            const int e = idx / 4, kk = (idx % 4) * 8;
            float v[8];
            if (e < E) {
                load8<TIn>(wr + (int64_t)e * H + k0 + kk, v);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) ws[kk + i][e] = v[i];
        }
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 8
        for (int kk = 0; kk < kBK; ++kk) {
            const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][4 * ty]);
            const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][4 * tx]);
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
            const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float y = acc[i][j] - comp[i][j];
                const float t = sum[i][j] + y;
                comp[i][j] = (t - sum[i][j]) - y;
                sum[i][j] = t;
            }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = 4 * tx + j;
            float v = sum[i][j];
            if (a.bias != nullptr && e < E) v += a.bias[e];
            lg[4 * ty + i][e] = v;
            const int t = t0 + 4 * ty + i;
            if (a.logits != nullptr && t < a.T && e < E) a.logits[(int64_t)t * E + e] = v;
        }
    __syncthreads();

    // top-k: one warp per token
    const int warp = tid / 32, lane = tid % 32;
    for (int tl = warp; tl < kRouterTokens; tl += kThreads / 32) {
        const int t = t0 + tl;
        if (t >= a.T) break;
        const int e0 = lane, e1 = lane + 32;
        const float v0 = e0 < E ? lg[tl][e0] : -FLT_MAX;
        const float v1 = e1 < E ? lg[tl][e1] : -FLT_MAX;
        bool taken0 = e0 >= E, taken1 = e1 >= E;
        int my_e = 0;
        float my_v = 0.f;
        for (int j = 0; j < a.k; ++j) {
            float bv = -INFINITY;
            int be = INT_MAX;
            if (!taken0) { bv = v0; be = e0; }
            if (!taken1 && (be == INT_MAX || ranks_above(v1, e1, bv, be))) { bv = v1; be = e1; }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (oe != INT_MAX && (be == INT_MAX || ranks_above(ov, oe, bv, be))) { bv = ov; be = oe; }
            }
            if (be < 0 || be >= E) {  // only NaN logits can leave no winner
                if (lane == 0) atomicOr(a.err, kErrCheck);
                be = 0;
            }
            if (be == e0) taken0 = true;
            if (be == e1) taken1 = true;
            if (lane == j) { my_e = be; my_v = bv; }
        }
        // renormalised softmax over the selected k: exp(l_j - l_max) / sum
        const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
        const float ex = lane < a.k ? expf(my_v - vmax) : 0.f;
        float den = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        if (lane < a.k) {
            a.ids[(int64_t)t * a.k + lane] = my_e;
            a.w[(int64_t)t * a.k + lane] = ex / den;
            atomicAdd(&hist[my_e], 1);
        }
    }
    __syncthreads();
    if (tid < E) a.blk_hist[(int64_t)blockIdx.x * E + tid] = hist[tid];
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
    const int nb = (a.T + kRouterTokens - 1) / kRouterTokens;
    if (nb == 0) return cudaSuccess;
    if (a.bf16)
        router_kernel<__nv_bfloat16><<<nb, kThreads, 0, s>>>(a);
    else
        router_kernel<float><<<nb, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
