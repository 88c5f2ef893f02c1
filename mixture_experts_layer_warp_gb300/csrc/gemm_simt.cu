// gemm_simt.cu - exact-fp32 grouped GEMMs for fp32 layers.
//
// tcgen05 has no fp32-input MMA and tf32 rounding (about 2^-11) would break a
// 1e-5 output tolerance, so fp32 layers run these FFMA kernels. They compute
// the same two grouped GEMMs as the tensor-core path (the multi-micro layer of
// "HunyuanImage3 Hybrid Parallelism", section 6.1):
//   SwiGLU form: out[r][m*I + n] = silu(A_r . G_m,e[n]) * (A_r . U_m,e[n])
//   down form:   out[r][n]       = sum_m A_r[m*I : (m+1)*I] . D_m,e[n]
// for rows r of expert e's segment. Tile: 32 rows x 64 columns, K staged in
// shared memory 32 at a time, 2 rows x 4 columns per thread.
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBM = kSimtBM;  // 32
constexpr int kBN = 64;
constexpr int kBK = 32;
constexpr int kThreads = 256;

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads) simt_gemm_kernel(SimtGemmArgs a) {
    __shared__ float As[kBK][kBM + 1];
    __shared__ float Gs[kBK][kBN + 1];
    __shared__ float Us[SWIGLU ? kBK : 1][kBN + 1];

    const int tile = blockIdx.y;
    if (tile >= a.tiles[a.G]) return;
    int g = 0;
    while (g + 1 < a.G && a.tiles[g + 1] <= tile) ++g;
    const int row0 = a.seg[g] + (tile - a.tiles[g]) * kBM;
    const int row_end = a.seg[g + 1];
    const int n0 = blockIdx.x * kBN;
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;  // columns 4tx.., rows 2ty..

    float acc_g[2][4] = {}, acc_u[2][4] = {};
    const int m_first = SWIGLU ? blockIdx.z : 0;
    const int m_last = SWIGLU ? blockIdx.z + 1 : a.n_micro;
    for (int m = m_first; m < m_last; ++m) {
        const float* B = a.b[m] + (int64_t)g * a.b_rows_per_group * a.K;
        const int a_col0 = SWIGLU ? 0 : m * a.a_micro_cols;
        for (int k0 = 0; k0 < a.K; k0 += kBK) {
            for (int i = tid; i < kBM * kBK; i += kThreads) {
                const int r = i / kBK, kk = i % kBK;
                const int row = row0 + r;
                As[kk][r] = row < row_end ? a.a[(int64_t)row * a.lda + a_col0 + k0 + kk] : 0.f;
            }
            for (int i = tid; i < kBN * kBK; i += kThreads) {
                const int c = i / kBK, kk = i % kBK;
                Gs[kk][c] = B[(int64_t)(n0 + c) * a.K + k0 + kk];
                if (SWIGLU) Us[kk][c] = B[(int64_t)(a.N + n0 + c) * a.K + k0 + kk];
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < kBK; ++kk) {
                const float x0 = As[kk][2 * ty], x1 = As[kk][2 * ty + 1];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float gv = Gs[kk][4 * tx + j];
                    acc_g[0][j] = fmaf(x0, gv, acc_g[0][j]);
                    acc_g[1][j] = fmaf(x1, gv, acc_g[1][j]);
                    if (SWIGLU) {
                        const float uv = Us[kk][4 * tx + j];
                        acc_u[0][j] = fmaf(x0, uv, acc_u[0][j]);
                        acc_u[1][j] = fmaf(x1, uv, acc_u[1][j]);
                    }
                }
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int row = row0 + 2 * ty + i;
        if (row >= row_end) continue;
        float* out = a.out + (int64_t)row * a.out_ld + (SWIGLU ? blockIdx.z * a.out_micro_cols : 0) + n0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            out[4 * tx + j] = SWIGLU ? silu(acc_g[i][j]) * acc_u[i][j] : acc_g[i][j];
    }
}

cudaError_t launch(const SimtGemmArgs& a, bool swiglu, cudaStream_t s) {
    if (a.max_tiles == 0) return cudaSuccess;
    dim3 grid(a.N / kBN, a.max_tiles, swiglu ? a.n_micro : 1);
    if (swiglu)
        simt_gemm_kernel<true><<<grid, kThreads, 0, s>>>(a);
    else
        simt_gemm_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_gemm_swiglu(const SimtGemmArgs& a, cudaStream_t s) { return launch(a, true, s); }
cudaError_t launch_simt_gemm_down(const SimtGemmArgs& a, cudaStream_t s) { return launch(a, false, s); }

}  // namespace moe
