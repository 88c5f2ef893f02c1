// gemm_small.cu - the grouped GEMMs for batches of at most 16 tokens
// (AR-decode-sized calls), with the operands swapped.
//
// Same computation as gemm_tc.cu ("HunyuanImage3 Hybrid Parallelism",
// section 6.1: per micro grouped GEMM1 -> SwiGLU -> grouped GEMM2, micros
// summed in fp32), but with T <= 16 every expert owns at most 16 routes, so
// the expert WEIGHTS take the MMA's M side (128 rows) and the expert's token
// rows its N side (N = 16): each K stage moves 16 KB of weights and 2 KB of
// activations instead of 16 KB of mostly-padding activation rows. The layer is
// then a weight stream, bounded by HBM bandwidth.
//   SwiGLU (GEMM1): a tile is (expert e, micro m, 64 columns of h): the A
//       tile stacks 64 gate rows of w13[m][e] over the matching 64 up rows,
//       so TMEM lanes 0-63 hold gate and 64-127 up for the 16 tokens; the
//       epilogue pairs them through shared memory and writes silu(gate) * up.
//   down (GEMM2): a tile is (expert e, 128 output columns), K runs over all
//       micros into one accumulator.
// Persistent CTAs, 8-stage TMA ring, one MMA issuer, four epilogue warps on a
// double-buffered 2 x 16-column TMEM accumulator. All waits are bounded.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTok = kSmallTokens;             // 16: MMA N
constexpr int kM = 128;                        // MMA M: weight rows
constexpr int kStages = 8;
constexpr int kABytes = kM * kTcBK * 2;        // 16 KB
constexpr int kBBytes = kTok * kTcBK * 2;      // 2 KB
constexpr int kStageBytes = kABytes + kBBytes; // 18 KB (a multiple of 1024)
constexpr int kTmemCols = 32;                  // 2 accumulators x 16 columns
constexpr int kThreads = 256;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kM, kTok);

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int seg[kMaxExperts + 1];
    int tiles[kMaxExperts + 1];
    float up[64][kTok + 1];
    int ep_ok[4];
};

constexpr int kSmemBytes = kStages * kStageBytes + (int)sizeof(Ctl) + 1024;

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void fail(Ctl& c, int* err) {
    c.abort = 1;
    atomicOr(err, kErrTimeout);
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
    tc_small_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                    const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                    const __grid_constant__ CUtensorMap tmW3, const TcGemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl& c = *reinterpret_cast<Ctl*>(smem + kStages * kStageBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&c.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&c.tfull[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.tempty[b]), 4);
        }
        ptx::mbar_init(ptx::smem_u32(&c.drain), 1);
        c.abort = 0;
        ptx::fence_mbar_init();
    }
    for (int i = threadIdx.x; i <= a.G; i += kThreads) {
        c.seg[i] = a.seg[i];
        c.tiles[i] = a.tiles[i];
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmW0);
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_u32(&c.tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const uint32_t tmem = c.tmem_base;
    const int total = (SWIGLU ? a.n_micro : 1) * c.tiles[a.G] * a.n_tiles;
    const int n_micro_k = SWIGLU ? 1 : a.n_micro;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0, last_par[kStages];
        int issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode_group_tile(tile, c.seg, c.tiles, a.G, a.n_tiles, a.n_micro, SWIGLU, kTcBM);
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = SWIGLU ? t.m : mi;
                const CUtensorMap* tw = pick_map(m, tmW0, tmW1, tmW2, tmW3);
                const int wrow = t.g * a.b_rows_per_group + t.nt * (SWIGLU ? 64 : kM);
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, a.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint32_t fb = ptx::smem_u32(&c.full[stage]);
                    ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                    if (SWIGLU) {
                        ptx::tma_load_2d(sa, tw, kb * kTcBK, wrow, fb);                       // 64 gate rows
                        ptx::tma_load_2d(sa + kABytes / 2, tw, kb * kTcBK, wrow + a.up_offset, fb);  // 64 up rows
                    } else {
                        ptx::tma_load_2d(sa, tw, kb * kTcBK, wrow, fb);                       // 128 rows
                    }
                    const int kx = (SWIGLU ? 0 : m * a.a_micro_cols) + kb * kTcBK;
                    ptx::tma_load_2d(sa + kABytes, &tmX, kx, t.row0, fb);                      // 16 token rows
                    last_par[stage] = phase;
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (!ok) {
            fail(c, a.err);
            const int n = issued < kStages ? issued : kStages;
            for (int s = 0; s < n; ++s) ptx::mbar_wait(ptx::smem_u32(&c.full[s]), last_par[s], a.limit_ns, nullptr);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int local = 0;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            if (!ptx::mbar_wait(ptx::smem_u32(&c.tempty[acc]), acc_par ^ 1u, a.limit_ns, &c.abort)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * kTok);
            uint32_t accumulate = 0;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.full[stage]), phase, a.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint64_t adesc = ptx::sw128_desc(sa), bdesc = ptx::sw128_desc(sa + kABytes);
#pragma unroll
                    for (int k = 0; k < kTcBK / 16; ++k) {
                        ptx::mma_bf16(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, accumulate);
                        accumulate = 1;
                    }
                    ptx::mma_commit(ptx::smem_u32(&c.empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok) ptx::mma_commit(ptx::smem_u32(&c.tfull[acc]));
        }
        if (!ok) fail(c, a.err);
        ptx::mma_commit(ptx::smem_u32(&c.drain));
        ptx::mbar_wait(ptx::smem_u32(&c.drain), 0, a.limit_ns, nullptr);
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int q = warp - 4;            // TMEM lanes 32q .. 32q+31 = weight rows
        const int r = q * 32 + lane;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
        int local = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            const Tile t = decode_group_tile(tile, c.seg, c.tiles, a.G, a.n_tiles, a.n_micro, SWIGLU, kTcBM);
            bool ready = false;
            if (lane == 0)
                ready = ptx::mbar_wait(ptx::smem_u32(&c.tfull[acc]), acc_par, a.limit_ns, &c.abort);
            ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
            if (SWIGLU) {
                // the four epilogue warps meet at named barriers below, so they
                // take the continue-or-stop decision together
                if (lane == 0) c.ep_ok[q] = ready ? 1 : 0;
                epilogue_bar();
                ready = c.ep_ok[0] && c.ep_ok[1] && c.ep_ok[2] && c.ep_ok[3];
            }
            if (!ready) {
                if (lane == 0) fail(c, a.err);
                break;
            }
            ptx::tc_fence_after();
            uint32_t v[kTok];
            ptx::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kTok), v);
            const int cnt = min(kTok, t.row_end - t.row0);
            if (SWIGLU) {
                if (q >= 2) {
#pragma unroll
                    for (int j = 0; j < kTok; ++j) c.up[r - 64][j] = __uint_as_float(v[j]);
                }
                epilogue_bar();
                if (q < 2) {
                    const int64_t col = (int64_t)t.m * a.out_micro_cols + t.nt * 64 + r;
                    for (int j = 0; j < cnt; ++j) {
                        const float h = silu(__uint_as_float(v[j])) * c.up[r][j];
                        out[(int64_t)(t.row0 + j) * a.out_ld + col] = __float2bfloat16_rn(h);
                    }
                }
                epilogue_bar();
            } else {
                const int64_t col = (int64_t)t.nt * kM + r;
                for (int j = 0; j < cnt; ++j)
                    out[(int64_t)(t.row0 + j) * a.out_ld + col] = __float2bfloat16_rn(__uint_as_float(v[j]));
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&c.tempty[acc]));
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool SWIGLU>
cudaError_t launch_small(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW, int num_sms,
                         cudaStream_t s) {
    if (a.max_tiles <= 0) return cudaSuccess;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tc_small_kernel<SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int grid = a.max_tiles < num_sms ? a.max_tiles : num_sms;
    const CUtensorMap& w1 = a.n_micro > 1 ? tmW[1] : tmW[0];
    const CUtensorMap& w2 = a.n_micro > 2 ? tmW[2] : tmW[0];
    const CUtensorMap& w3 = a.n_micro > 3 ? tmW[3] : tmW[0];
    tc_small_kernel<SWIGLU><<<grid, kThreads, kSmemBytes, s>>>(tmX, tmW[0], w1, w2, w3, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_small_swiglu(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW,
                                   int num_sms, cudaStream_t s) {
    return launch_small<true>(a, tmX, tmW, num_sms, s);
}

cudaError_t launch_tc_small_down(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW,
                                 int num_sms, cudaStream_t s) {
    return launch_small<false>(a, tmX, tmW, num_sms, s);
}

}  // namespace moe
