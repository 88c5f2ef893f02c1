// gemm_tc.cu - tcgen05/TMEM grouped GEMMs of the routed experts (sm_103a).
//
// "HunyuanImage3 Hybrid Parallelism", section 6.1/6.2: every micro-shard runs
// grouped GEMM1 -> split gate/up -> SwiGLU -> grouped GEMM2 over the
// expert-sorted routes; the micro partials are added in fp32 and the finalize
// runs once. Ascend Hunyuan Image 3.0 guide, section 2.2: the expert is
// down(SiLU(gate(x)) * up(x)) with w13 = [gate; up].
//
// Two kernels from one template:
//   SwiGLU (GEMM1): a tile is (micro m, expert e, 128 rows, 128 columns of h).
//       Each K stage loads the gate rows [nt*128, +128) and the up rows
//       [I + nt*128, +128) of w13[m][e] into one 256-row B tile (one box of a
//       3D map {H, I, 2E}), so a single
//       M=128 x N=256 MMA fills gate (TMEM columns 0-127) and up (128-255)
//       side by side; the epilogue writes silu(gate) * up as bf16.
//   down (GEMM2): a tile is (expert e, 128 rows, 256 output columns). The K
//       loop runs over micro 0's I columns of h against w2[0][e], then micro
//       1's against w2[1][e], ..., into ONE fp32 TMEM accumulator: the
//       per-micro partial outputs of the pages never exist and the fp32 sum
//       over micros happens inside the tensor core.
//
// Structure: persistent CTAs (one per SM), static round-robin over tiles (see
// decode_tile for their order). 8 warps: warp 0 issues TMA loads into a
// 4-stage ring (128B-swizzled K-major tiles), warp 1 issues tcgen05.mma into
// one of two TMEM accumulators (2 x 256 fp32 columns), warp 2 owns the TMEM
// allocation, warps 4-7 drain an accumulator (one TMEM lane quarter each)
// while the next tile accumulates into the other. All waits are bounded.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kBN = 256;                           // MMA N
constexpr int kABytes = kTcBM * kTcBK * 2;         // 16 KB
constexpr int kBBytes = kBN * kTcBK * 2;           // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;     // 48 KB
constexpr int kTmemCols = 2 * kBN;                 // two accumulators
constexpr int kThreads = 256;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTcBM, kBN);

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
};

constexpr int kSmemBytes = kStages * kStageBytes + (int)sizeof(Ctl) + 1024;

// Row blocks of a (group, micro) with more than kRowChunk of them run in
// chunks: every n-tile of chunk 0, then every n-tile of chunk 1, ... A
// chunk's activation rows (16 MB at K = 4096) then stay in L2 while the
// n-tiles sweep them; in the plain order a large group (the dense shared
// expert: 256 row blocks, 268 MB of x) re-read all its rows from DRAM once per
// n-tile. Smaller groups keep the plain order (n-tile, then row block).
constexpr int kRowChunk = 16;

template <bool SWIGLU>
__device__ __forceinline__ Tile decode_tile(int tile, const Ctl& c, const TcGemmArgs& a) {
    Tile t = decode_group_tile(tile, c.seg, c.tiles, a.G, a.n_tiles, a.n_micro, SWIGLU, kTcBM);
    const int mtiles = c.tiles[t.g + 1] - c.tiles[t.g];
    if (mtiles <= kRowChunk) return t;
    // the tile's index within its (group, micro) in the plain order, mapped
    // onto the chunked order (full chunks of kRowChunk row blocks, then the rest)
    const int local = t.nt * mtiles + (t.row0 - c.seg[t.g]) / kTcBM;
    const int span = kRowChunk * a.n_tiles, nfull = mtiles / kRowChunk;
    const int chunk = min(local / span, nfull);
    const int rows = chunk < nfull ? kRowChunk : mtiles - nfull * kRowChunk;
    const int off = local - chunk * span;
    t.nt = off / rows;
    t.row0 = c.seg[t.g] + (chunk * kRowChunk + off % rows) * kTcBM;
    return t;
}

__device__ __forceinline__ void fail(Ctl& c, int* err) {
    c.abort = 1;
    atomicOr(err, kErrTimeout);
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmB3, const TcGemmArgs a) {
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
    // launched early (a.early): the segments and A rows are complete past here.
    // No early trigger for the next kernel: it starts when this grid ends (a
    // trigger at the last tile let the finalize's waiting blocks crowd the last
    // tiles and measured slower on the long steps)
    ptx::griddep_wait();
    if (a.seg != nullptr) {
        for (int i = threadIdx.x; i <= a.G; i += kThreads) {
            c.seg[i] = a.seg[i];
            c.tiles[i] = a.tiles[i];
        }
    } else if (threadIdx.x == 0) {  // one dense segment (the shared expert over all T rows)
        c.seg[0] = 0;
        c.seg[1] = a.dense_rows;
        c.tiles[0] = 0;
        c.tiles[1] = (a.dense_rows + kTcBM - 1) / kTcBM;
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB0);
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
        uint32_t phase = 0;
        uint32_t last_par[kStages];
        int issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode_tile<SWIGLU>(tile, c, a);
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = SWIGLU ? t.m : mi;
                const CUtensorMap* tb = pick_map(m, tmB0, tmB1, tmB2, tmB3);
                const int brow = t.g * a.b_rows_per_group + t.nt * kBN;  // down tiles
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, a.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
                    const uint32_t fb = ptx::smem_u32(&c.full[stage]);
                    ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                    const int ka = (SWIGLU ? 0 : m * a.a_micro_cols) + kb * kTcBK;
                    ptx::tma_load_2d(sa, &tmA, ka, t.row0, fb);
                    // one box per operand: the TMA instructions, not the bytes, set the
                    // producer's pace (SwiGLU: 128 gate rows, then the matching up
                    // rows, as half 2g + 1 of the 3D map; down: 256 rows)
                    if (SWIGLU)
                        ptx::tma_load_3d(sb, tb, kb * kTcBK, t.nt * 128, 2 * t.g, fb);
                    else
                        ptx::tma_load_2d(sb, tb, kb * kTcBK, brow, fb);
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
            // let every load still in flight land before the CTA can exit
            const int n = issued < kStages ? issued : kStages;
            for (int s = 0; s < n; ++s)
                ptx::mbar_wait(ptx::smem_u32(&c.full[s]), last_par[s], a.limit_ns, nullptr);
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
            const uint32_t d = tmem + (uint32_t)(acc * kBN);
            uint32_t accumulate = 0;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.full[stage]), phase, a.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint64_t adesc = ptx::sw128_desc(sa);
                    const uint64_t bdesc = ptx::sw128_desc(sa + kABytes);
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
        // every MMA issued so far completes before TMEM can be released
        ptx::mma_commit(ptx::smem_u32(&c.drain));
        ptx::mbar_wait(ptx::smem_u32(&c.drain), 0, a.limit_ns, nullptr);
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int q = warp - 4;  // TMEM lanes 32q .. 32q+31 = tile rows
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
        int local = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            const Tile t = decode_tile<SWIGLU>(tile, c, a);
            bool ready = false;
            if (lane == 0)
                ready = ptx::mbar_wait(ptx::smem_u32(&c.tfull[acc]), acc_par, a.limit_ns, &c.abort);
            ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
            if (!ready) {
                if (lane == 0) fail(c, a.err);
                break;
            }
            ptx::tc_fence_after();
            const int grow = t.row0 + q * 32 + lane;
            const bool valid = grow < t.row_end;
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
            if (SWIGLU) {
                __nv_bfloat16* dst = out + (int64_t)grow * a.out_ld + (int64_t)t.m * a.out_micro_cols + t.nt * 128;
#pragma unroll 1
                for (int col = 0; col < 128; col += 32) {
                    uint32_t g[32], u[32];
                    ptx::tmem_ld32(tbase + col, g);
                    ptx::tmem_ld32(tbase + 128 + col, u);
                    uint32_t p[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                        const float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                        p[i] = pack_bf16x2(h0, h1);
                    }
                    if (valid) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
                    }
                }
            } else {
                __nv_bfloat16* dst = out + (int64_t)grow * a.out_ld + t.nt * kBN;
#pragma unroll 1
                for (int col = 0; col < kBN; col += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + col, v);
                    uint32_t p[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    if (valid) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
                    }
                }
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
cudaError_t launch_tc(const TcGemmArgs& a, const CUtensorMap& tmA, const CUtensorMap* tmB, int num_sms,
                      cudaStream_t s) {
    if (a.max_tiles <= 0) return cudaSuccess;
    if (cudaError_t e = ensure_smem_limit<tc_gemm_kernel<SWIGLU>>(kSmemBytes); e != cudaSuccess) return e;
    const int grid = a.max_tiles < num_sms ? a.max_tiles : num_sms;
    const CUtensorMap& b1 = a.n_micro > 1 ? tmB[1] : tmB[0];
    const CUtensorMap& b2 = a.n_micro > 2 ? tmB[2] : tmB[0];
    const CUtensorMap& b3 = a.n_micro > 3 ? tmB[3] : tmB[0];
    return launch_kernel(tc_gemm_kernel<SWIGLU>, dim3(grid), dim3(kThreads), kSmemBytes, s, a.early != 0, tmA,
                         tmB[0], b1, b2, b3, a);
}

}  // namespace

cudaError_t launch_tc_gemm_swiglu(const TcGemmArgs& a, const CUtensorMap& tmA, const CUtensorMap* tmB,
                                  int num_sms, cudaStream_t s) {
    return launch_tc<true>(a, tmA, tmB, num_sms, s);
}

cudaError_t launch_tc_gemm_down(const TcGemmArgs& a, const CUtensorMap& tmA, const CUtensorMap* tmB,
                                int num_sms, cudaStream_t s) {
    return launch_tc<false>(a, tmA, tmB, num_sms, s);
}

}  // namespace moe
