// router_tc.cu - the gate of bf16 layers on the 5th-generation tensor core.
//
// "HunyuanImage3 Hybrid Parallelism", section 6.1: the router yields expert ids
// and routing scores of shape [num_tokens, top_k]; Ascend Hunyuan Image 3.0
// guide, section 5.2: the gate is computed in fp32. Reading taken: softmax over
// all experts, top-k (ties to the lower index), renormalised k weights.
//
// One CTA scores 128 tokens against all E <= 64 experts: x [128 x H] and
// Wr [64 x H] stream through a 6-stage TMA ring (128B-swizzled K-major tiles)
// into tcgen05.mma M=128 x N=64. K-block kb accumulates into TMEM partial
// kb % 8, and the epilogue adds the eight partials with compensated (Kahan)
// addition, so each fp32 logit stays within a few ulps of the exact dot
// product and near-ties between experts stay rare. Each thread then owns one
// token (its TMEM lane): softmax top-k over its 64 logits, renormalised
// weights, and the CTA's expert histogram. When one CTA covers all tokens
// (T <= 128: decode-sized batches) it also computes the offsets and places
// every route itself, so routing is a single launch.
#include <cuda_bf16.h>

#include <cfloat>

#include "kernels.h"
#include "place.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTok = kRouterTokensTc;   // 128 tokens per CTA = MMA M
constexpr int kN = 64;                  // MMA N: experts, padded to 64
constexpr int kStages = 6;
constexpr int kABytes = kTok * kTcBK * 2;   // 16 KB
constexpr int kBBytes = kN * kTcBK * 2;     // 8 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kParts = 8;                   // partial accumulators
constexpr int kTmemCols = kParts * kN;      // 512
constexpr int kThreads = 128;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTok, kN);

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t done;
    uint32_t tmem;
    int abort;
    int hist[kMaxExperts];
    int off[kMaxExperts + 1];
    int cnt[4][kMaxExperts];
    int run[4][kMaxExperts];
};

constexpr int kLgBytes = kTok * (kMaxExperts + 1) * 4;
constexpr int kIdsBytes = kTok * kMaxTopK * 4;
constexpr int kSmemBytes = kStages * kStageBytes + kLgBytes + kIdsBytes + (int)sizeof(Ctl) + 1024;

__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const RouterTcArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float (*lg)[kMaxExperts + 1] = reinterpret_cast<float (*)[kMaxExperts + 1]>(smem + kStages * kStageBytes);
    int* sid = reinterpret_cast<int*>(smem + kStages * kStageBytes + kLgBytes);
    Ctl& c = *reinterpret_cast<Ctl*>(smem + kStages * kStageBytes + kLgBytes + kIdsBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t0 = blockIdx.x * kTok;
    const int E = a.E, k = a.k;
    const int kb_total = a.H / kTcBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&c.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&c.done), 1);
        c.abort = 0;
        ptx::fence_mbar_init();
    }
    if (threadIdx.x < kMaxExperts) c.hist[threadIdx.x] = 0;
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_u32(&c.tmem), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = c.tmem;

    if (warp == 0 && lane == 0) {
        // TMA producer
        int stage = 0;
        uint32_t phase = 0, last_par[kStages];
        int issued = 0;
        bool ok = true;
        for (int kb = 0; kb < kb_total; ++kb) {
            if (!ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, a.limit_ns, &c.abort)) {
                ok = false;
                break;
            }
            const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
            const uint32_t fb = ptx::smem_u32(&c.full[stage]);
            ptx::mbar_arrive_expect_tx(fb, kStageBytes);
            ptx::tma_load_2d(sa, &tmX, kb * kTcBK, t0, fb);
            ptx::tma_load_2d(sa + kABytes, &tmW, kb * kTcBK, 0, fb);
            last_par[stage] = phase;
            ++issued;
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) {
            c.abort = 1;
            atomicOr(a.err, kErrTimeout);
            const int n = issued < kStages ? issued : kStages;
            for (int s = 0; s < n; ++s) ptx::mbar_wait(ptx::smem_u32(&c.full[s]), last_par[s], a.limit_ns, nullptr);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: K-block kb goes to partial accumulator kb % 8
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int kb = 0; kb < kb_total; ++kb) {
            if (!ptx::mbar_wait(ptx::smem_u32(&c.full[stage]), phase, a.limit_ns, &c.abort)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
            const uint64_t adesc = ptx::sw128_desc(sa), bdesc = ptx::sw128_desc(sa + kABytes);
            const uint32_t d = tmem + (uint32_t)((kb % kParts) * kN);
#pragma unroll
            for (int kk = 0; kk < kTcBK / 16; ++kk)
                ptx::mma_bf16(d, adesc + 2u * kk, bdesc + 2u * kk, kIdesc, (kb >= kParts || kk > 0) ? 1u : 0u);
            ptx::mma_commit(ptx::smem_u32(&c.empty[stage]));
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) {
            c.abort = 1;
            atomicOr(a.err, kErrTimeout);
        }
        ptx::mma_commit(ptx::smem_u32(&c.done));
    }

    // every thread waits for the last MMA (lane 0 of each warp polls)
    bool ready = false;
    if (lane == 0)
        ready = ptx::mbar_wait(ptx::smem_u32(&c.done), 0, a.limit_ns, nullptr) &&
                *static_cast<volatile int*>(&c.abort) == 0;
    ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
    ptx::tc_fence_after();

    const int row = warp * 32 + lane;
    const int t = t0 + row;
    if (ready) {
        // combine the partials: logits of token `row`, experts 0..63
        const int nparts = kb_total < kParts ? kb_total : kParts;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int col = 0; col < kN; col += 16) {
            float sum[16], comp[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sum[i] = comp[i] = 0.f;
#pragma unroll 1
            for (int p = 0; p < nparts; ++p) {
                uint32_t v[16];
                ptx::tmem_ld16(lane_base + (uint32_t)(p * kN + col), v);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float y = __uint_as_float(v[i]) - comp[i];
                    const float s2 = sum[i] + y;
                    comp[i] = (s2 - sum[i]) - y;
                    sum[i] = s2;
                }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = col + i;
                float l = sum[i];
                if (a.bias != nullptr && e < E) l += a.bias[e];
                lg[row][e] = l;
                if (a.logits != nullptr && t < a.T && e < E) a.logits[(int64_t)t * E + e] = l;
            }
        }
        // top-k over this token's logits: larger logit first, ties to the lower index
        if (t < a.T) {
            uint64_t taken = 0;
            float v0 = 0.f, den = 0.f;
            float vals[kMaxTopK];
            int ids[kMaxTopK];
            for (int j = 0; j < k; ++j) {
                int best = -1;
                float bv = -INFINITY;
                for (int e = 0; e < E; ++e) {
                    if ((taken >> e) & 1ull) continue;
                    const float v = lg[row][e];
                    if (best < 0 || v > bv) {
                        best = e;
                        bv = v;
                    }
                }
                if (bv != bv) atomicOr(a.err, kErrCheck);  // NaN logit
                taken |= 1ull << best;
                ids[j] = best;
                vals[j] = bv;
            }
            v0 = vals[0];
            for (int j = 0; j < k; ++j) {
                vals[j] = expf(vals[j] - v0);
                den += vals[j];
            }
            for (int j = 0; j < k; ++j) {
                a.ids[(int64_t)t * k + j] = ids[j];
                a.w[(int64_t)t * k + j] = vals[j] / den;
                sid[row * k + j] = ids[j];
                atomicAdd(&c.hist[ids[j]], 1);
            }
        }
    }
    __syncthreads();

    const int n_tok = min(kTok, a.T - t0);
    if (gridDim.x == 1) {
        // single CTA: offsets, tile prefixes and the placement of every route
        if (threadIdx.x == 0) {
            int ttc = 0, tsi = 0;
            c.off[0] = 0;
            a.tiles_tc[0] = 0;
            a.tiles_simt[0] = 0;
            for (int e = 0; e < E; ++e) {
                c.off[e + 1] = c.off[e] + c.hist[e];
                ttc += (c.hist[e] + kTcBM - 1) / kTcBM;
                tsi += (c.hist[e] + kSimtBM - 1) / kSimtBM;
                a.tiles_tc[e + 1] = ttc;
                a.tiles_simt[e + 1] = tsi;
            }
            a.shared_seg[0] = 0;
            a.shared_seg[1] = a.T;
            a.shared_tiles_tc[0] = 0;
            a.shared_tiles_tc[1] = (a.T + kTcBM - 1) / kTcBM;
            a.shared_tiles_simt[0] = 0;
            a.shared_tiles_simt[1] = (a.T + kSimtBM - 1) / kSimtBM;
        }
        __syncthreads();
        if ((int)threadIdx.x <= E) a.offsets[threadIdx.x] = c.off[threadIdx.x];
        place_chunk<4>(sid, n_tok * k, 0, E, (int64_t)a.T * k, [&](int e) { return c.off[e]; }, c.cnt, c.run,
                       a.perm, a.inv, a.err);
    } else if ((int)threadIdx.x < E) {
        a.blk_hist[(int64_t)blockIdx.x * E + threadIdx.x] = c.hist[threadIdx.x];
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_router_tc(const RouterTcArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                             cudaStream_t s) {
    const int nb = (a.T + kTok - 1) / kTok;
    if (nb == 0) return cudaSuccess;
    static bool configured = false;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    router_tc_kernel<<<nb, kThreads, kSmemBytes, s>>>(tmX, tmW, a);
    return cudaGetLastError();
}

}  // namespace moe
