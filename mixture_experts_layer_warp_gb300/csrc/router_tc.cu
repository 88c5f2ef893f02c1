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
// token (its TMEM lane) and keeps its 64 logits in registers: softmax top-k,
// renormalised weights, and the CTA's expert histogram. When one CTA covers all tokens
// (T <= 128: decode-sized batches) it also computes the offsets and places
// every route itself, so routing is a single launch. Batches of at most 16
// tokens use an 8-CTA cluster that splits K (router_tc_cluster_kernel below).
#include <cuda_bf16.h>

#include <cfloat>

#include "kernels.h"
#include "place.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTok = kRouterTokensTc;   // 128 tokens per CTA = MMA M
constexpr int kN = 64;                  // MMA N: experts, padded to 64
constexpr int kStages = 6;  // even: a slot holds K-blocks of one parity (one MMA issuer)
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

constexpr int kIdsBytes = kTok * kMaxTopK * 4;
constexpr int kSmemBytes = kStages * kStageBytes + kIdsBytes + (int)sizeof(Ctl) + 1024;

// Kahan step: adds v into (sum, comp).
__device__ __forceinline__ void kahan_add(float& sum, float& comp, float v) {
    const float y = v - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
}

// Top-k of one token from its 64 fp32 logits held in registers (experts >= E
// are -inf): k rounds of a pairwise tournament, larger logit first and the
// lower index on equal logits; the chosen expert is then masked to -inf. Weights exp(l_j - l_0) / sum_j' exp(l_j' - l_0) are the
// softmax over all experts restricted to the k and renormalised. Writes the
// token's ids and weights, keeps the ids in shared memory (sid) and counts them
// in the CTA histogram.
__device__ __forceinline__ void select_topk(float (&l)[kN], int k, int64_t t, int row, const RouterTcArgs& a,
                                            int* sid, int* hist) {
    float vals[kMaxTopK];
    int ids[kMaxTopK];
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        // pairwise tournament: a right (higher-index) entry wins only when strictly
        // larger, and every left subtree holds lower indices, so ties go to the
        // lower expert index exactly as a scan with strict '>' would
        float v[kN / 2];
        int ix[kN / 2];
#pragma unroll
        for (int i = 0; i < kN / 2; ++i) {
            const bool r = l[2 * i + 1] > l[2 * i];
            v[i] = r ? l[2 * i + 1] : l[2 * i];
            ix[i] = r ? 2 * i + 1 : 2 * i;
        }
#pragma unroll
        for (int w = kN / 4; w >= 1; w >>= 1) {
#pragma unroll
            for (int i = 0; i < w; ++i) {
                const bool r = v[2 * i + 1] > v[2 * i];
                v[i] = r ? v[2 * i + 1] : v[2 * i];
                ix[i] = r ? ix[2 * i + 1] : ix[2 * i];
            }
        }
        const float bv = v[0];
        const int be = ix[0];
        if (bv != bv || be >= a.E) atomicOr(a.err, kErrCheck);  // NaN logits only
#pragma unroll
        for (int e = 0; e < kN; ++e) l[e] = (e == be) ? -INFINITY : l[e];
        ids[j] = be;
        vals[j] = bv;
    }
    const float v0 = vals[0];
    float den = 0.f;
    for (int j = 0; j < k; ++j) {
        vals[j] = expf(vals[j] - v0);
        den += vals[j];
    }
    for (int j = 0; j < k; ++j) {
        a.ids[t * k + j] = ids[j];
        a.w[t * k + j] = vals[j] / den;
        sid[row * k + j] = ids[j];
        atomicAdd(&hist[ids[j]], 1);
    }
}

// Adds the router bias, writes the optional logits output and masks experts >= E.
__device__ __forceinline__ void finish_logits(float (&l)[kN], int64_t t, const RouterTcArgs& a) {
#pragma unroll
    for (int e = 0; e < kN; ++e) {
        if (e < a.E) {
            if (a.bias != nullptr) l[e] += a.bias[e];
            if (a.logits != nullptr) a.logits[t * a.E + e] = l[e];
        } else {
            l[e] = -INFINITY;
        }
    }
}

// When one CTA holds every route: offsets, tile prefixes, the shared expert's
// segment, and the stable placement of all T*k routes.
template <int NW>
__device__ __forceinline__ void finish_single(const RouterTcArgs& a, const int* hist, int* off,
                                              int (*cnt)[kMaxExperts], int (*run)[kMaxExperts], const int* sid) {
    const int E = a.E;
    if (threadIdx.x < 32) {
        // warp-wide exclusive scans over the (up to 64) experts, two per lane
        const int lane = threadIdx.x;
        const int e0 = 2 * lane, e1 = 2 * lane + 1;
        const int c0 = e0 < E ? hist[e0] : 0, c1 = e1 < E ? hist[e1] : 0;
        int s_cnt = c0 + c1;
        int s_tc = (c0 + kTcBM - 1) / kTcBM + (c1 + kTcBM - 1) / kTcBM;
        int s_si = (c0 + kSimtBM - 1) / kSimtBM + (c1 + kSimtBM - 1) / kSimtBM;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int a0 = __shfl_up_sync(0xffffffffu, s_cnt, d);
            const int a1 = __shfl_up_sync(0xffffffffu, s_tc, d);
            const int a2 = __shfl_up_sync(0xffffffffu, s_si, d);
            if (lane >= d) {
                s_cnt += a0;
                s_tc += a1;
                s_si += a2;
            }
        }
        // inclusive sums up to e1; the value before e0 is the exclusive sum
        const int x_cnt = s_cnt - c0 - c1, x_tc = s_tc - (c0 + kTcBM - 1) / kTcBM - (c1 + kTcBM - 1) / kTcBM;
        const int x_si = s_si - (c0 + kSimtBM - 1) / kSimtBM - (c1 + kSimtBM - 1) / kSimtBM;
        if (e0 <= E) {
            off[e0] = x_cnt;
            a.tiles_tc[e0] = x_tc;
            a.tiles_simt[e0] = x_si;
        }
        if (e1 <= E) {
            off[e1] = x_cnt + c0;
            a.tiles_tc[e1] = x_tc + (c0 + kTcBM - 1) / kTcBM;
            a.tiles_simt[e1] = x_si + (c0 + kSimtBM - 1) / kSimtBM;
        }
        if (E == 64 && lane == 31) {
            off[64] = s_cnt;
            a.tiles_tc[64] = s_tc;
            a.tiles_simt[64] = s_si;
        }
        if (lane == 0) {
            a.shared_seg[0] = 0;
            a.shared_seg[1] = a.T;
            a.shared_tiles_tc[0] = 0;
            a.shared_tiles_tc[1] = (a.T + kTcBM - 1) / kTcBM;
            a.shared_tiles_simt[0] = 0;
            a.shared_tiles_simt[1] = (a.T + kSimtBM - 1) / kSimtBM;
        }
    }
    __syncthreads();
    if ((int)threadIdx.x <= E) a.offsets[threadIdx.x] = off[threadIdx.x];
    if (a.zero_counters != nullptr)
        for (int i = threadIdx.x; i < a.zero_count; i += blockDim.x) a.zero_counters[i] = 0;
    place_chunk<NW>(sid, a.T * a.k, 0, E, (int64_t)a.T * a.k, [&](int e) { return off[e]; }, cnt, run, a.perm,
                    a.inv, a.err);
}

__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const RouterTcArgs a) {
    // the next kernel (the fused GEMMs) may place its CTAs as SMs free up: it
    // only sets up its shared memory and TMEM before waiting for this grid
    ptx::griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* sid = reinterpret_cast<int*>(smem + kStages * kStageBytes);
    Ctl& c = *reinterpret_cast<Ctl*>(smem + kStages * kStageBytes + kIdsBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t0 = blockIdx.x * kTok;
    const int E = a.E, k = a.k;
    const int kb_total = a.H / kTcBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&c.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&c.done), 2);  // both MMA issuers' final commits
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
    // launched early (programmatic dependent launch): no global memory is
    // touched before the previous kernel in the stream has completed
    ptx::griddep_wait();
    const uint32_t tmem = c.tmem;

    if (warp == 0 && lane == 0) {
        // TMA producer
        const uint64_t wpol = ptx::policy_evict_last();  // the router matrix is read on every call
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
            ptx::tma_load_2d_hint(sa + kABytes, &tmW, kb * kTcBK, 0, fb, wpol);
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
    } else if ((warp == 1 || warp == 3) && lane == 0) {
        // MMA issuers: K-block kb goes to partial accumulator kb % 8, issued by
        // warp 1 for even kb and warp 3 for odd kb (one thread issues an MMA
        // about every 75 cycles; two halve the issue time). The partials and
        // the K-blocks summed into each are those of a single issuer, so the
        // logits are unchanged; with an even ring, slot s only ever holds
        // K-blocks of one parity, so each slot's barriers have one consumer.
        const int j = warp == 1 ? 0 : 1;
        int stage = j;
        uint32_t phase = 0;
        bool ok = true;
        for (int kb = j; kb < kb_total; kb += 2) {
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
            stage += 2;
            if (stage >= kStages) {
                stage -= kStages;
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
        // combine the partials of token `row` (its TMEM lane): four partials per
        // batched load, compensated addition in partial order 0..7
        const int nparts = kb_total < kParts ? kb_total : kParts;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float l[kN], comp[kN];
#pragma unroll
        for (int e = 0; e < kN; ++e) l[e] = comp[e] = 0.f;
#pragma unroll 1
        for (int p0 = 0; p0 < nparts; p0 += 4) {
#pragma unroll
            for (int col = 0; col < kN; col += 16) {
                uint32_t v[64];
                const uint32_t base = lane_base + (uint32_t)col;
                ptx::tmem_ld16x4(base + (uint32_t)(p0 * kN), base + (uint32_t)(min(p0 + 1, nparts - 1) * kN),
                                 base + (uint32_t)(min(p0 + 2, nparts - 1) * kN),
                                 base + (uint32_t)(min(p0 + 3, nparts - 1) * kN), v);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (p0 + q < nparts) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            kahan_add(l[col + i], comp[col + i], __uint_as_float(v[q * 16 + i]));
                    }
            }
        }
        if (t < a.T) {
            finish_logits(l, t, a);
            select_topk(l, k, t, row, a, sid, c.hist);
        }
    }
    __syncthreads();

    if (gridDim.x == 1) {
        finish_single<4>(a, c.hist, c.off, c.cnt, c.run, sid);
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


// ------------------------------------------------------------------------
// Batches of at most kSmallTokens tokens: a cluster of 8 CTAs splits K. CTA c
// accumulates exactly the K-blocks kb = c, c+8, c+16, ... that form partial c
// of router_tc_kernel, in the same order, sends its partial logits to CTA 0
// with st.async (completing bytes on CTA 0's exchange barrier), and CTA 0
// combines the partials in the same compensated order. The logits are
// therefore bit-identical to the 128-token kernel's (routing does not depend
// on the batch size), while eight SMs instead of one stream the router weights.
//
// Only 16 of the 128 A rows carry tokens, so the stages are packed 10 KB apart
// (2 KB of x, then 8 KB of Wr): the MMA's rows 16..127 read whatever follows
// (the next stage or the pad) and land in TMEM lanes nobody reads. With eight
// stages, every K-block of a 4096-wide hidden state is in flight at once.
constexpr int kCluster = kRouterClusterCtas;
constexpr int kCStages = 8;
constexpr int kCTok = kSmallTokens;
constexpr int kXBytesSmall = kCTok * kTcBK * 2;                    // 2 KB of x per stage
constexpr int kCStageBytes = kXBytesSmall + kBBytes;               // 10 KB, a multiple of 1024
constexpr int kCRingBytes = kCStages * kCStageBytes + (kABytes - kCStageBytes);  // + pad: last stage's rows 16..127
constexpr int kPartBytes = kCluster * kCTok * kN * 4;              // 32 KB
constexpr int kCIdsBytes = kCTok * kMaxTopK * 4;
constexpr int kGroup = kThreads / kCTok;                           // 8 threads per token in the top-k
constexpr int kPerThread = kN / kGroup;                            // 8 experts per thread
static_assert(kCStageBytes % 1024 == 0, "128B-swizzled tiles need 1024-byte aligned stages");
static_assert(kGroup == 8 && kPerThread == 8, "top-k layout assumes 16 tokens x 8 threads x 8 experts");

struct CCtl {
    uint64_t full[kCStages];
    uint64_t empty[kCStages];
    uint64_t done;
    uint64_t xfer;   // CTA 0: completes when every other CTA's partial has arrived
    uint32_t tmem;
    int abort;
    int hist[kMaxExperts];
    int off[kMaxExperts + 1];
    int cnt[4][kMaxExperts];
    int run[4][kMaxExperts];
};
constexpr int kCSmemBytes = kCRingBytes + kPartBytes + kCIdsBytes + (int)sizeof(CCtl) + 1024;

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    router_tc_cluster_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                             const RouterTcArgs a) {
    // the next kernel (the fused GEMMs) may place its CTAs as SMs free up: it
    // only sets up its shared memory and TMEM before waiting for this grid
    ptx::griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* part = reinterpret_cast<float*>(smem + kCRingBytes);   // [kCluster][kCTok][kN] on CTA 0
    int* sid = reinterpret_cast<int*>(smem + kCRingBytes + kPartBytes);
    CCtl& c = *reinterpret_cast<CCtl*>(smem + kCRingBytes + kPartBytes + kCIdsBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = (int)ptx::cluster_ctarank();
    const int k = a.k;
    const int kb_total = a.H / kTcBK;
    const int my_blocks = kb_total > rank ? (kb_total - rank + kCluster - 1) / kCluster : 0;
    const int nparts = kb_total < kCluster ? kb_total : kCluster;
    const uint32_t xfer = ptx::smem_u32(&c.xfer);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kCStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&c.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&c.done), 1);
        ptx::mbar_init(xfer, 1);
        // CTA 0 announces the bytes the other CTAs will send before any can
        // start (they first pass the cluster barrier that follows the init)
        if (rank == 0) ptx::mbar_arrive_expect_tx(xfer, (uint32_t)((nparts - 1) * a.T * kN * 4));
        c.abort = 0;
        ptx::fence_mbar_init();
    }
    if (threadIdx.x < kMaxExperts) c.hist[threadIdx.x] = 0;
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_u32(&c.tmem), kN);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_arrive();   // first phase: barrier inits visible cluster-wide
    // launched early (programmatic dependent launch): no global memory is
    // touched before the previous kernel in the stream has completed
    ptx::griddep_wait();
    const uint32_t tmem = c.tmem;

    if (warp == 0 && lane == 0) {
        const uint64_t wpol = ptx::policy_evict_last();  // the router matrix is read on every call
        int stage = 0;
        uint32_t phase = 0, last_par[kCStages];
        int issued = 0;
        bool ok = true;
        for (int i = 0; i < my_blocks; ++i) {
            const int kb = rank + i * kCluster;
            if (!ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, a.limit_ns, &c.abort)) {
                ok = false;
                break;
            }
            const uint32_t sa = ptx::smem_u32(smem + stage * kCStageBytes);
            const uint32_t fb = ptx::smem_u32(&c.full[stage]);
            ptx::mbar_arrive_expect_tx(fb, kXBytesSmall + kBBytes);
            ptx::tma_load_2d(sa, &tmX, kb * kTcBK, 0, fb);  // 16 token rows
            ptx::tma_load_2d_hint(sa + kXBytesSmall, &tmW, kb * kTcBK, 0, fb, wpol);
            last_par[stage] = phase;
            ++issued;
            if (++stage == kCStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) {
            c.abort = 1;
            atomicOr(a.err, kErrTimeout);
            const int n = issued < kCStages ? issued : kCStages;
            for (int s = 0; s < n; ++s) ptx::mbar_wait(ptx::smem_u32(&c.full[s]), last_par[s], a.limit_ns, nullptr);
        }
    } else if (warp == 1 && lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int i = 0; i < my_blocks; ++i) {
            if (!ptx::mbar_wait(ptx::smem_u32(&c.full[stage]), phase, a.limit_ns, &c.abort)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = ptx::smem_u32(smem + stage * kCStageBytes);
            const uint64_t adesc = ptx::sw128_desc(sa), bdesc = ptx::sw128_desc(sa + kXBytesSmall);
#pragma unroll
            for (int kk = 0; kk < kTcBK / 16; ++kk)
                ptx::mma_bf16(tmem, adesc + 2u * kk, bdesc + 2u * kk, kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(ptx::smem_u32(&c.empty[stage]));
            if (++stage == kCStages) {
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

    bool ready = false;
    if (lane == 0)
        ready = ptx::mbar_wait(ptx::smem_u32(&c.done), 0, a.limit_ns, nullptr) &&
                *static_cast<volatile int*>(&c.abort) == 0;
    ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
    ptx::tc_fence_after();
    ptx::cluster_wait();
    const int row = warp * 32 + lane;
    if (ready && my_blocks > 0 && warp == 0) {  // rows 0..15 live in warp 0's lanes
        uint32_t v[kN];
        ptx::tmem_ld16x4(tmem, tmem + 16u, tmem + 32u, tmem + 48u, v);
        if (row < a.T) {
            float* mine = part + ((size_t)rank * kCTok + row) * kN;
            if (rank == 0) {
#pragma unroll
                for (int q = 0; q < kN / 4; ++q)
                    reinterpret_cast<float4*>(mine)[q] = make_float4(
                        __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                        __uint_as_float(v[4 * q + 3]));
            } else {
                const uint32_t dst = ptx::map_to_rank(ptx::smem_u32(mine), 0);
                const uint32_t bar = ptx::map_to_rank(xfer, 0);
#pragma unroll
                for (int q = 0; q < kN / 4; ++q)
                    ptx::st_async_v4(dst + 16u * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], bar);
            }
        }
    }

    if (rank == 0) {
        // the other partials: bounded wait on the exchange barrier (also when
        // this CTA failed, so that no write lands after it has exited)
        bool got = true;
        if (threadIdx.x == 0) {
            got = ptx::mbar_wait_cluster(xfer, 0, a.limit_ns);
            if (!got || !ready) atomicOr(a.err, kErrTimeout);
        }
        const bool go = __syncthreads_and(got && ready) != 0;
        ptx::cluster_arrive_relaxed();   // second phase: CTA 0 has received everything
        if (go) {
            // thread (token r, lane-group position g) owns experts 8g..8g+7
            const int r = threadIdx.x / kGroup, g = threadIdx.x % kGroup;
            const unsigned gmask = 0xffu << (lane & ~(kGroup - 1));
            if (r < a.T) {
                float l[kPerThread];
                {
                    float sum[kPerThread], comp[kPerThread];
#pragma unroll
                    for (int i = 0; i < kPerThread; ++i) sum[i] = comp[i] = 0.f;
                    for (int p = 0; p < nparts; ++p) {  // partials in order 0..7, as router_tc_kernel
                        const float4* src =
                            reinterpret_cast<const float4*>(part + ((size_t)p * kCTok + r) * kN + g * kPerThread);
                        const float4 v0 = src[0], v1 = src[1];
                        kahan_add(sum[0], comp[0], v0.x);
                        kahan_add(sum[1], comp[1], v0.y);
                        kahan_add(sum[2], comp[2], v0.z);
                        kahan_add(sum[3], comp[3], v0.w);
                        kahan_add(sum[4], comp[4], v1.x);
                        kahan_add(sum[5], comp[5], v1.y);
                        kahan_add(sum[6], comp[6], v1.z);
                        kahan_add(sum[7], comp[7], v1.w);
                    }
#pragma unroll
                    for (int i = 0; i < kPerThread; ++i) {
                        const int e = g * kPerThread + i;
                        l[i] = sum[i];
                        if (e < a.E) {
                            if (a.bias != nullptr) l[i] += a.bias[e];
                            if (a.logits != nullptr) a.logits[(int64_t)r * a.E + e] = l[i];
                        } else {
                            l[i] = -INFINITY;
                        }
                    }
                }
                // k rounds: the group's maximum logit, lower expert index on
                // equal logits (the rule of select_topk), then masked out.
                // Weights exp(l_j - l_0) / sum_j' exp(l_j' - l_0), summed in
                // round order exactly as select_topk does.
                float v0 = 0.f, den = 0.f, w_lo = 0.f, w_hi = 0.f;
                int id_lo = 0, id_hi = 0;
#pragma unroll 1
                for (int j = 0; j < k; ++j) {
                    float bv = l[0];
                    int bi = 0;
#pragma unroll
                    for (int i = 1; i < kPerThread; ++i)
                        if (l[i] > bv) {
                            bv = l[i];
                            bi = i;
                        }
                    bi += g * kPerThread;
#pragma unroll
                    for (int d = 1; d < kGroup; d <<= 1) {
                        const float ov = __shfl_xor_sync(gmask, bv, d);
                        const int oi = __shfl_xor_sync(gmask, bi, d);
                        if (ov > bv || (ov == bv && oi < bi)) {
                            bv = ov;
                            bi = oi;
                        }
                    }
                    if (g == 0 && (bv != bv || bi >= a.E)) atomicOr(a.err, kErrCheck);  // NaN logits only
#pragma unroll
                    for (int i = 0; i < kPerThread; ++i)
                        if (g * kPerThread + i == bi) l[i] = -INFINITY;
                    if (j == 0) v0 = bv;
                    const float ej = expf(bv - v0);
                    den += ej;
                    if (j == g) {
                        w_lo = ej;
                        id_lo = bi;
                    } else if (j == g + kGroup) {
                        w_hi = ej;
                        id_hi = bi;
                    }
                }
                if (g < k) {
                    a.ids[(int64_t)r * k + g] = id_lo;
                    a.w[(int64_t)r * k + g] = w_lo / den;
                    sid[r * k + g] = id_lo;
                    atomicAdd(&c.hist[id_lo], 1);
                }
                if (g + kGroup < k) {
                    a.ids[(int64_t)r * k + g + kGroup] = id_hi;
                    a.w[(int64_t)r * k + g + kGroup] = w_hi / den;
                    sid[r * k + g + kGroup] = id_hi;
                    atomicAdd(&c.hist[id_hi], 1);
                }
            }
            __syncthreads();
            finish_single<4>(a, c.hist, c.off, c.cnt, c.run, sid);
        }
    } else {
        ptx::cluster_arrive_relaxed();   // second phase: this CTA's partial is on its way
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kN);
    }
    ptx::cluster_wait();   // no CTA leaves before CTA 0 holds every partial
}

// ------------------------------------------------------------------------
// Mid-size batches (a few thousand tokens): a cluster of kSplit = 4 CTAs per
// 128-token block splits K, so the batch fills the GPU instead of one SM per
// 128 tokens. CTA r accumulates exactly the K-blocks of partials 2r and 2r+1 of
// router_tc_kernel (kb = 8i + 2r and 8i + 2r + 1), in the same order, into two
// TMEM accumulators. Then every CTA sends each 32-token slice of its two
// partials to the CTA that owns the slice (st.async completing bytes on the
// owner's exchange barrier), and CTA r combines the eight partials of tokens
// 32r .. 32r+31 in the same compensated order as router_tc_kernel: the logits
// are bit-identical to the other kernels'. Eight threads per token (256 per
// CTA; warps 4-7 wait out the loads) select the top-k. The four CTAs add their expert counts into CTA 0 (shared-memory
// reductions across the cluster), which writes the 128-token block's histogram
// row, as router_tc_kernel does.
constexpr int kSplit = 4;
constexpr int kSplitTok = kTok / kSplit;              // 32 tokens combined per CTA
constexpr int kSPartsPer = kParts / kSplit;           // 2 partials accumulated per CTA
constexpr int kSStages = 6;
constexpr int kSRecvBytes = kParts * kSplitTok * kN * 4;   // [partial][token][expert] fp32: 64 KB
constexpr int kSSendBytes = kSPartsPer * kSplitTok * kN * 4;  // one CTA's contribution to a slice: 16 KB
constexpr int kSThreads = 256;                        // warps 4-7 join for the combine and the top-k
constexpr int kSGroup = kSThreads / kSplitTok;        // 8 threads per token in the top-k
constexpr int kSPer = kN / kSGroup;                   // 8 experts per thread
static_assert(kSplitTok == 32 && kSGroup == 8, "32 tokens combined per CTA, 8 threads each");
static_assert(kSplit * kSSendBytes <= kSStages * kStageBytes, "send slices staged in the load ring");

// The float4 slot of logits 4q .. 4q+3 within row `row` of a received slice:
// XOR-swizzled by the row, so that the 32 rows written one per lane and the
// 8 float4 of a token read by its 8 threads fall in distinct banks.
__device__ __forceinline__ int recv_q(int q, int row) { return q ^ (row & 15); }

struct SCtl {
    uint64_t full[kSStages];
    uint64_t empty[kSStages];
    uint64_t done;
    uint64_t xfer;  // completes when the other CTAs' slices of this CTA's tokens have arrived
    uint32_t tmem;
    int abort;
    int hist[kMaxExperts];
    int hist_all[kMaxExperts];  // CTA 0: the four CTAs' counts
};
constexpr int kSSmemBytes = kSStages * kStageBytes + kSRecvBytes + (int)sizeof(SCtl) + 1024;

__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kSThreads, 1)
    router_tc_split_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                           const RouterTcArgs a) {
    ptx::griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* recv = reinterpret_cast<float*>(smem + kSStages * kStageBytes);
    SCtl& c = *reinterpret_cast<SCtl*>(smem + kSStages * kStageBytes + kSRecvBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = (int)ptx::cluster_ctarank();
    const int blk = blockIdx.x / kSplit;
    const int t0 = blk * kTok;
    const int E = a.E, k = a.k;
    const int kb_total = a.H / kTcBK;
    const int nparts = kb_total < kParts ? kb_total : kParts;
    // this CTA's K-blocks, in increasing kb: q -> 8 (q / 2) + 2 rank + q % 2
    int my_blocks = 0;
    for (int kb0 = 2 * rank; kb0 < kb_total; kb0 += kParts) my_blocks += (kb0 + 1 < kb_total) ? 2 : 1;
    const uint32_t xfer = ptx::smem_u32(&c.xfer);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&c.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&c.done), 1);
        ptx::mbar_init(xfer, 1);
        // the bytes the other three CTAs will send, announced before any can
        // start (they first pass the cluster barrier that follows the init)
        ptx::mbar_arrive_expect_tx(xfer, (uint32_t)((kSplit - 1) * kSSendBytes));
        c.abort = 0;
        ptx::fence_mbar_init();
    }
    if (threadIdx.x < kMaxExperts) c.hist[threadIdx.x] = c.hist_all[threadIdx.x] = 0;
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_u32(&c.tmem), kSPartsPer * kN);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_arrive();   // first phase: barrier inits visible cluster-wide
    // launched early (programmatic dependent launch): no global memory is
    // touched before the previous kernel in the stream has completed
    ptx::griddep_wait();
    const uint32_t tmem = c.tmem;

    if (warp == 0) {
        // TMA producer (whole warp; one elected lane issues)
        const bool issuer = ptx::elect_one();
        const uint64_t wpol = ptx::policy_evict_last();  // the router matrix is read on every call
        int stage = 0;
        uint32_t phase = 0, last_par[kSStages];
        int issued = 0;
        bool ok = true;
        for (int q = 0; q < my_blocks; ++q) {
            const int kb = kParts * (q / 2) + 2 * rank + (q & 1);
            const bool got = ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, a.limit_ns, &c.abort);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
            const uint32_t fb = ptx::smem_u32(&c.full[stage]);
            if (issuer) {
                ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                ptx::tma_load_2d(sa, &tmX, kb * kTcBK, t0, fb);
                ptx::tma_load_2d_hint(sa + kABytes, &tmW, kb * kTcBK, 0, fb, wpol);
            }
            __syncwarp();
            last_par[stage] = phase;
            ++issued;
            if (++stage == kSStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok && issuer) {
            c.abort = 1;
            atomicOr(a.err, kErrTimeout);
            const int n = issued < kSStages ? issued : kSStages;
            for (int s = 0; s < n; ++s) ptx::mbar_wait(ptx::smem_u32(&c.full[s]), last_par[s], a.limit_ns, nullptr);
        }
    } else if (warp == 1) {
        // MMA issuer (whole warp; one elected lane issues): K-block q goes to
        // accumulator q % 2 (partial 2 rank + q % 2)
        const bool issuer = ptx::elect_one();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int q = 0; q < my_blocks; ++q) {
            const bool got = ptx::mbar_wait(ptx::smem_u32(&c.full[stage]), phase, a.limit_ns, &c.abort);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
            const uint64_t adesc = ptx::sw128_desc(sa), bdesc = ptx::sw128_desc(sa + kABytes);
            const uint32_t d = tmem + (uint32_t)((q & 1) * kN);
            if (issuer) {
#pragma unroll
                for (int kk = 0; kk < kTcBK / 16; ++kk)
                    ptx::mma_bf16(d, adesc + 2u * kk, bdesc + 2u * kk, kIdesc, (q >= 2 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(ptx::smem_u32(&c.empty[stage]));
            }
            __syncwarp();
            if (++stage == kSStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (issuer) {
            if (!ok) {
                c.abort = 1;
                atomicOr(a.err, kErrTimeout);
            }
            ptx::mma_commit(ptx::smem_u32(&c.done));
        }
        __syncwarp();
    }

    bool ready = false;
    if (lane == 0)
        ready = ptx::mbar_wait(ptx::smem_u32(&c.done), 0, a.limit_ns, nullptr) &&
                *static_cast<volatile int*>(&c.abort) == 0;
    ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
    ptx::tc_fence_after();
    ptx::cluster_wait();   // every CTA's exchange barrier is armed before anyone sends

    // warp w < 4 holds TMEM lanes 32w.. = the tokens CTA w combines: send both
    // partials of each of them there (partial slot 2 rank + j of its buffer).
    // Every CTA sends, also one without K-blocks (H < 512): the owner expects
    // the bytes and skips the partials that do not exist. A slice for another
    // CTA is written in the owner's layout into the (now idle) load ring and
    // goes over in one bulk copy.
    if (warp >= 4) {
    } else if (ready) {
        const int dst_cta = warp;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float* slice = dst_cta == rank ? recv + (size_t)kSPartsPer * rank * kSplitTok * kN
                                       : reinterpret_cast<float*>(smem) + (size_t)warp * (kSSendBytes / 4);
#pragma unroll
        for (int j = 0; j < kSPartsPer; ++j) {
            uint32_t v[kN];
            const uint32_t b = lane_base + (uint32_t)(j * kN);
            ptx::tmem_ld16x4(b, b + 16u, b + 32u, b + 48u, v);
            float4* row = reinterpret_cast<float4*>(slice + ((size_t)j * kSplitTok + lane) * kN);
#pragma unroll
            for (int q = 0; q < kN / 4; ++q)
                row[recv_q(q, lane)] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
        if (dst_cta != rank) {
            ptx::fence_proxy_async_smem();  // the slice, visible to the bulk copy
            __syncwarp();
            if (lane == 0)
                ptx::bulk_copy_s2c(ptx::map_to_rank(ptx::smem_u32(recv + (size_t)kSPartsPer * rank * kSplitTok * kN),
                                                    (uint32_t)dst_cta),
                                   ptx::smem_u32(slice), (uint32_t)kSSendBytes,
                                   ptx::map_to_rank(xfer, (uint32_t)dst_cta));
        }
    } else if (lane == 0) {
        atomicOr(a.err, kErrTimeout);
    }
    __syncthreads();  // this CTA's own slice is in shared memory

    // the other CTAs' slices: bounded wait on the exchange barrier (also when
    // this CTA failed, so that no write lands after it has exited)
    bool got = true;
    if (threadIdx.x == 0) {
        got = ptx::mbar_wait_cluster(xfer, 0, a.limit_ns);
        if (!got) atomicOr(a.err, kErrTimeout);
    }
    const bool go = __syncthreads_and(got && ready) != 0;

    const int r = threadIdx.x / kSGroup, g = threadIdx.x % kSGroup;
    const int64_t t = (int64_t)t0 + kSplitTok * rank + r;
    if (go && t < a.T) {
        // thread (token r, group position g) owns experts 16g .. 16g+15
        const unsigned gmask = ((1u << kSGroup) - 1u) << (lane & ~(kSGroup - 1));
        float l[kSPer];
        {
            float sum[kSPer], comp[kSPer];
#pragma unroll
            for (int i = 0; i < kSPer; ++i) sum[i] = comp[i] = 0.f;
#pragma unroll
            for (int p = 0; p < kParts; ++p) {  // partials in order 0..7, as router_tc_kernel
                if (p >= nparts) break;
                const float4* src = reinterpret_cast<const float4*>(recv + ((size_t)p * kSplitTok + r) * kN);
#pragma unroll
                for (int q = 0; q < kSPer / 4; ++q) {
                    const float4 v = src[recv_q(g * (kSPer / 4) + q, r)];
                    kahan_add(sum[4 * q], comp[4 * q], v.x);
                    kahan_add(sum[4 * q + 1], comp[4 * q + 1], v.y);
                    kahan_add(sum[4 * q + 2], comp[4 * q + 2], v.z);
                    kahan_add(sum[4 * q + 3], comp[4 * q + 3], v.w);
                }
            }
#pragma unroll
            for (int i = 0; i < kSPer; ++i) {
                const int e = g * kSPer + i;
                l[i] = sum[i];
                if (e < E) {
                    if (a.bias != nullptr) l[i] += a.bias[e];
                    if (a.logits != nullptr) a.logits[t * E + e] = l[i];
                } else {
                    l[i] = -INFINITY;
                }
            }
        }
        // k rounds: the group's maximum logit, lower expert index on equal
        // logits (the rule of select_topk), then masked out; weights summed in
        // round order as select_topk does. Thread g keeps slots g, g+4, g+8, g+12.
        float v0 = 0.f, den = 0.f, wk[kMaxTopK / kSGroup];
        int idk[kMaxTopK / kSGroup];
#pragma unroll
        for (int u = 0; u < kMaxTopK / kSGroup; ++u) {
            wk[u] = 0.f;
            idk[u] = 0;
        }
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
            float bv = l[0];
            int bi = 0;
#pragma unroll
            for (int i = 1; i < kSPer; ++i)
                if (l[i] > bv) {
                    bv = l[i];
                    bi = i;
                }
            bi += g * kSPer;
#pragma unroll
            for (int d = 1; d < kSGroup; d <<= 1) {
                const float ov = __shfl_xor_sync(gmask, bv, d);
                const int oi = __shfl_xor_sync(gmask, bi, d);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (g == 0 && (bv != bv || bi >= E)) atomicOr(a.err, kErrCheck);  // NaN logits only
#pragma unroll
            for (int i = 0; i < kSPer; ++i)
                if (g * kSPer + i == bi) l[i] = -INFINITY;
            if (j == 0) v0 = bv;
            const float ej = expf(bv - v0);
            den += ej;
#pragma unroll
            for (int u = 0; u < kMaxTopK / kSGroup; ++u)
                if (j == g + kSGroup * u) {
                    wk[u] = ej;
                    idk[u] = bi;
                }
        }
#pragma unroll
        for (int u = 0; u < kMaxTopK / kSGroup; ++u) {
            const int slot = g + kSGroup * u;
            if (slot < k) {
                a.ids[t * k + slot] = idk[u];
                a.w[t * k + slot] = wk[u] / den;
                atomicAdd(&c.hist[idk[u]], 1);
            }
        }
    }
    __syncthreads();
    // this CTA's counts into CTA 0's; the second cluster phase orders them
    // before CTA 0 reads the sum (and keeps every CTA alive until all hold their slices)
    if ((int)threadIdx.x < E && c.hist[threadIdx.x] != 0)
        ptx::red_add_cluster(ptx::map_to_rank(ptx::smem_u32(&c.hist_all[threadIdx.x]), 0),
                             (uint32_t)c.hist[threadIdx.x]);
    ptx::tc_fence_before();
    ptx::cluster_arrive();
    ptx::cluster_wait();
    if (rank == 0 && (int)threadIdx.x < E) a.blk_hist[(int64_t)blk * E + threadIdx.x] = c.hist_all[threadIdx.x];
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kSPartsPer * kN);
    }
}

// Launch with programmatic stream serialization: the CTAs may be placed while
// the previous kernel in the stream finishes (its CTAs free SMs); each kernel
// here waits for it (griddep_wait) after its shared-memory and TMEM set-up.
template <typename K>
cudaError_t launch_early(K kernel, dim3 grid, int smem, cudaStream_t s, const CUtensorMap& tmX,
                         const CUtensorMap& tmW, const RouterTcArgs& a, int threads = kThreads) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tmX, tmW, a);
}

}  // namespace

cudaError_t launch_router_tc(const RouterTcArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                             cudaStream_t s) {
    const int nb = (a.T + kTok - 1) / kTok;
    if (nb == 0) return cudaSuccess;
    if (cudaError_t e = ensure_smem_limit<router_tc_kernel>(kSmemBytes); e != cudaSuccess) return e;
    return launch_early(router_tc_kernel, dim3(nb), kSmemBytes, s, tmX, tmW, a);
}

cudaError_t launch_router_tc_split(const RouterTcArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                                   cudaStream_t s) {
    const int nb = (a.T + kTok - 1) / kTok;
    if (nb == 0) return cudaSuccess;
    if (cudaError_t e = ensure_smem_limit<router_tc_split_kernel>(kSSmemBytes); e != cudaSuccess) return e;
    return launch_early(router_tc_split_kernel, dim3(nb * kSplit), kSSmemBytes, s, tmX, tmW, a, kSThreads);
}

cudaError_t launch_router_tc_small(const RouterTcArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                                   cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    if (a.T > kCTok) return cudaErrorInvalidValue;
    if (cudaError_t e = ensure_smem_limit<router_tc_cluster_kernel>(kCSmemBytes); e != cudaSuccess) return e;
    return launch_early(router_tc_cluster_kernel, dim3(kCluster), kCSmemBytes, s, tmX, tmW, a);
}

}  // namespace moe
