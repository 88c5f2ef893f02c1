// permute.cu - expert offsets, the stable route permutation and the gather.
//
// "HunyuanImage3 Hybrid Parallelism", section 6.1: the flattened expert ids
// are sorted by expert into permuted_to_expanded, bincount(...).cumsum(...)
// gives the expert offsets, and the input is index_select-ed once by the
// permutation; section 6.2 lists the permutation inverse. Here the sort is a
// deterministic counting sort without atomics on the output order:
//   router block b owns routes [b*n*k, (b+1)*n*k) (n tokens per router block)
//   and wrote its histogram row;
//   scan:  offsets[e] = sum of all counts of experts < e, and
//          base[b][e] = offsets[e] + counts of expert e in blocks < b;
//   place: block b walks its routes in order and gives the i-th route of
//          expert e the position base[b][e] + i (warp rounds, place.cuh).
// So within an expert the routes keep ascending r = t*k + j (a stable sort).
#include <algorithm>

#include "kernels.h"
#include "place.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
    __shared__ int part[kScanThreads];   // [parts][E]
    __shared__ int off[kMaxExperts + 1];
    ptx::griddep_wait();  // launched early: the router's histograms are complete past here
    const int E = a.E, NB = a.NB;
    const int parts = kScanThreads / E;
    const int tid = threadIdx.x;
    const int e = tid % E, p = tid / E;
    const bool active = p < parts;
    const int b0 = active ? (int)((int64_t)p * NB / parts) : 0;
    const int b1 = active ? (int)((int64_t)(p + 1) * NB / parts) : 0;

    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += a.blk_hist[(int64_t)b * E + e];
    if (active) part[p * E + e] = sum;
    __syncthreads();
    if (tid < E) {  // exclusive prefix over parts, per expert
        int run = 0;
        for (int q = 0; q < parts; ++q) {
            const int c = part[q * E + tid];
            part[q * E + tid] = run;
            run += c;
        }
        off[tid + 1] = run;  // total count of expert tid, turned into offsets below
    }
    __syncthreads();
    if (tid == 0) {
        off[0] = 0;
        for (int i = 0; i < E; ++i) off[i + 1] += off[i];
        int ttc = 0, tsi = 0;
        a.tiles_tc[0] = 0;
        a.tiles_simt[0] = 0;
        for (int i = 0; i < E; ++i) {
            const int c = off[i + 1] - off[i];
            ttc += (c + kTcBM - 1) / kTcBM;
            tsi += (c + kSimtBM - 1) / kSimtBM;
            a.tiles_tc[i + 1] = ttc;
            a.tiles_simt[i + 1] = tsi;
        }
        for (int i = 0; i <= E; ++i) a.offsets[i] = off[i];
        a.shared_seg[0] = 0;
        a.shared_seg[1] = a.T;
        a.shared_tiles_tc[0] = 0;
        a.shared_tiles_tc[1] = (a.T + kTcBM - 1) / kTcBM;
        a.shared_tiles_simt[0] = 0;
        a.shared_tiles_simt[1] = (a.T + kSimtBM - 1) / kSimtBM;
    }
    __syncthreads();
    if (active) {
        int run = off[e] + part[p * E + e];
        for (int b = b0; b < b1; ++b) {
            a.blk_base[(int64_t)b * E + e] = run;
            run += a.blk_hist[(int64_t)b * E + e];
        }
    }
    // the next kernel is placed once every CTA got here (a trigger at the start
    // let the next kernels' waiting CTAs crowd this one and measured slower)
    ptx::griddep_launch_dependents();
}

constexpr int kPlaceWarps = 8;

__global__ void __launch_bounds__(kPlaceWarps * 32) place_kernel(PlaceArgs a) {
    __shared__ int sid[kRouterTokensTc * kMaxTopK];
    __shared__ int cnt[kPlaceWarps][kMaxExperts];
    __shared__ int run[kPlaceWarps][kMaxExperts];
    ptx::griddep_wait();  // launched early: the scan's bases are complete past here
    const int64_t R = (int64_t)a.T * a.k;
    const int64_t r0 = (int64_t)blockIdx.x * a.tok_per_blk * a.k;
    const int64_t left = R - r0;
    const int n = (int)(left < (int64_t)a.tok_per_blk * a.k ? left : (int64_t)a.tok_per_blk * a.k);
    for (int i = threadIdx.x; i < n; i += blockDim.x) sid[i] = a.ids[r0 + i];
    __syncthreads();
    const int32_t* base = a.blk_base + (int64_t)blockIdx.x * a.E;
    place_chunk<kPlaceWarps>(sid, n, r0, a.E, R, [&](int e) { return base[e]; }, cnt, run, a.perm, a.inv, a.err);
    ptx::griddep_launch_dependents();
}

// Scan and placement in one launch, for batches whose block histograms are
// small enough for every block to read them all (NB * E <= kScanPlaceMaxInts):
// block b sums every histogram row itself, which gives offsets[e] (all routes
// of experts < e) and its own base[b][e] = offsets[e] + (routes of expert e in
// blocks < b) without a separate pass; block 0 also writes the offsets, the
// tile prefixes and the shared expert's segment. The placement is the same
// stable warp-round placement as place_kernel.
// 8 warps (32 measured slower: the per-expert scans and sums then take longer
// than the rounds they save).
constexpr int kSPWarps = 8;
constexpr int kSumParts = kSPWarps * 32 / kMaxExperts;  // 4 threads per expert sum the rows
constexpr int kSPIds = kRouterTokensTc * kMaxTopK / (kSPWarps * 32);  // ids per thread

__global__ void __launch_bounds__(kSPWarps * 32) scan_place_kernel(ScanArgs sa, PlaceArgs a) {
    __shared__ int sid[kRouterTokensTc * kMaxTopK];
    __shared__ int cnt[kSPWarps][kMaxExperts];
    __shared__ int run[kSPWarps][kMaxExperts];
    __shared__ int tot_part[kSumParts][kMaxExperts];
    __shared__ int bef_part[kSumParts][kMaxExperts];
    __shared__ int off[kMaxExperts + 1];
    __shared__ int base[kMaxExperts];
    ptx::griddep_wait();  // launched early: the router's ids and histograms are complete past here
    const int E = a.E, NB = a.NB, b = blockIdx.x, tid = threadIdx.x;
    const int64_t R = (int64_t)a.T * a.k;
    const int64_t r0 = (int64_t)b * a.tok_per_blk * a.k;
    const int64_t left = R - r0;
    const int n = (int)(left < (int64_t)a.tok_per_blk * a.k ? left : (int64_t)a.tok_per_blk * a.k);
    {
        // the block's ids and the histogram rows, all loads in flight together
        int ids[kSPIds];
#pragma unroll
        for (int u = 0; u < kSPIds; ++u) {
            const int i = tid + u * kSPWarps * 32;
            ids[u] = i < n ? a.ids[r0 + i] : 0;
        }
        const int e = tid % kMaxExperts, q = tid / kMaxExperts;
        int tot = 0, bef = 0;
        if (e < E) {
#pragma unroll 4
            for (int row = q; row < NB; row += kSumParts) {
                const int v = sa.blk_hist[(int64_t)row * E + e];
                tot += v;
                bef += row < b ? v : 0;
            }
        }
        tot_part[q][e] = tot;
        bef_part[q][e] = bef;
#pragma unroll
        for (int u = 0; u < kSPIds; ++u) {
            const int i = tid + u * kSPWarps * 32;
            if (i < n) sid[i] = ids[u];
        }
    }
    __syncthreads();
    if (tid < 32) {
        // warp-wide exclusive scan of the expert totals (two experts per lane)
        const int lane = tid, e0 = 2 * lane, e1 = 2 * lane + 1;
        int c0 = 0, c1 = 0;
#pragma unroll
        for (int q = 0; q < kSumParts; ++q) {
            c0 += tot_part[q][e0];
            c1 += tot_part[q][e1];
        }
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
        const int x_cnt = s_cnt - c0 - c1;
        const int x_tc = s_tc - (c0 + kTcBM - 1) / kTcBM - (c1 + kTcBM - 1) / kTcBM;
        const int x_si = s_si - (c0 + kSimtBM - 1) / kSimtBM - (c1 + kSimtBM - 1) / kSimtBM;
        if (e0 <= E) off[e0] = x_cnt;
        if (e1 <= E) off[e1] = x_cnt + c0;
        if (E == kMaxExperts && lane == 31) off[kMaxExperts] = s_cnt;
        if (b == 0) {
            if (e0 <= E) {
                sa.offsets[e0] = x_cnt;
                sa.tiles_tc[e0] = x_tc;
                sa.tiles_simt[e0] = x_si;
            }
            if (e1 <= E) {
                sa.offsets[e1] = x_cnt + c0;
                sa.tiles_tc[e1] = x_tc + (c0 + kTcBM - 1) / kTcBM;
                sa.tiles_simt[e1] = x_si + (c0 + kSimtBM - 1) / kSimtBM;
            }
            if (E == kMaxExperts && lane == 31) {
                sa.offsets[kMaxExperts] = s_cnt;
                sa.tiles_tc[kMaxExperts] = s_tc;
                sa.tiles_simt[kMaxExperts] = s_si;
            }
            if (lane == 0) {
                sa.shared_seg[0] = 0;
                sa.shared_seg[1] = sa.T;
                sa.shared_tiles_tc[0] = 0;
                sa.shared_tiles_tc[1] = (sa.T + kTcBM - 1) / kTcBM;
                sa.shared_tiles_simt[0] = 0;
                sa.shared_tiles_simt[1] = (sa.T + kSimtBM - 1) / kSimtBM;
            }
        }
    }
    __syncthreads();
    if (tid < E) {
        int bef = off[tid];
#pragma unroll
        for (int q = 0; q < kSumParts; ++q) bef += bef_part[q][tid];
        base[tid] = bef;
    }
    __syncthreads();
    place_chunk<kSPWarps>(sid, n, r0, E, R, [&](int e) { return base[e]; }, cnt, run, a.perm, a.inv, a.err);
    ptx::griddep_launch_dependents();
}

// The gather xp[i] = x[perm[i] / k], run as the equivalent scatter
// xp[inv[t*k + j]] = x[t]: one warp per token reads its row once (16-byte
// vector loads on the read-only path, sixteen per lane in flight: a whole
// 8 KB row of a 4096-wide bf16 layer; four left the kernel at 0.82 of the HBM
// bandwidth at T = 4096) and writes it to its k routes' rows. Read in route
// order, every row of x would be fetched k times, from DRAM once x outgrows L2.
constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 16;

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherArgs a) {
    ptx::griddep_wait();  // launched early: the permutation is complete past here
    const int lane = threadIdx.x & 31;
    const int64_t T = a.R / a.k;
    const int64_t nwarps = ((int64_t)gridDim.x * kGatherThreads) >> 5;
    const int nvec = (int)(a.row_bytes / 16);
    const uint4* __restrict__ x = static_cast<const uint4*>(a.x);
    uint4* __restrict__ xp = static_cast<uint4*>(a.xp);
    for (int64_t t = ((int64_t)blockIdx.x * kGatherThreads + threadIdx.x) >> 5; t < T; t += nwarps) {
        // lane j < k holds the row of route t*k + j
        const int dst = lane < a.k ? a.inv[t * a.k + lane] : 0;
        if (__any_sync(0xffffffffu, dst < 0 || dst >= a.R)) {
            if (lane == 0) atomicOr(a.err, kErrCheck);
            continue;
        }
        const uint4* src = x + t * nvec;
        for (int v = lane; v < nvec; v += 32 * kGatherUnroll) {
            uint4 buf[kGatherUnroll];
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u)
                if (v + 32 * u < nvec) buf[u] = ld_nc_v4(src + v + 32 * u);
            for (int j = 0; j < a.k; ++j) {
                uint4* out = xp + (int64_t)__shfl_sync(0xffffffffu, dst, j) * nvec;
#pragma unroll
                for (int u = 0; u < kGatherUnroll; ++u)
                    if (v + 32 * u < nvec) out[v + 32 * u] = buf[u];
            }
        }
    }
    ptx::griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s) {
    return launch_kernel(scan_kernel, dim3(1), dim3(kScanThreads), 0, s, true, a);
}

cudaError_t launch_place(const PlaceArgs& a, cudaStream_t s) {
    if (a.NB == 0) return cudaSuccess;
    return launch_kernel(place_kernel, dim3(a.NB), dim3(kPlaceWarps * 32), 0, s, true, a);
}

cudaError_t launch_scan_place(const ScanArgs& sa, const PlaceArgs& a, cudaStream_t s) {
    if (a.NB == 0) return cudaSuccess;
    if ((int64_t)a.NB * a.E > kScanPlaceMaxInts) return cudaErrorInvalidValue;
    return launch_kernel(scan_place_kernel, dim3(a.NB), dim3(kSPWarps * 32), 0, s, true, sa, a);
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s) {
    if (a.R == 0) return cudaSuccess;
    constexpr int kWarps = kGatherThreads / 32;
    const int64_t T = a.R / a.k;
    const int64_t grid = std::min<int64_t>((T + kWarps - 1) / kWarps, (int64_t)a.num_sms * 8);
    return launch_kernel(gather_kernel, dim3((unsigned)grid), dim3(kGatherThreads), 0, s, a.early != 0, a);
}

}  // namespace moe
