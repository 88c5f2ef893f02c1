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
}

constexpr int kPlaceWarps = 8;

__global__ void __launch_bounds__(kPlaceWarps * 32) place_kernel(PlaceArgs a) {
    __shared__ int sid[kRouterTokensTc * kMaxTopK];
    __shared__ int cnt[kPlaceWarps][kMaxExperts];
    __shared__ int run[kPlaceWarps][kMaxExperts];
    const int64_t R = (int64_t)a.T * a.k;
    const int64_t r0 = (int64_t)blockIdx.x * a.tok_per_blk * a.k;
    const int64_t left = R - r0;
    const int n = (int)(left < (int64_t)a.tok_per_blk * a.k ? left : (int64_t)a.tok_per_blk * a.k);
    for (int i = threadIdx.x; i < n; i += blockDim.x) sid[i] = a.ids[r0 + i];
    __syncthreads();
    const int32_t* base = a.blk_base + (int64_t)blockIdx.x * a.E;
    place_chunk<kPlaceWarps>(sid, n, r0, a.E, R, [&](int e) { return base[e]; }, cnt, run, a.perm, a.inv, a.err);
}

// Gather xp[i] = x[perm[i] / k]: each single-warp block moves one row chunk
// at a time global -> shared -> global with bulk (TMA engine) copies; many
// blocks per SM keep enough bytes in flight to stream at HBM rate.
constexpr uint32_t kGatherChunk = 16384;

__global__ void __launch_bounds__(32) gather_kernel(GatherArgs a) {
    __shared__ __align__(128) unsigned char buf[kGatherChunk];
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t sbuf = ptx::smem_u32(buf), sbar = ptx::smem_u32(&bar);
    ptx::mbar_init(sbar, 1);
    ptx::fence_mbar_init();
    const uint32_t chunks = (a.row_bytes + kGatherChunk - 1) / kGatherChunk;
    const int64_t units = (int64_t)a.R * chunks;
    const unsigned char* x = static_cast<const unsigned char*>(a.x);
    unsigned char* xp = static_cast<unsigned char*>(a.xp);
    uint32_t phase = 0;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t i = u / chunks;
        const uint32_t c = (uint32_t)(u - i * chunks);
        const uint32_t bytes = min(kGatherChunk, a.row_bytes - c * kGatherChunk);
        const int32_t r = a.perm[i];
        if (r < 0 || r >= a.R) {
            atomicOr(a.err, kErrCheck);
            continue;
        }
        const int64_t t = r / a.k;
        ptx::bulk_wait_read_all();  // the previous store has finished reading buf
        ptx::mbar_arrive_expect_tx(sbar, bytes);
        ptx::bulk_g2s(sbuf, x + t * a.row_bytes + (int64_t)c * kGatherChunk, bytes, sbar);
        if (!ptx::mbar_wait(sbar, phase, a.limit_ns, nullptr)) {
            atomicOr(a.err, kErrTimeout);
            ptx::mbar_wait(sbar, phase, a.limit_ns, nullptr);  // let the copy land before exit
            break;
        }
        phase ^= 1u;
        ptx::fence_proxy_async_smem();
        ptx::bulk_s2g(xp + i * a.row_bytes + (int64_t)c * kGatherChunk, sbuf, bytes);
        ptx::bulk_commit();
    }
    ptx::bulk_wait_all();
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s) {
    scan_kernel<<<1, kScanThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_place(const PlaceArgs& a, cudaStream_t s) {
    if (a.NB == 0) return cudaSuccess;
    place_kernel<<<a.NB, kPlaceWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s) {
    if (a.R == 0) return cudaSuccess;
    const int64_t chunks = (a.row_bytes + kGatherChunk - 1) / kGatherChunk;
    const int64_t units = (int64_t)a.R * chunks;
    const int64_t grid = std::min<int64_t>(units, (int64_t)a.num_sms * 12);
    gather_kernel<<<(unsigned)grid, 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
