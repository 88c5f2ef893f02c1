// place.cuh - stable placement of a contiguous chunk of routes, one warp-round
// of 32 routes at a time.
//
// Routes r0 .. r0+n-1 (flattened r = t*k + j, ids in shared memory) are split
// into NW contiguous sub-chunks, one per warp. Each warp counts its
// sub-chunk per expert, the counts are scanned across warps per expert from
// base[e] (the first sorted position of this chunk's expert-e routes), and
// each warp then writes perm[pos] = r and inv[r] = pos. Within a 32-route round
// __match_any_sync groups the lanes that carry the same expert and a lane's
// rank is the number of lower lanes in its group, so the order of routes
// inside an expert is ascending r: the counting sort is stable and involves no
// atomics on the output order.
#pragma once

#include "kernels.h"

namespace moe {

// Scratch in shared memory: cnt[NW][kMaxExperts], run[NW][kMaxExperts].
// base_e(e) gives this chunk's first sorted position for expert e.
template <int NW, typename BaseFn>
__device__ __forceinline__ void place_chunk(const int* sid, int n, int64_t r0, int E, int64_t R, BaseFn base_e,
                                            int (*cnt)[kMaxExperts], int (*run)[kMaxExperts], int32_t* perm,
                                            int32_t* inv, int* err) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int per = (n + NW - 1) / NW;
    const int lo = min(n, warp * per), hi = min(n, lo + per);
    const unsigned lt = (1u << lane) - 1u;
    for (int e = lane; e < kMaxExperts; e += 32) cnt[warp][e] = 0;
    __syncwarp();
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const int id = i < hi ? sid[i] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        if (id >= 0 && (peers & lt) == 0) cnt[warp][id] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    if ((int)threadIdx.x < E) {
        int acc = base_e(threadIdx.x);
        for (int w = 0; w < NW; ++w) {
            run[w][threadIdx.x] = acc;
            acc += cnt[w][threadIdx.x];
        }
    }
    __syncthreads();
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const int id = i < hi ? sid[i] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        if (id >= 0 && id < E) {
            const int pos = run[warp][id] + __popc(peers & lt);
            if (pos >= 0 && pos < R) {
                perm[pos] = (int32_t)(r0 + i);
                inv[r0 + i] = pos;
            } else {
                atomicOr(err, kErrCheck);
            }
        } else if (id >= 0) {
            atomicOr(err, kErrCheck);
        }
        __syncwarp();
        if (id >= 0 && id < E && (peers & lt) == 0) run[warp][id] += __popc(peers);
        __syncwarp();
    }
}

}  // namespace moe
