// place.cuh - stable placement of a contiguous chunk of routes, one warp-round
// of 32 routes at a time.
//
// Routes r0 .. r0+n-1 (flattened r = t*k + j, ids in shared memory) are split
// into NW contiguous sub-chunks, one per warp. Each warp counts its
// sub-chunk per expert, the counts are scanned across warps per expert from
// base[e] (the first sorted position of this chunk's expert-e routes), and
// each warp then writes perm[pos] = r and inv[r] = pos. Within a 32-route round
// the lanes that carry the same expert form a group (match_expert) and a
// lane's rank is the number of lower lanes in its group, so the order of
// routes inside an expert is ascending r: the counting sort is stable and
// involves no atomics on the output order.
#pragma once

#include "kernels.h"

namespace moe {

// The lanes of the warp that hold the same expert id as this lane (ids in
// [0, 64); -1: no route): the AND over the id's six bits of the ballot of
// lanes agreeing on that bit, restricted to lanes that hold a route. Seven
// ballots, where __match_any_sync took about a thousand cycles per round.
__device__ __forceinline__ unsigned match_expert(int id) {
    unsigned m = __ballot_sync(0xffffffffu, id >= 0);
#pragma unroll
    for (int b = 0; b < 6; ++b) {
        const bool bit = (id >> b) & 1;
        const unsigned v = __ballot_sync(0xffffffffu, bit);
        m &= bit ? v : ~v;
    }
    return m;
}
static_assert(kMaxExperts <= 64, "match_expert compares six bits; 32 warps scan two experts each");

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
        int id = i < hi ? sid[i] : -1;
        if (id >= kMaxExperts || id < -1) id = -1;  // flagged in the second pass
        const unsigned peers = match_expert(id);
        if (id >= 0 && (peers & lt) == 0) cnt[warp][id] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    if (NW == 32) {
        // warp v scans experts 2v and 2v+1 across the 32 warps' counts (lane = warp)
        for (int e = 2 * warp; e < 2 * warp + 2; ++e) {
            if (e >= E) break;
            const int c = cnt[lane][e];
            int incl = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += o;
            }
            run[lane][e] = base_e(e) + incl - c;
        }
    } else if ((int)threadIdx.x < E) {
        int acc = base_e(threadIdx.x);
        for (int w = 0; w < NW; ++w) {
            run[w][threadIdx.x] = acc;
            acc += cnt[w][threadIdx.x];
        }
    }
    __syncthreads();
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const int raw = i < hi ? sid[i] : -1;
        const int id = raw >= kMaxExperts || raw < -1 ? -1 : raw;
        if (i < hi && id < 0) atomicOr(err, kErrCheck);  // an id no expert has
        const unsigned peers = match_expert(id);
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
