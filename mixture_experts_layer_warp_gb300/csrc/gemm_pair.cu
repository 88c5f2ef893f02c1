// gemm_pair.cu - grouped GEMMs of the routed experts on CTA pairs (sm_103a).
//
// "HunyuanImage3 Hybrid Parallelism", section 6.1/6.2: every micro-shard runs
// grouped GEMM1 -> split gate/up -> SwiGLU -> grouped GEMM2 over the
// expert-sorted routes; the micro partials are added in fp32 and the finalize
// runs once. Ascend Hunyuan Image 3.0 guide, section 2.2: the expert is
// down(SiLU(gate(x)) * up(x)) with w13 = [gate; up].
//
// Operand roles. The two CTAs of a cluster issue one tcgen05.mma.cta_group::2
// of M = 256 weight rows (128 held by each CTA) by N tokens (N/2 token rows
// held by each CTA), so each CTA stages 16 KB of weights and at most 16 KB of
// token rows per 64-deep K stage: half the operand bytes per SM of a one-SM
// 128 x 256 tile for the same tensor-core work. Tokens on N let a group's
// rows be cut into chunks of at most 256 padded to a multiple of 16 (a group
// of c routes costs about c columns, not ceil(c / 128) * 128 rows; M = 256
// pair MMAs take any N that is a multiple of 16 up to 256).
//
//   SwiGLU (GEMM1): a tile is (micro m, expert e, 128 features f*128.., one
//       chunk of e's routes). CTA r holds features f*128 + r*64 + [0, 64) as
//       four groups of 16 gate rows followed by the 16 matching up rows (one
//       box of a 5D map over w13), so TMEM lanes 32j..32j+15 of each CTA hold
//       gate and lanes 32j+16..32j+31 the up values of the same 16 features:
//       an epilogue warp pairs them with one shuffle per two tokens and writes
//       silu(gate) * up as bf16 into h[route][m*I + feature].
//   down (GEMM2): a tile is (expert e, 256 output columns f*256.., one chunk).
//       CTA r holds w2 rows f*256 + r*128 + [0, 128). The K loop runs over
//       micro 0's I columns of h against w2[0][e], then micro 1's against
//       w2[1][e], ... into ONE fp32 TMEM accumulator: the per-micro partial
//       outputs of the pages never exist.
//
// Structure: persistent pairs, static round-robin over tiles in the order
// expert -> micro -> feature tile -> chunk, so the pairs working at the same
// time share one expert's token rows and weight tiles through L2. 8 warps per
// CTA: warp 0 issues TMA loads into a 6-stage ring (both CTAs; completion
// counted on the leader's barrier), warp 1 of the leader issues the MMAs into
// one of two TMEM accumulators (2 x 256 fp32 columns), warp 2 owns the TMEM
// allocation, warps 4-7 drain an accumulator (one TMEM lane quarter each,
// transposed through shared memory into 16-byte stores of token rows) while
// the next tile accumulates into the other. With block-scaled FP8 operands
// warp 3 loads the scales into a ring of their own and warps 8-15 (two sets
// taking alternate stages) copy them into TMEM (see Cfg). All waits are bounded, and every load a CTA issues has
// landed before it exits.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStages = 6;
constexpr int kWRows = 128;                          // weight rows per CTA (MMA M = 256 per pair)
constexpr int kABytes = 16384;                       // weight rows of a stage: 128 rows x 128 bytes
constexpr int kBBytes = 16384;                       // up to 128 token rows x 128 bytes per CTA
constexpr int kTmemCols = 512;                       // all of TMEM
constexpr int kEpiArrivals = 8;                      // 4 epilogue warps in each CTA of the pair

// bf16 operands (MX = false): 64 K per stage, chunks of up to 256 routes, two
// 256-column accumulators. MXFP8 operands (MX = true, block-scaled FP8 MMA):
// 128 K per stage (E4M3 codes, one byte each), chunks of up to 208 routes so
// that two accumulators (416 columns) and six scale-factor buffers (16 columns
// each: the weights' words at +0, the routes' at +8) fit the 512 TMEM columns;
// 16 warps. Each stage's scales (the weights' 128 rows x 4 blocks, 512 bytes;
// the token rows' stage-major scale words, 65 x 16 bytes from the chunk's
// first route rounded down to 4) come through a ring of their own, loaded by
// warp 3, so that they run ahead of the operand stages; warps 8-15 (two sets
// of four, alternate stages) copy them into a TMEM buffer as soon as the MMAs
// that read that buffer six stages earlier have completed. (Scales that shared the operand slots could only
// load once a slot freed, and the MMAs then waited out the load latency plus
// the copy into TMEM on every stage.)
template <bool MX>
struct Cfg {
    static constexpr int kSfBufs = kStages;           // scale-factor buffers in TMEM (MX): one per ring slot
    static constexpr int kChunk = MX ? 208 : 256;     // routes per tile at most (MMA N)
    static constexpr int kK = MX ? 128 : 64;          // K elements per stage
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSfStages = MX ? 8 : 0;      // scale ring slots
    static constexpr int kSfaOff = 0;                 // within a scale slot
    static constexpr int kSfaBytes = 512;
    static constexpr int kSfbOff = kSfaOff + kSfaBytes;
    static constexpr int kSfbRows = 65;               // 16-byte rows: 4 routes' scale words each
    static constexpr int kSfbBytes = kSfbRows * 16;
    static constexpr int kSfSlotBytes = 1664;         // 128-byte multiple
    static constexpr int kThreads = MX ? 384 : 256;
    static constexpr int kSfCol = 2 * kChunk;         // scale-factor buffers of 16 columns: SFA at +0, SFB at +8
};
static_assert(Cfg<true>::kSfbOff + Cfg<true>::kSfbBytes <= Cfg<true>::kSfSlotBytes, "scale slot layout");
static_assert(Cfg<true>::kSfCol + Cfg<true>::kSfBufs * 16 <= kTmemCols, "TMEM layout");

struct Ctl {
    uint64_t full[kStages];   // leader: both CTAs' loads of a stage have landed
    uint64_t empty[kStages];  // both CTAs: the MMAs reading a stage are done
    uint64_t tfull[2];        // both CTAs: an accumulator is complete
    uint64_t tempty[2];       // leader: both CTAs' epilogues drained an accumulator
    uint64_t drain;           // leader: every MMA issued has completed
    uint64_t sfs_full[8];     // MX, each CTA: this CTA's scales of a stage have landed in a ring slot
    uint64_t sfs_empty[8];    // MX, each CTA: its 4 scale warps have read a ring slot
    uint64_t sf_full[6];      // MX, leader: both CTAs wrote a scale-factor buffer
    uint64_t rfull[8];        // both CTAs: a tile is in the hand-out ring slot
    uint64_t rempty[8];       // leader: every consuming warp of both CTAs has taken it
    uint2 tring[8];           // the hand-out ring: decoded tiles (pack_tile), x = -1: no more tiles
    uint32_t tmem_base;
    int abort;
    int seg[kMaxExperts + 1];
    int chunks[kMaxExperts + 1];  // prefix over groups of ceil(rows / chunk)
};
constexpr int kDynamicTilesPerPair = 64;  // tiles per pair (bound) from which the hand-out is dynamic
constexpr int kFeed = 4;  // hand-out ring slots: the scheduler runs at most ~2 tiles ahead of the producer

// Epilogue staging, per epilogue warp: one 32-token block of its accumulator
// lanes, transposed through shared memory so that each thread stores 16-byte
// pieces of token rows (GEMM2: 32 x 33 fp32 with a pad column against bank
// conflicts; GEMM1: 32 tokens x 16 features of bf16).
constexpr int kEpiFloats = 32 * 33;
constexpr int kEpiBytes = 4 * kEpiFloats * 4;
// MXFP8 SwiGLU epilogue: past the warp's 32 x 16 bf16 of h, two slots of 32
// per-token |max| read by the partner warp
constexpr int kEpiAmaxOff = 32 * 16 / 2;
static_assert(kEpiAmaxOff + 64 <= kEpiFloats, "epilogue staging");

// Scale-warp sets and threads of a kernel: the MXFP8 down GEMM runs two sets
// of four scale warps on alternate stages (one set took ~700 cycles per stage
// against ~350-420 of MMA work; -8% cycles), the MXFP8 SwiGLU GEMM one (its
// h-quantising epilogue keeps the SM sub-partitions busy enough that four more
// warps slowed it, +7% cycles).
template <bool SWIGLU, bool MX>
constexpr int kSfSets = MX && !SWIGLU ? 2 : 1;
template <bool SWIGLU, bool MX>
constexpr int kPairThreads = Cfg<MX>::kThreads + (kSfSets<SWIGLU, MX> - 1) * 128;

template <bool MX>
constexpr int smem_bytes() {
    return kStages * Cfg<MX>::kStageBytes + Cfg<MX>::kSfStages * Cfg<MX>::kSfSlotBytes + kEpiBytes + (int)sizeof(Ctl) +
           1024;
}
static_assert(smem_bytes<true>() <= 232448 && smem_bytes<false>() <= 232448, "shared memory per CTA");

struct PairTile {
    int m, g, f;
    int start;  // first route row of the chunk
    int len;    // routes in the chunk (<= the chunk size)
    int n;      // MMA N: len rounded up to a multiple of 16 (each CTA holds n/2 rows, whole 8-row atoms)
};

// Token-row map of a chunk: the smallest box (32, 64, 96 or 128 rows) that
// covers the n/2 rows each CTA holds.
__device__ __forceinline__ int token_box(const PairTile& t) { return (t.n / 2 + 31) / 32 - 1; }

// Chunks of one group: ceil(rows / chunk) of near-equal length, so no chunk
// is a nearly empty remainder (the weight bytes of a tile do not shrink with N).
__device__ __forceinline__ PairTile make_tile(int g, int m, int f, int ch, int C, const Ctl& c) {
    PairTile t;
    t.g = g;
    t.m = m;
    t.f = f;
    const int rows = c.seg[g + 1] - c.seg[g];
    const int base = rows / C, rem = rows % C;
    t.start = c.seg[g] + ch * base + min(ch, rem);
    t.len = base + (ch < rem ? 1 : 0);
    t.n = (t.len + 15) & ~15;
    return t;
}

// A pair's walk over its tiles: tiles pair, pair + npairs, ... of the global
// order group -> block of a.chunk_block chunks -> micro -> feature tile ->
// chunk within the block. The pairs running at once take consecutive tiles,
// which share a weight tile and (within a block) token rows through L2; every
// pair gets the same number of tiles within one. A block's token rows stay in
// L2 while every weight tile of the group passes over them, where a group of
// many chunks (the shared expert's dense segment) would otherwise stream all
// its rows once per feature tile. (Handing each pair whole units of one weight
// tile over consecutive chunks instead tripled the DRAM traffic of the CFG
// GEMMs: the pairs then stream several experts' rows at once.)
struct Walk {
    int tile;
    PairTile t;
};

template <bool SWIGLU>
__device__ __forceinline__ bool walk_load(Walk& w, const Ctl& c, const PairGemmArgs& a) {
    const int per = (SWIGLU ? a.n_micro : 1) * a.n_ftiles;  // tiles of a chunk (micros x feature tiles)
    if (w.tile >= per * c.chunks[a.G]) return false;
    int lo = 0, hi = a.G - 1;  // largest g with chunks[g] * per <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (c.chunks[mid] * per <= w.tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int C = c.chunks[lo + 1] - c.chunks[lo];
    int local = w.tile - c.chunks[lo] * per;
    const int Bc = a.chunk_block > 0 && a.chunk_block < C ? a.chunk_block : C;
    const int b = local / (Bc * per) < (C - 1) / Bc ? local / (Bc * per) : (C - 1) / Bc;
    local -= b * Bc * per;
    const int cb = C - b * Bc < Bc ? C - b * Bc : Bc;  // chunks in this block
    int m = 0;
    if (SWIGLU) {
        m = local / (a.n_ftiles * cb);
        local -= m * a.n_ftiles * cb;
    }
    const int f = local / cb;
    w.t = make_tile(lo, m, f, b * Bc + local - f * cb, C, c);
    return true;
}

__device__ __forceinline__ void fail(Ctl& c, int* err) {
    c.abort = 1;
    atomicOr(err, kErrTimeout);
}

// A decoded tile in two words: the chunk's first route row, then len (9 bits,
// <= 256), group (7 bits), micro (3 bits) and feature tile (13 bits).
__device__ __forceinline__ uint2 pack_tile(const PairTile& t) {
    return make_uint2((uint32_t)t.start,
                      (uint32_t)t.len | ((uint32_t)t.g << 9) | ((uint32_t)t.m << 16) | ((uint32_t)t.f << 19));
}
__device__ __forceinline__ PairTile unpack_tile(uint2 w) {
    PairTile t;
    t.start = (int)w.x;
    t.len = (int)(w.y & 511u);
    t.g = (int)((w.y >> 9) & 127u);
    t.m = (int)((w.y >> 16) & 7u);
    t.f = (int)(w.y >> 19);
    t.n = (t.len + 15) & ~15;
    return t;
}

// Tile hand-out. The pairs take tiles of the order above from a global counter
// (a.sched[0]) as they become free, so the pairs running at once stay on
// consecutive tiles for the whole launch (statically assigned, every pair's
// share was the same but the pairs drifted apart over the ~320 rounds of a
// large launch, and a weight tile shared by neighbouring pairs was fetched
// from HBM again: 13-20 GB of DRAM traffic for the CFG GEMM1's 7 GB). The
// leader's warp 2 (otherwise idle between the TMEM allocation and release)
// takes tiles ahead of use and publishes each index to every warp of the
// pair that walks the tiles: into this CTA's ring slot, and into the peer's
// slot by st.async completing on the peer's barrier; -1 ends the walk. A
// slot is reused once every consuming warp of both CTAs has taken it.
// With few tiles per pair (a.dynamic == 0) the scheduler hands out the static
// sequence pair, pair + npairs, ... instead: pairs that reserve a tile or two
// ahead would leave the last tiles of a short launch unevenly spread (denoise
// GEMMs, ~30-40 tiles per pair: 0.51 -> 0.57 ms), where drift never builds up.
// The scheduler also decodes each tile (walk_load) before it publishes it, so
// no consuming warp spends the binary search and divisions between two tiles:
// in the MMA warp they left the tensor pipe idle ~900 cycles per tile (7% of
// the denoise GEMM2, whose tiles are short).
//   take: the next tile for a consuming warp (0; -1: no more; -2: a wait ran out).
//   hand_out: the scheduler warp's loop.
__device__ __forceinline__ int feed_take(Ctl& c, int& n, bool leader, uint32_t rempty0, const PairGemmArgs& a,
                                         PairTile& t) {
    const int slot = n % kFeed;
    const bool got = ptx::mbar_wait(ptx::smem_u32(&c.rfull[slot]), (uint32_t)(n / kFeed) & 1u, a.limit_ns, &c.abort);
    if (!__all_sync(0xffffffffu, got)) return -2;
    // the shuffles need the loaded values, so the reads are complete before the
    // arrival below lets the scheduler write the slot again
    const volatile uint2* src = &c.tring[slot];
    uint2 w;
    w.x = __shfl_sync(0xffffffffu, src->x, 0);
    w.y = __shfl_sync(0xffffffffu, src->y, 0);
    if ((threadIdx.x & 31) == 0) {
        if (leader)
            ptx::mbar_arrive(ptx::smem_u32(&c.rempty[slot]));
        else
            ptx::mbar_arrive_remote(rempty0 + (uint32_t)(slot * sizeof(uint64_t)));
    }
    ++n;
    if ((int)w.x < 0) return -1;
    t = unpack_tile(w);
    return 0;
}

template <bool SWIGLU>
__device__ __forceinline__ void hand_out(Ctl& c, int total, const PairGemmArgs& a, int pair, int npairs) {
    const uint32_t peer_tring = ptx::map_to_rank(ptx::smem_u32(&c.tring[0]), 1);
    const uint32_t peer_rfull = ptx::map_to_rank(ptx::smem_u32(&c.rfull[0]), 1);
    for (int n = 0;; ++n) {
        const int slot = n % kFeed;
        const bool got = ptx::mbar_wait(ptx::smem_u32(&c.rempty[slot]), ((uint32_t)(n / kFeed) & 1u) ^ 1u, a.limit_ns,
                                        &c.abort);
        if (!__all_sync(0xffffffffu, got)) {
            if ((threadIdx.x & 31) == 0) fail(c, a.err);
            return;
        }
        int end = 0;
        if ((threadIdx.x & 31) == 0) {
            const int tile = a.dynamic ? atomicAdd(a.sched, 1) : pair + n * npairs;
            Walk w{tile, {}};
            const bool live = tile < total && walk_load<SWIGLU>(w, c, a);
            const uint2 word = live ? pack_tile(w.t) : make_uint2(0xffffffffu, 0u);
            end = live ? 0 : 1;
            c.tring[slot] = word;
            ptx::mbar_arrive(ptx::smem_u32(&c.rfull[slot]));
            const uint32_t rf = peer_rfull + (uint32_t)(slot * sizeof(uint64_t));
            ptx::mbar_arrive_expect_tx_remote(rf, 8);
            ptx::st_async_u32(peer_tring + (uint32_t)(slot * 8), word.x, rf);
            ptx::st_async_u32(peer_tring + (uint32_t)(slot * 8 + 4), word.y, rf);
        }
        if (__shfl_sync(0xffffffffu, end, 0)) return;
    }
}

// Failure path of a CTA whose loads complete on the other CTA's barrier: it
// cannot wait for them itself, so it gives any copy still in flight 1 ms to
// land before the CTA can leave (copies take microseconds).
__device__ __forceinline__ void settle_inflight_copies() {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 1000000ull) {
    }
}

template <bool SWIGLU, bool MX>
__global__ void __launch_bounds__(kPairThreads<SWIGLU, MX>, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                     const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmW3,
                     const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
                     const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmX3,
                     const __grid_constant__ CUtensorMap tmSA0, const __grid_constant__ CUtensorMap tmSA1,
                     const __grid_constant__ CUtensorMap tmSA2, const __grid_constant__ CUtensorMap tmSA3,
                     const __grid_constant__ CUtensorMap tmSB, const PairGemmArgs a) {
    using C = Cfg<MX>;
    constexpr int kChunk = C::kChunk;
    constexpr int kStageBytes = C::kStageBytes;
    constexpr int kThreads = kPairThreads<SWIGLU, MX>;
    extern __shared__ unsigned char smem_raw[];
    // the same offset in both CTAs: the leader's MMA addresses the peer's
    // operands through its own shared-memory descriptors
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sf_ring = smem + kStages * kStageBytes;  // MX: C::kSfStages scale slots
    float* epi_buf = reinterpret_cast<float*>(sf_ring + C::kSfStages * C::kSfSlotBytes);
    Ctl& c = *reinterpret_cast<Ctl*>(sf_ring + C::kSfStages * C::kSfSlotBytes + kEpiBytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&c.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&c.tfull[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.tempty[b]), kEpiArrivals);
        }
        ptx::mbar_init(ptx::smem_u32(&c.drain), 1);
        // the warps that take every tile index: producer + MMA + 4 epilogue
        // warps (leader), producer + 4 epilogue warps (peer), and with MXFP8
        // operands the scale producer and the 4 or 8 scale warps of each CTA
        for (int r = 0; r < kFeed; ++r) {
            ptx::mbar_init(ptx::smem_u32(&c.rfull[r]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.rempty[r]), MX ? 21 + 8 * (kSfSets<SWIGLU, MX> - 1) : 11);
        }
        if (MX) {
            for (int s = 0; s < C::kSfStages; ++s) {
                ptx::mbar_init(ptx::smem_u32(&c.sfs_full[s]), 1);
                ptx::mbar_init(ptx::smem_u32(&c.sfs_empty[s]), 4);  // the 4 scale warps of this CTA
            }
            for (int b = 0; b < C::kSfBufs; ++b) {
                ptx::mbar_init(ptx::smem_u32(&c.sf_full[b]), 8);  // 4 scale-factor warps in each CTA
            }
        }
        c.abort = 0;
        ptx::fence_mbar_init();
    }
    // launched early (a.early): the segments and token rows are complete past here
    ptx::griddep_wait();
    if (a.seg != nullptr) {
        for (int i = threadIdx.x; i <= a.G; i += kThreads) c.seg[i] = a.seg[i];
    } else if (threadIdx.x == 0) {  // one dense segment (the shared expert over all T rows)
        c.seg[0] = 0;
        c.seg[1] = a.dense_rows;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        c.chunks[0] = 0;
        for (int g = 0; g < a.G; ++g) c.chunks[g + 1] = c.chunks[g] + (c.seg[g + 1] - c.seg[g] + kChunk - 1) / kChunk;
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmW0);
        ptx::prefetch_tmap(&tmX0);
    }
    if (warp == 2) {
        ptx::tmem_alloc_pair(ptx::smem_u32(&c.tmem_base), kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    // the barriers of both CTAs are initialised and the TMEM columns allocated
    // before either CTA signals the other
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();

    const uint32_t tmem = c.tmem_base;
    const int n_micro_k = SWIGLU ? 1 : a.n_micro;
    const int total = (SWIGLU ? a.n_micro : 1) * a.n_ftiles * c.chunks[a.G];
    const uint32_t rempty0 = ptx::map_to_rank(ptx::smem_u32(&c.rempty[0]), 0);  // the leader's

    // The producer and MMA roles run as whole warps: every lane takes part in
    // the waits and the bookkeeping (so the descriptors and coordinates are
    // warp-uniform values), and one elected lane issues the TMA and tcgen05
    // instructions. A single-lane loop issued each tcgen05.mma about 85 cycles
    // apart, close to the 128 tensor-core cycles of one M256 x N256 x K16 MMA.
    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        const bool issuer = ptx::elect_one();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t last_par[kStages];
        int issued = 0;
        bool ok = true;
        int fn = 0;
        while (ok) {
            PairTile t;
            const int got = feed_take(c, fn, leader, rempty0, a, t);
            if (got == -2) ok = false;
            if (got < 0) break;
            const int half = t.n / 2;               // token rows held by each CTA
            const int box = token_box(t);
            const CUtensorMap* tx = box == 0 ? &tmX0 : box == 1 ? &tmX1 : box == 2 ? &tmX2 : &tmX3;
            const uint32_t bytes = 2u * (uint32_t)(kABytes + (box + 1) * 32 * kTcBK * 2);
            const int xrow = t.start + (int)rank * half;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = SWIGLU ? t.m : mi;
                const CUtensorMap* tw = pick_map(m, tmW0, tmW1, tmW2, tmW3);
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    const bool got = ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, a.limit_ns, &c.abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
                    const uint32_t fb = ptx::smem_u32(&c.full[stage]);
                    const uint32_t fb_leader = ptx::map_to_rank(fb, 0);
                    if (issuer) {
                        if (leader) ptx::mbar_arrive_expect_tx(fb, bytes);
                        if (SWIGLU) {
                            // 4 groups of (16 gate rows, 16 up rows) of features f*128 + r*64 ..
                            ptx::tma_load_5d_pair(sa, tw, kb * C::kK, 0, 0, (t.f * 128 + (int)rank * 64) / 16, t.g,
                                                  fb_leader);
                            ptx::tma_load_2d_pair(sb, tx, kb * C::kK, xrow, fb_leader);
                        } else {
                            ptx::tma_load_2d_pair(sa, tw, kb * C::kK,
                                                  t.g * a.w_rows_per_group + t.f * 256 + (int)rank * 128, fb_leader);
                            ptx::tma_load_2d_pair(sb, tx, m * a.x_micro_cols + kb * C::kK, xrow, fb_leader);
                        }
                    }
                    __syncwarp();
                    last_par[stage] = phase;
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (!ok && issuer) fail(c, a.err);
        if (issuer) {
            if (leader) {
                // every load issued (either CTA's) lands before the pair can exit, also
                // when another role gave up on it: the last phase of each slot completes
                const int n = issued < kStages ? issued : kStages;
                for (int s = 0; s < n; ++s)
                    ptx::mbar_wait(ptx::smem_u32(&c.full[s]), last_par[s], a.limit_ns, nullptr);
            } else if (!ok) {
                settle_inflight_copies();
            }
        }
    } else if (warp == 2 && leader) {
        // ------------------------------------------------ tile scheduler (leader)
        hand_out<SWIGLU>(c, total, a, pair, npairs);
    } else if (warp == 1 && leader) {
        // ------------------------------------------------ MMA issuer (leader)
        const bool issuer = ptx::elect_one();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int local = 0;
        int sfi = 0;  // MX: stages consumed, which picks the scale-factor buffer and its phase
        int fn = 0;
        for (; ok; ++local) {
            PairTile t;
            const int got = feed_take(c, fn, true, rempty0, a, t);
            if (got == -2) ok = false;
            if (got < 0) break;
            const uint32_t idesc = ptx::idesc_bf16_f32(2 * kWRows, t.n);
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            const bool drained = ptx::mbar_wait(ptx::smem_u32(&c.tempty[acc]), acc_par ^ 1u, a.limit_ns, &c.abort);
            if (!__all_sync(0xffffffffu, drained)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * kChunk);
            uint32_t accumulate = 0;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    const int sfb = sfi % C::kSfBufs;  // MX: scale-factor buffer of this stage
                    bool got = ptx::mbar_wait(ptx::smem_u32(&c.full[stage]), phase, a.limit_ns, &c.abort);
                    if (MX)  // both CTAs' scale words are in tensor memory
                        got = got && ptx::mbar_wait(ptx::smem_u32(&c.sf_full[sfb]), (uint32_t)(sfi / C::kSfBufs) & 1u,
                                                    a.limit_ns, &c.abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint64_t adesc = ptx::sw128_desc(sa);
                    const uint64_t bdesc = ptx::sw128_desc(sa + kABytes);
                    if (issuer) {
                        if (MX) {
                            // 4 MMAs of 32 codes; byte k of every scale word belongs to the k-th
                            const uint32_t sfa_t = tmem + (uint32_t)(C::kSfCol + sfb * 16);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                ptx::mma_mx_pair(d, adesc + 2u * k, bdesc + 2u * k, ptx::idesc_mx(2 * kWRows, t.n, k, k),
                                                 sfa_t, sfa_t + 8u, accumulate | (uint32_t)k);
                            // frees the ring slot and its scale buffer (buffer sfb = slot stage)
                            ptx::mma_commit_pair_both(ptx::smem_u32(&c.empty[stage]));
                        } else {
#pragma unroll
                            for (int k = 0; k < kTcBK / 16; ++k)
                                ptx::mma_bf16_pair(d, adesc + 2u * k, bdesc + 2u * k, idesc, accumulate | (uint32_t)k);
                            ptx::mma_commit_pair_both(ptx::smem_u32(&c.empty[stage]));
                        }
                    }
                    __syncwarp();
                    accumulate = 1;
                    ++sfi;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok && issuer) ptx::mma_commit_pair_both(ptx::smem_u32(&c.tfull[acc]));
            __syncwarp();
        }
        if (issuer) {
            if (!ok) fail(c, a.err);
            // every MMA issued so far completes before either CTA's TMEM is released
            ptx::mma_commit_pair_local(ptx::smem_u32(&c.drain));
            ptx::mbar_wait(ptx::smem_u32(&c.drain), 0, a.limit_ns, nullptr);
        }
        __syncwarp();
    } else if (MX && warp == 3) {
        // ------------------------------------------------ scale producer (both CTAs)
        // This CTA's scales of every stage into the scale ring, on its own
        // barriers: the weight rows' 4 blocks (the row order of the weight
        // tile) and every route's scale word of the chunk (both CTAs' halves).
        const bool issuer = ptx::elect_one();
        int slot = 0, issued = 0;
        uint32_t phase = 0;
        uint32_t last_par[C::kSfStages > 0 ? C::kSfStages : 1];
        bool ok = true;
        int fn = 0;
        while (ok) {
            PairTile t;
            const int got = feed_take(c, fn, leader, rempty0, a, t);
            if (got == -2) ok = false;
            if (got < 0) break;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = SWIGLU ? t.m : mi;
                const CUtensorMap* tsa = pick_map(m, tmSA0, tmSA1, tmSA2, tmSA3);
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    const bool got =
                        ptx::mbar_wait(ptx::smem_u32(&c.sfs_empty[slot]), phase ^ 1u, a.limit_ns, &c.abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ptx::smem_u32(sf_ring + slot * C::kSfSlotBytes);
                    const uint32_t bar = ptx::smem_u32(&c.sfs_full[slot]);
                    if (issuer) {
                        ptx::mbar_arrive_expect_tx(bar, (uint32_t)(C::kSfaBytes + C::kSfbBytes));
                        if (SWIGLU)
                            ptx::tma_load_5d(dst + C::kSfaOff, tsa, 0, 0, (t.f * 128 + (int)rank * 64) / 16, kb * 4, t.g,
                                             bar);
                        else
                            ptx::tma_load_3d(dst + C::kSfaOff, tsa, t.f * 256 + (int)rank * 128, kb * 4, t.g, bar);
                        ptx::tma_load_3d(dst + C::kSfbOff, &tmSB, 0, t.start >> 2, (SWIGLU ? 0 : m) * a.k_blocks + kb,
                                         bar);
                    }
                    __syncwarp();
                    last_par[slot] = phase;
                    ++issued;
                    if (++slot == C::kSfStages) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (!ok && issuer) fail(c, a.err);
        if (issuer) {
            // every scale load issued lands before the CTA can exit, also when the
            // scale warps gave up on it: the last phase of each slot completes
            const int n = issued < C::kSfStages ? issued : C::kSfStages;
            for (int s2 = 0; s2 < n; ++s2)
                ptx::mbar_wait(ptx::smem_u32(&c.sfs_full[s2]), last_par[s2], a.limit_ns, nullptr);
        }
        __syncwarp();
    } else if (MX && warp >= 8) {
        // ------------------------------------------------ scale factors into TMEM (both CTAs)
        // With two sets of four warps (the down GEMM) they take alternate stages
        // (set p the stages of parity p, so also the ring slots and buffers of
        // parity p). Warp 8 + 4p + q writes lane quarter q of a scale-factor
        // buffer (the MMA reads every quarter):
        // column j, lane L holds the four block scales of weight row L + 32 j
        // (columns +0..3) and the scale word of route L + 32 j of the chunk
        // (columns +8..15); byte i of a word is K block i of the stage.
        constexpr int kSets = kSfSets<SWIGLU, MX>;
        const int q = warp & 3, set = (warp - 8) >> 2;
        static_assert(C::kSfStages % 2 == 0 && C::kSfBufs % 2 == 0, "a set keeps to slots of its parity");
        const uint32_t sf_full0 = ptx::map_to_rank(ptx::smem_u32(&c.sf_full[0]), 0);
        int slot = 0, sfi = 0;
        uint32_t phase = 0;
        bool ok = true;
        int fn = 0;
        while (ok) {
            PairTile t;
            const int got = feed_take(c, fn, leader, rempty0, a, t);
            if (got == -2) ok = false;
            if (got < 0) break;
            const int off = t.start & 3;  // the chunk's first scale word in the loaded 16-byte rows
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    const int sfb = sfi % C::kSfBufs;
                    if (kSets == 2 && (sfi & 1) != set) {  // the other set's stage
                        ++sfi;
                        if (++slot == C::kSfStages) {
                            slot = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    // the stage's scales into registers (the ring slot is then free),
                    // then wait for the TMEM buffer
                    bool got = ptx::mbar_wait(ptx::smem_u32(&c.sfs_full[slot]), phase, a.limit_ns, &c.abort);
                    uint32_t wa[4], wb[8];
                    if (got) {
                        const unsigned char* sfa = sf_ring + slot * C::kSfSlotBytes + C::kSfaOff;  // [4 blocks][128 rows]
                        const uint32_t* sfw =
                            reinterpret_cast<const uint32_t*>(sf_ring + slot * C::kSfSlotBytes + C::kSfbOff);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int r = lane + 32 * j;
                            wa[j] = (uint32_t)sfa[r] | ((uint32_t)sfa[128 + r] << 8) | ((uint32_t)sfa[256 + r] << 16) |
                                    ((uint32_t)sfa[384 + r] << 24);
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) wb[j] = sfw[off + lane + 32 * j];  // routes past the chunk: unused
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&c.sfs_empty[slot]));
                        // the buffer is free once the MMAs of its previous use are done:
                        // buffer sfb goes with ring slot sfb, whose empty barrier the MMA
                        // commit completes (one commit per stage frees both)
                        got = ptx::mbar_wait(ptx::smem_u32(&c.empty[sfb]),
                                             ((uint32_t)(sfi / C::kSfBufs) & 1u) ^ 1u, a.limit_ns, &c.abort);
                    }
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t col = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(C::kSfCol + sfb * 16);
                    ptx::tmem_st4(col, wa[0], wa[1], wa[2], wa[3]);
                    ptx::tmem_st8(col + 8u, wb);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            ptx::mbar_arrive(ptx::smem_u32(&c.sf_full[sfb]));
                        else
                            ptx::mbar_arrive_remote(sf_full0 + (uint32_t)(sfb * sizeof(uint64_t)));
                    }
                    ++sfi;
                    if (++slot == C::kSfStages) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (!ok && lane == 0) fail(c, a.err);
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ epilogue (both CTAs)
        const int q = warp - 4;  // TMEM lanes 32q .. 32q+31
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
        const uint32_t tempty_leader0 = ptx::map_to_rank(ptx::smem_u32(&c.tempty[0]), 0);
        int local = 0, fn = 0;
        for (;; ++local) {
            PairTile t;
            const int got = feed_take(c, fn, leader, rempty0, a, t);
            // the MXFP8 SwiGLU epilogue's warp pairs agree first (see below)
            bool live = got >= 0;
            if (MX && SWIGLU) live = ptx::named_barrier_and(1 + (q >> 1), 64, live);
            if (!live) {
                if (got == -2 && lane == 0) fail(c, a.err);
                break;
            }
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            bool ready = false;
            if (lane == 0)
                ready = ptx::mbar_wait(ptx::smem_u32(&c.tfull[acc]), acc_par, a.limit_ns, &c.abort);
            ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
            // the MXFP8 SwiGLU epilogue pairs warps q and q^1 at a named barrier
            // per 32 tokens: they take the tile, or leave, together
            if (MX && SWIGLU) ready = ptx::named_barrier_and(1 + (q >> 1), 64, ready);
            if (!ready) {
                if (lane == 0) fail(c, a.err);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kChunk);
            float* buf = epi_buf + q * kEpiFloats;
            if (SWIGLU) {
                // lanes 0-15: gate of features feat0 + lane; lanes 16-31: up of the same
                const int feat0 = t.m * a.out_micro_cols + t.f * 128 + (int)rank * 64 + q * 16;
                const bool is_gate = lane < 16;
                __nv_bfloat16* hb = reinterpret_cast<__nv_bfloat16*>(buf);  // [32 tokens][16 features]
#pragma unroll 1
                for (int c0 = 0, it = 0; c0 < t.n; c0 += 32, ++it) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        // token 2i goes to the gate lane, 2i+1 to the up lane; either way
                        // element (token, feature) lands at hb[32 i + lane]
                        const float v0 = __uint_as_float(v[2 * i]), v1 = __uint_as_float(v[2 * i + 1]);
                        const float other = __shfl_xor_sync(0xffffffffu, is_gate ? v1 : v0, 16);
                        const float h = is_gate ? silu(v0) * other : silu(other) * v1;
                        hb[32 * i + lane] = __float2bfloat16_rn(h);
                    }
                    __syncwarp();
                    if (MX) {
                        // MXFP8 of h: lane = token; this warp holds features 16 (q%2) .. +16
                        // of block q/2 of the CTA's 64, the partner warp q^1 the other 16:
                        // each posts its per-token |max| (two slots by chunk parity) and
                        // the pair meets at a named barrier
                        const uint4* hr = reinterpret_cast<const uint4*>(hb + lane * 16);
                        const uint4 p0 = hr[0], p1 = hr[1];
                        const __nv_bfloat162* hv0 = reinterpret_cast<const __nv_bfloat162*>(&p0);
                        const __nv_bfloat162* hv1 = reinterpret_cast<const __nv_bfloat162*>(&p1);
                        float2 f[8];
                        float am = 0.f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            f[i] = __bfloat1622float2(hv0[i]);
                            f[4 + i] = __bfloat1622float2(hv1[i]);
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) am = fmaxf(am, fmaxf(fabsf(f[i].x), fabsf(f[i].y)));
                        float* amx = buf + kEpiAmaxOff;
                        amx[(it & 1) * 32 + lane] = am;
                        ptx::named_barrier_sync(1 + (q >> 1), 64);
                        am = fmaxf(am, epi_buf[(q ^ 1) * kEpiFloats + kEpiAmaxOff + (it & 1) * 32 + lane]);
                        const int shared = mx_shared_exp(am);
                        const float sc = pow2f(-shared);  // exact: a power-of-two scaling
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            w[i] = e4m3x2(f[2 * i].x * sc, f[2 * i].y * sc) |
                                   (e4m3x2(f[2 * i + 1].x * sc, f[2 * i + 1].y * sc) << 16);
                        if (c0 + lane < t.len) {
                            const int64_t row = t.start + c0 + lane;
                            unsigned char* codes = static_cast<unsigned char*>(a.out);
                            *reinterpret_cast<uint4*>(codes + row * a.out_ld + feat0) = make_uint4(w[0], w[1], w[2], w[3]);
                            if ((q & 1) == 0) {  // one scale byte per block: K block feat0/32 of the row
                                const int kblk = feat0 / 32;
                                static_cast<unsigned char*>(a.out_scales)[((int64_t)(kblk / 4) * a.out_rows_pad + row) * 4 +
                                                                         (kblk & 3)] = (unsigned char)(shared + 127);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int piece = lane + 32 * j, tok = piece >> 1, half = piece & 1;
                            const uint4 u = *reinterpret_cast<const uint4*>(hb + tok * 16 + half * 8);
                            if (c0 + tok < t.len)
                                *reinterpret_cast<uint4*>(out + (int64_t)(t.start + c0 + tok) * a.out_ld + feat0 + half * 8) = u;
                        }
                    }
                    __syncwarp();
                }
            } else {
                // lane = output feature feat0 + lane; each thread then stores 8
                // features of 4 tokens
                const int feat0 = t.f * 256 + (int)rank * 128 + q * 32;
                const int sub = lane & 3;
#pragma unroll 1
                for (int c0 = 0; c0 < t.n; c0 += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tbase + c0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) buf[i * 33 + lane] = __uint_as_float(v[i]);
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int tok = j * 8 + (lane >> 2);
                        const float* r = buf + tok * 33 + sub * 8;
                        const uint4 u = make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]),
                                                   pack_bf16x2(r[4], r[5]), pack_bf16x2(r[6], r[7]));
                        if (c0 + tok < t.len)
                            *reinterpret_cast<uint4*>(out + (int64_t)(t.start + c0 + tok) * a.out_ld + feat0 + sub * 8) = u;
                    }
                    __syncwarp();
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    ptx::mbar_arrive(ptx::smem_u32(&c.tempty[acc]));
                else
                    ptx::mbar_arrive_remote(tempty_leader0 + (uint32_t)(acc * sizeof(uint64_t)));
            }
        }
    }

    // neither CTA leaves (or frees TMEM) while the other may still signal it
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();
    if (leader && threadIdx.x == 0) {
        // the last pair to finish (every pair has stopped taking tiles) resets
        // the hand-out counter for the next launch in the stream
        __threadfence();
        if (atomicAdd(a.sched + 1, 1) == npairs - 1) {
            a.sched[0] = 0;
            a.sched[1] = 0;
            __threadfence();
        }
    }
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// Pairs resident at once (one per TPC at most), looked up once per device.
template <bool SWIGLU, bool MX>
int max_pairs() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] > 0) return cached[dev];
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kPairThreads<SWIGLU, MX>);
    cfg.dynamicSmemBytes = smem_bytes<MX>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, pair_gemm_kernel<SWIGLU, MX>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    cached[dev] = n;
    return n;
}

template <bool SWIGLU, bool MX>
cudaError_t launch_pair(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                        const CUtensorMap* tmSA, const CUtensorMap& tmSB, cudaStream_t s) {
    if (a.max_tiles <= 0) return cudaSuccess;
    constexpr int smem = smem_bytes<MX>();
    if (cudaError_t e = ensure_smem_limit<pair_gemm_kernel<SWIGLU, MX>>(smem); e != cudaSuccess) return e;
    const int pairs_max = max_pairs<SWIGLU, MX>();
    if (pairs_max <= 0) return cudaErrorLaunchOutOfResources;
    const int pairs = a.max_tiles < pairs_max ? a.max_tiles : pairs_max;
    PairGemmArgs ad = a;
    ad.dynamic = a.max_tiles >= kDynamicTilesPerPair * pairs ? 1 : 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kPairThreads<SWIGLU, MX>);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.early ? 2 : 1;
    const int nm = a.n_micro;
    return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<SWIGLU, MX>, tmW[0], tmW[nm > 1 ? 1 : 0], tmW[nm > 2 ? 2 : 0],
                              tmW[nm > 3 ? 3 : 0], tmX[0], tmX[1], tmX[2], tmX[3], tmSA[0], tmSA[nm > 1 ? 1 : 0],
                              tmSA[nm > 2 ? 2 : 0], tmSA[nm > 3 ? 3 : 0], tmSB, ad);
}

}  // namespace

// bf16 operands: the scale-map parameters are unused (any valid map).
cudaError_t launch_pair_gemm_swiglu(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                    cudaStream_t s) {
    return launch_pair<true, false>(a, tmW, tmX, tmW, tmX[0], s);
}

cudaError_t launch_pair_gemm_down(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                  cudaStream_t s) {
    return launch_pair<false, false>(a, tmW, tmX, tmW, tmX[0], s);
}

cudaError_t launch_pair_gemm_swiglu_mx(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                       const CUtensorMap* tmSA, const CUtensorMap& tmSB, cudaStream_t s) {
    return launch_pair<true, true>(a, tmW, tmX, tmSA, tmSB, s);
}

cudaError_t launch_pair_gemm_down_mx(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                     const CUtensorMap* tmSA, const CUtensorMap& tmSB, cudaStream_t s) {
    return launch_pair<false, true>(a, tmW, tmX, tmSA, tmSB, s);
}

}  // namespace moe
