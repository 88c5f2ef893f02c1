// gemm_small.cu - the grouped GEMMs for batches of at most 16 tokens
// (AR-decode-sized calls), with the operands swapped.
//
// Same computation as gemm_pair.cu ("HunyuanImage3 Hybrid Parallelism",
// section 6.1: per micro grouped GEMM1 -> SwiGLU -> grouped GEMM2, micros
// summed in fp32), but with T <= 16 every expert owns at most 16 routes, so
// the expert WEIGHTS take the MMA's M side (128 rows) and the expert's token
// rows its N side (N = 16): each K stage moves 16 KB of weights and 2 KB of
// activations instead of 16 KB of mostly-padding activation rows. The layer is
// then a weight stream, bounded by HBM bandwidth.
//   SwiGLU tile (GEMM1): (expert e, micro m, 64 columns of h): the A tile
//       stacks 64 gate rows of w13[m][e] over the matching 64 up rows, so TMEM
//       lanes 0-63 hold gate and 64-127 up for the 16 tokens; the epilogue
//       pairs them through shared memory and writes silu(gate) * up.
//   down tile (GEMM2): (expert e, 128 output columns), K runs over all micros
//       into one accumulator.
// The routed layer runs both in ONE persistent launch: the work list is every
// SwiGLU tile (expert order) followed by every down tile. A down tile of
// expert e first waits until all SwiGLU tiles of e have stored their h rows (a
// per-expert counter, bounded wait), so the down projection's weight stream
// starts on SMs as soon as they run out of SwiGLU tiles instead of after the
// slowest one, and one kernel boundary disappears. CTA b starts with tile b;
// the later tiles (and the finalize items) are handed out in increasing order
// to CTAs that are running. A down tile therefore only waits for SwiGLU tiles
// held by CTAs that are running or start as soon as an SM frees up, and no CTA
// needs all others to be resident: the launch is an ordinary one with
// programmatic dependent launch, so the CTAs that find a free SM set up while
// the router still runs and the rest join when the router's SMs free up. Before its tiles, each of the first kGatherCtas
// CTAs' epilogue warps gather a share of the routed token rows (a SwiGLU tile
// waits only for its expert's rows, and its weight stages are issued
// meanwhile); after its tiles they take finalize items from a global counter
// (the CTAs that run out of tiles first take them), each gated on the down
// tiles of its token's experts. The whole routed layer after routing is
// therefore one launch.
// Structure: 12-stage TMA ring, one MMA issuer, four epilogue warps on a
// double-buffered 2 x 16-column TMEM accumulator. In the fused mode a fifth
// role, the scheduler thread, claims the next tile from the global counter and
// waits for its dependency (the expert's SwiGLU tiles, or its gathered rows)
// while the producer streams the current one, so neither global round trip
// sits between two tiles of the weight stream. All waits are bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTok = kSmallTokens;             // 16: MMA N
constexpr int kM = 128;                        // MMA M: weight rows
constexpr int kStages = 12;
constexpr int kABytes = kM * kTcBK * 2;        // 16 KB
constexpr int kBBytes = kTok * kTcBK * 2;      // 2 KB
constexpr int kStageBytes = kABytes + kBBytes; // 18 KB (a multiple of 1024)
constexpr int kTmemCols = 32;                  // 2 accumulators x 16 columns
constexpr int kThreads = 256;
constexpr int kGatherCtas = 128;               // kFused: CTAs that gather token rows
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kM, kTok);

// MXFP8 expert weights (fused mode, moe_forward_mxfp8): a stage covers 256 K
// as two 128-K code chunks, so each weight row moves 128 contiguous bytes of
// E4M3 codes per TMA row (a 64-byte row halves the sustained stream rate) and
// a stage is three TMA instructions for 32 KB of codes (the producer thread's
// TMA issue, about as slow per instruction whatever the box, bounds the stream
// otherwise); the codes arrive 128-byte swizzled with the eight E8M0 scales of
// each row and four 64-K token-row tiles. A layer whose K is an odd multiple of
// 128 ends with half a stage: the boxes past the weights read zero codes. Eight dequant warps (8..15:
// two per TMEM lane quadrant, taking alternate stages) turn each weight row's
// 128 codes into f16, code * 2^(S-127) rounded to f16, in registers and store
// them into one of kF8Dq A buffers in tensor memory; the MMA reads A from
// tensor memory and the token rows (f16: the gathered rows and h) from shared
// memory, into fp32 accumulators as before; two threads issue the MMAs (a
// tile's even and odd stages, into two accumulator halves the epilogue adds).
// No dequantised tile passes through shared memory.
constexpr int kF8Stages = 5;
constexpr int kF8Chunks = 4;                         // 64-K MMA chunks per stage
constexpr int kF8K = kF8Chunks * kTcBK;              // 256 K per stage
constexpr int kF8CodeBytes = kM * kF8K;              // 32 KB of codes: two [128 rows][128 K] chunks
constexpr int kF8ScaleBytes = kM * (kF8K / 32);      // 1 KB of scales
constexpr int kF8BBytes = kF8Chunks * kBBytes;       // four 64-K token-row tiles
constexpr int kF8Dq = 3;                             // TMEM A buffers
constexpr int kF8Threads = 512;                      // warps 8..15 dequantise
constexpr int kF8CodeOff = kF8Stages * kF8BBytes;    // after the token-row tiles (1024-aligned)
constexpr int kF8ScaleOff = kF8CodeOff + kF8Stages * kF8CodeBytes;
constexpr int kF8CtlOff = kF8ScaleOff + kF8Stages * kF8ScaleBytes;
constexpr int kF8TmemCols = 512;                     // accumulators at 0..63, A buffers from kF8ACol
constexpr int kF8ACol = 64;                          // A buffer b: columns kF8ACol + kF8ABuf b ..
constexpr int kF8ABuf = kF8K / 2;                    // 128 columns: the stage's f16 pairs
constexpr uint32_t kIdescF16 = ptx::idesc_f16_f32(kM, kTok);
constexpr int kMaxStages = kF8Stages > kStages ? kF8Stages : kStages;
static_assert(kF8ACol + kF8Dq * kF8ABuf <= kF8TmemCols, "A buffers exceed the TMEM allocation");

// Stages of one micro's K (k_blocks 64-K blocks) with MXFP8 weights.
__device__ __forceinline__ int f8_stages(int k_blocks) { return (k_blocks + kF8Chunks - 1) / kF8Chunks; }
static_assert(kF8CodeOff % 1024 == 0 && kF8CodeBytes % 1024 == 0, "128-byte swizzled tiles need 1024-byte alignment");

enum Mode { kSwiGLUOnly = 0, kDownOnly = 1, kFused = 2 };

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t drain2;  // MXFP8: the second MMA issuer's
    uint32_t tmem_base;
    int abort;
    int seg[kMaxExperts + 1];
    int tiles[kMaxExperts + 1];
    float up[64][kTok + 1];
    int ep_ok[4];
    int fin_fail;
    int fin_item;
    // kFused: tiles fetched from a global counter by the producer and handed to
    // the MMA and epilogue warps through this ring
    uint64_t tq_full[4];
    uint64_t tq_empty[4];
    int tq[4];
    // kFused: the scheduler thread's one-deep queue to the producer (a tile
    // claimed and resolved while the previous one streams)
    uint64_t sq_full;
    uint64_t sq_empty;
    int sq_tile;
    int sq_rows;
    // MXFP8. A stage is taken by dequant set p = (stage number) % 2 and MMA
    // issuer j = (index in its tile) % 2, and uses code slot (stage number) %
    // kF8Stages and A buffer (stage number) % kF8Dq. Every barrier below has
    // one consumer, which waits all its completions in order (phase bits per
    // slot), so no parity wait can run a phase ahead: a slot's next use for
    // that consumer is armed only after the slot passed through it.
    uint64_t fullD[2][kF8Stages];  // codes + scales landed, for dequant set p
    uint64_t fullB[2][kF8Stages];  // token rows landed, for issuer j
    uint64_t dq_full[2][kF8Dq];    // A buffer written, for issuer j (the four warps of a set)
    uint64_t dq_empty[2][kF8Dq];   // A buffer read by the MMAs, for the set that writes it next
};

constexpr int kSmemBytes = kStages * kStageBytes + (int)sizeof(Ctl) + 1024;
constexpr int kF8SmemBytes = kF8CtlOff + (int)sizeof(Ctl) + 1024;
static_assert(kF8SmemBytes <= 227 * 1024, "MXFP8 ring exceeds the shared memory of a CTA");

struct SmallParams {
    TcGemmArgs g1;     // SwiGLU tiles (unused in kDownOnly)
    TcGemmArgs g2;     // down tiles (unused in kSwiGLUOnly)
    int* done;         // kFused: [E] finished SwiGLU tiles, [E] finished down tiles, [1] next
                       // tile to hand out, [E] gathered rows, [1] next finalize item;
                       // zero at launch
    FinalizeArgs fin;  // kFused: the finalize run after the tiles (fin.y null = none)
    // kFused: the gather xp[i] = x[perm[i] / k] run at the start (x null = none)
    const void* gx;
    void* gxp;
    const int32_t* gperm;
    int gk;
    int grow_bytes;
    // MXFP8: token rows per 64-K tile that the loads fill (8 when the batch has
    // at most 8 tokens, as no expert then owns more routes; else 16). The MMA
    // still reads 16 rows: rows past the loaded ones only feed output columns
    // that the epilogue drops.
    int brows;
};

// With MXFP8 weights every stage is three TMA instructions (the producer
// thread's issue rate bounds the stream otherwise): the gate and up rows of a
// SwiGLU stage come as one 3D box, so do their scales, and so do the two 64-K
// token-row tiles.
struct SmallMaps {
    CUtensorMap x1;      // SwiGLU token rows [R][H], box {64, 16} (MXFP8: 3D {64, R, H/64}, box {64, 16, 2})
    CUtensorMap x2;      // down token rows (h) [R][M*I], box {64, 16} (MXFP8: 3D as x1)
    CUtensorMap w1[kMaxMicro];  // w13[m] 3D {H, I, 2E}, box {64, 64, 2} (MXFP8: uint8 codes, box {128, 64, 2})
    CUtensorMap w2[kMaxMicro];  // w2[m] [E*H][I], box {64, 128} (MXFP8: uint8 codes, box {128, 128})
    CUtensorMap s1[kMaxMicro];  // MXFP8: w13[m] scales 3D {I, 2, E*H/32}, box {64, 2, 4}: [4][gate, up][64]
    CUtensorMap s2[kMaxMicro];  // MXFP8: w2[m] scales [E*I/32][H] uint8, box {128, 4}: [4][128]
};

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void fail(Ctl& c, int* err) {
    c.abort = 1;
    atomicOr(err, kErrTimeout);
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Expert whose segment [seg[g], seg[g+1]) holds sorted position pos.
__device__ __forceinline__ int expert_of(const int* seg, int G, int pos) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg[mid] <= pos)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Eight bf16 to eight f16 (nearest, ties to even).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The gather xp[i] = x[perm[i] / k] (blog section 6.1: index_select once), as
// the fused kernel's first phase, run by the four epilogue warps: CTA b <
// kGatherCtas copies rows b, b + kGatherCtas, ... and counts each finished row
// for its expert, so a SwiGLU tile only waits for the rows of its own expert.
// With MXFP8 weights the rows are written as f16.
template <bool F8>
__device__ __forceinline__ void gather_rows(const Ctl& c, const SmallParams& p) {
    const int tid = threadIdx.x - 128;
    const int R = c.seg[p.g1.G];
    const int nvec = p.grow_bytes / 16;
    const uint4* __restrict__ src = static_cast<const uint4*>(p.gx);
    uint4* __restrict__ dst = static_cast<uint4*>(p.gxp);
    const int gctas = (int)gridDim.x < kGatherCtas ? (int)gridDim.x : kGatherCtas;
    for (int i = blockIdx.x; i < R; i += gctas) {
        const int64_t tok = p.gperm[i] / p.gk;
        constexpr int kBatch = 8;
        for (int v0 = tid; v0 < nvec; v0 += 128 * kBatch) {
            uint4 buf[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (v0 + u * 128 < nvec) buf[u] = src[tok * nvec + v0 + u * 128];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (v0 + u * 128 < nvec) dst[(int64_t)i * nvec + v0 + u * 128] = F8 ? bf16x8_to_f16x8(buf[u]) : buf[u];
        }
        fence_proxy_async_global();  // the rows are read next by TMA (async proxy)
        epilogue_bar();
        if (tid == 0) {
            __threadfence();
            atomicAdd(p.done + 2 * p.g1.G + 1 + expert_of(c.seg, p.g1.G, i), 1);
        }
    }
}

// The finalize ("HunyuanImage3 Hybrid Parallelism", section 6.1: routing scale
// applied once, top-k reduced once) as the fused kernel's last phase, run by
// the four epilogue warps once their CTA has no tiles left: items are taken
// from a global counter, and item (token t, 1024 columns) waits until the down
// tiles of t's k experts have stored their o rows, then
//     y[t] = sum_j w[t][j] * o[inv[t*k + j]] (+ shared[t]) (+ y[t] when
//     accumulating), fp32 accumulate.
// o rows come from other CTAs, so they are read through L2 (ld.global.cg).
__device__ __forceinline__ void finalize_items(Ctl& c, const SmallParams& p) {
    const FinalizeArgs& f = p.fin;
    const int tid = threadIdx.x - 128;  // 0..127: the epilogue warps
    const int G = p.g1.G;
    const int target = p.g2.n_tiles;    // down tiles per expert (one row block each)
    const int nvec = f.H / 8;
    const int chunks = (nvec + 127) / 128;
    const int items = f.T * chunks;
    const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(f.o);
    const __nv_bfloat16* sh = static_cast<const __nv_bfloat16*>(f.shared);
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(f.y);
    for (;;) {
        if (tid == 0) c.fin_item = atomicAdd(p.done + 3 * G + 1, 1);
        epilogue_bar();
        const int item = c.fin_item;
        if (item >= items) break;
        const int t = item / chunks, ch = item % chunks;
        if (tid < f.k) {
            const int* cnt = p.done + G + expert_of(c.seg, G, f.inv[(int64_t)t * f.k + tid]);
            if (ld_acquire(cnt) < target) {
                const uint64_t t0 = ptx::globaltimer();
                uint32_t it = 0;
                while (ld_acquire(cnt) < target) {
                    if ((++it & 15u) == 0u && (c.abort || ptx::globaltimer() - t0 > p.g2.limit_ns)) {
                        c.fin_fail = 1;
                        fail(c, p.g2.err);
                        break;
                    }
                    __nanosleep(64);
                }
            }
        }
        epilogue_bar();
        if (c.fin_fail) break;
        const int v = ch * 128 + tid;
        if (v < nvec) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint4 u[kMaxTopK];  // all k rows in flight before the arithmetic
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                if (j < f.k)
                    u[j] = __ldcg(reinterpret_cast<const uint4*>(o + (int64_t)f.inv[(int64_t)t * f.k + j] * f.H) + v);
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                if (j < f.k) {
                    const float wj = f.w[(int64_t)t * f.k + j];
                    const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u[j]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 x2 = __bfloat1622float2(hv[i]);
                        acc[2 * i] = fmaf(wj, x2.x, acc[2 * i]);
                        acc[2 * i + 1] = fmaf(wj, x2.y, acc[2 * i + 1]);
                    }
                }
            }
            for (int extra = 0; extra < 2; ++extra) {  // shared expert, then the previous y
                const __nv_bfloat16* src = extra == 0 ? sh : (f.accumulate ? y : nullptr);
                if (src == nullptr) continue;
                const uint4 u = *(reinterpret_cast<const uint4*>(src + (int64_t)t * f.H) + v);
                const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 x2 = __bfloat1622float2(hv[i]);
                    acc[2 * i] += x2.x;
                    acc[2 * i + 1] += x2.y;
                }
            }
            uint4 out;
            __nv_bfloat162* ov = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
            for (int i = 0; i < 4; ++i) ov[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
            *(reinterpret_cast<uint4*>(y + (int64_t)t * f.H) + v) = out;
        }
        epilogue_bar();
    }
}

// Tile list position -> (is a SwiGLU tile, tile) for the given mode.
template <int MODE>
__device__ __forceinline__ Tile locate(int tile, const Ctl& c, const SmallParams& p, bool& swiglu) {
    if (MODE == kSwiGLUOnly) {
        swiglu = true;
        return decode_group_tile(tile, c.seg, c.tiles, p.g1.G, p.g1.n_tiles, p.g1.n_micro, true, kTcBM);
    }
    if (MODE == kDownOnly) {
        swiglu = false;
        return decode_group_tile(tile, c.seg, c.tiles, p.g2.G, p.g2.n_tiles, p.g2.n_micro, false, kTcBM);
    }
    const int n1 = p.g1.n_micro * c.tiles[p.g1.G] * p.g1.n_tiles;
    swiglu = tile < n1;
    return swiglu ? decode_group_tile(tile, c.seg, c.tiles, p.g1.G, p.g1.n_tiles, p.g1.n_micro, true, kTcBM)
                  : decode_group_tile(tile - n1, c.seg, c.tiles, p.g2.G, p.g2.n_tiles, p.g2.n_micro, false, kTcBM);
}

// Tile sequence of one CTA. Static modes stride over the list (blockIdx.x,
// + gridDim.x, ...). The fused mode hands tiles out dynamically: the scheduler
// thread takes the next list position from a global counter (so every position
// is taken in increasing order and CTAs that drew cheap tiles take more), the
// producer takes it from the scheduler and passes it through the shared ring
// to the MMA and epilogue warps; -1 ends.
struct TileStream {
    int slot = 0;
    uint32_t phase = 0;
    int next_static;
};

// Producer side (one thread). Returns the tile to process, or -1 when done or failed.
// In the fused mode `t` is the tile taken from the scheduler (-1 to end).
template <int MODE>
__device__ __forceinline__ int produce_tile(Ctl& c, TileStream& ts, int total, int t, uint64_t limit_ns,
                                            bool& ok) {
    if (MODE != kFused) {
        const int ts_t = ts.next_static;
        ts.next_static += gridDim.x;
        return ts_t < total ? ts_t : -1;
    }
    if (!ptx::mbar_wait(ptx::smem_u32(&c.tq_empty[ts.slot]), ts.phase ^ 1u, limit_ns, &c.abort)) {
        ok = false;
        t = -1;
    }
    c.tq[ts.slot] = t;
    ptx::mbar_arrive(ptx::smem_u32(&c.tq_full[ts.slot]));
    if (++ts.slot == 4) {
        ts.slot = 0;
        ts.phase ^= 1u;
    }
    return t;
}

// Consumer side (one thread per consuming warp). Returns -1 when done or failed.
template <int MODE>
__device__ __forceinline__ int consume_tile(Ctl& c, TileStream& ts, int total, uint64_t limit_ns) {
    if (MODE != kFused) {
        const int t = ts.next_static;
        ts.next_static += gridDim.x;
        return t < total ? t : -1;
    }
    int t = -1;
    if (ptx::mbar_wait(ptx::smem_u32(&c.tq_full[ts.slot]), ts.phase, limit_ns, &c.abort)) t = c.tq[ts.slot];
    ptx::mbar_arrive(ptx::smem_u32(&c.tq_empty[ts.slot]));
    if (++ts.slot == 4) {
        ts.slot = 0;
        ts.phase ^= 1u;
    }
    return t;
}

// Bounded spin until *cnt >= target (acquire); false on timeout or abort.
__device__ __forceinline__ bool wait_count(const int* cnt, int target, Ctl& c, uint64_t limit_ns) {
    if (ld_acquire(cnt) >= target) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t it = 0;
    while (ld_acquire(cnt) < target) {
        if ((++it & 15u) == 0u && (c.abort || ptx::globaltimer() - t0 > limit_ns)) return false;
        __nanosleep(64);
    }
    return true;
}

// Fused mode, scheduler thread: claims list positions one at a time (the
// first is the CTA's own index, so no claim delays the start), each only
// once the producer has taken the previous one (so a CTA holds at most one
// tile beyond the one it streams), waits until a down tile's SwiGLU tiles are
// all stored, notes whether a SwiGLU tile's gathered rows are complete, and
// hands the tile to the producer; -1 ends. The acquire loads here and the
// queue's mbarrier (release on arrive, acquire on wait) make the h and x rows
// visible to the producer's thread before it issues their loads.
__device__ __forceinline__ void schedule_tiles(Ctl& c, const SmallParams& p, int total) {
    const int target = p.g1.n_micro * p.g1.n_tiles;  // SwiGLU tiles per expert
    uint32_t phase = 0;
    bool ok = true;
    for (bool first = true;; first = false) {
        if (!ptx::mbar_wait(ptx::smem_u32(&c.sq_empty), phase ^ 1u, p.g1.limit_ns, &c.abort)) ok = false;
        int t = -1, rows = 0;
        if (ok) {
            // CTA b starts with tile b; the counter hands out the rest in order
            t = first ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.done + 2 * p.g1.G, 1);
            if (t >= total) t = -1;
        }
        if (t >= 0) {
            bool sw;
            const Tile tt = locate<kFused>(t, c, p, sw);
            if (!sw) {
                if (!wait_count(p.done + tt.g, target, c, p.g2.limit_ns)) {
                    ok = false;
                    t = -1;
                }
            } else {
                rows = p.gx == nullptr || ld_acquire(p.done + 2 * p.g1.G + 1 + tt.g) >= tt.row_end - tt.row0;
            }
        }
        c.sq_tile = t;
        c.sq_rows = rows;
        ptx::mbar_arrive(ptx::smem_u32(&c.sq_full));
        phase ^= 1u;
        if (t < 0) break;
    }
    if (!ok) fail(c, p.g1.err);
}

// Fused mode, producer: the next tile from the scheduler (-1 on end or failure,
// ok cleared on failure) and whether its gathered rows were already complete.
__device__ __forceinline__ int pop_scheduled(Ctl& c, uint32_t& phase, uint64_t limit_ns, bool& rows, bool& ok) {
    int t = -1;
    rows = false;
    if (ptx::mbar_wait(ptx::smem_u32(&c.sq_full), phase, limit_ns, &c.abort)) {
        t = c.sq_tile;
        rows = c.sq_rows != 0;
    } else {
        ok = false;
    }
    ptx::mbar_arrive(ptx::smem_u32(&c.sq_empty));
    phase ^= 1u;
    return t;
}

// Sixteen E4M3 codes (in K order) under the E8M0 scale S to sixteen f16: the
// f16 rounding of code * 2^(S-127).
// Fast form, for scales that are f16 numbers (2^-24 .. 2^15, dequant_in_f16
// true): one f16 multiply per pair of exact operands, branch-free.
__device__ __forceinline__ bool dequant_in_f16(int S) { return S >= 127 - 24 && S <= 127 + 15; }

__device__ __forceinline__ void dequant16_f16(uint4 q, int S, uint32_t* o) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    const int e = S - 127;
    const unsigned short hb = e >= -14 ? (unsigned short)((e + 15) << 10) : (unsigned short)(1u << ((e + 24) & 15));
    const __half2 sc = __halves2half2(__ushort_as_half(hb), __ushort_as_half(hb));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h[2];
        ptx::e4m3x4_to_f16x2x2(w[i], h[0], h[1]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&h[j]), sc);
            o[2 * i + j] = *reinterpret_cast<const uint32_t*>(&r);
        }
    }
}

// Any scale: through fp32, where the product is exact, rounded once to f16.
__device__ __forceinline__ void dequant16_f32(uint4 q, int S, uint32_t* o) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    const int e = S - 127;
    const float fs = e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h[2];
        ptx::e4m3x4_to_f16x2x2(w[i], h[0], h[1]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
            const __half2 r = __floats2half2_rn(f.x * fs, f.y * fs);
            o[2 * i + j] = *reinterpret_cast<const uint32_t*>(&r);
        }
    }
}

template <int MODE, bool F8>
__global__ void __launch_bounds__(F8 ? kF8Threads : kThreads, 1)
    tc_small_kernel(const __grid_constant__ SmallMaps maps, const SmallParams p) {
    static_assert(!F8 || MODE == kFused, "MXFP8 weights run in the fused mode only");
    constexpr int kSt = F8 ? kF8Stages : kStages;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl& c = *reinterpret_cast<Ctl*>(smem + (F8 ? kF8CtlOff : kStages * kStageBytes));
    // stage s: the A tile (bf16 weights, or MXFP8 codes; their scales apart) and the token-row B tile
    auto stage_a = [&](int st) { return smem + (F8 ? kF8CodeOff + st * kF8CodeBytes : st * kStageBytes); };
    auto stage_s = [&](int st) { return smem + kF8ScaleOff + st * kF8ScaleBytes; };
    auto stage_b = [&](int st) { return smem + (F8 ? st * kF8BBytes : st * kStageBytes + kABytes); };
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const TcGemmArgs& a0 = MODE == kDownOnly ? p.g2 : p.g1;  // seg, tiles, G, err, limit
    // the next routing call's kernels may be placed as SMs free up; they wait
    // for this grid to complete before touching memory
    if (MODE == kFused) ptx::griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSt; ++s) {
            ptx::mbar_init(ptx::smem_u32(&c.full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&c.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&c.tfull[b]), F8 ? 2 : 1);  // the MMA issuer(s)' commits
            ptx::mbar_init(ptx::smem_u32(&c.tempty[b]), 4);
        }
        for (int q = 0; q < 2; ++q) {
            for (int b = 0; b < kF8Dq; ++b) {
                ptx::mbar_init(ptx::smem_u32(&c.dq_full[q][b]), 4);  // the four warps of a dequant set
                ptx::mbar_init(ptx::smem_u32(&c.dq_empty[q][b]), 1);  // an MMA issuer's commit
            }
            for (int st = 0; st < kF8Stages; ++st) {
                ptx::mbar_init(ptx::smem_u32(&c.fullD[q][st]), 1);  // the producer's expect_tx arrive
                ptx::mbar_init(ptx::smem_u32(&c.fullB[q][st]), 1);
            }
        }
        ptx::mbar_init(ptx::smem_u32(&c.drain), 1);
        ptx::mbar_init(ptx::smem_u32(&c.drain2), 1);
        for (int q = 0; q < 4; ++q) {
            ptx::mbar_init(ptx::smem_u32(&c.tq_full[q]), 1);
            // MMA issuer + four epilogue warps (MXFP8: two MMA issuers, four epilogue
            // and eight dequant warps)
            ptx::mbar_init(ptx::smem_u32(&c.tq_empty[q]), F8 ? 14 : 5);
        }
        ptx::mbar_init(ptx::smem_u32(&c.sq_full), 1);
        ptx::mbar_init(ptx::smem_u32(&c.sq_empty), 1);
        c.abort = 0;
        c.fin_fail = 0;
        ptx::fence_mbar_init();
    }
    if (MODE != kFused) {
        for (int i = threadIdx.x; i <= a0.G; i += blockDim.x) {
            c.seg[i] = a0.seg[i];
            c.tiles[i] = a0.tiles[i];
        }
    }
    if (warp == 0 && lane == 0) {
        if (MODE != kDownOnly) ptx::prefetch_tmap(&maps.x1);
        if (MODE != kSwiGLUOnly) ptx::prefetch_tmap(&maps.x2);
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_u32(&c.tmem_base), F8 ? kF8TmemCols : kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (MODE == kFused) {
        // started early (programmatic dependent launch): nothing the router or
        // the shared expert's GEMMs write is read before this wait
        ptx::griddep_wait();
        for (int i = threadIdx.x; i <= a0.G; i += blockDim.x) {
            c.seg[i] = a0.seg[i];
            c.tiles[i] = a0.tiles[i];
        }
        __syncthreads();
    }

    const uint32_t tmem = c.tmem_base;
    const int n1 = MODE == kDownOnly ? 0 : p.g1.n_micro * c.tiles[p.g1.G] * p.g1.n_tiles;
    const int n2 = MODE == kSwiGLUOnly ? 0 : c.tiles[p.g2.G] * p.g2.n_tiles;
    const int total = n1 + n2;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        const uint64_t wpol = ptx::policy_evict_first();  // each weight byte is read once per call
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        int gs = 0;  // stage number (MXFP8: picks the dequant set)
        // MXFP8: per slot, the barriers it armed last and their phase parities
        // (to wait out loads still in flight on failure); arm_* flip per arm
        uint32_t last_d[kSt], last_b[kSt], last_dpar = 0, last_bpar = 0, arm_d[2] = {0, 0}, arm_b[2] = {0, 0};
        bool ok = true;
        TileStream ts;
        ts.next_static = blockIdx.x;
        uint32_t sq_phase = 0;
        for (;;) {
            bool rows_seen = false;
            const int next = MODE == kFused ? pop_scheduled(c, sq_phase, a0.limit_ns, rows_seen, ok) : -1;
            const int tile = produce_tile<MODE>(c, ts, total, next, a0.limit_ns, ok);
            if (tile < 0) break;
            bool sw;
            const Tile t = locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            // kFused: a down tile comes from the scheduler only once all SwiGLU
            // tiles of its expert stored their h rows; the token rows of a SwiGLU
            // tile exist once the gather phase counted all rows of its expert
            // (until then only weights are loaded)
            const int* gcnt = (MODE == kFused && sw && p.gx != nullptr) ? p.done + 2 * p.g1.G + 1 + t.g : nullptr;
            bool rows_ready = gcnt == nullptr || rows_seen || ld_acquire(gcnt) >= t.row_end - t.row0;
            if (MODE == kFused) fence_proxy_async_global();  // the rows are read by TMA (async proxy)
            int pend_stage[kSt], pend_kb[kSt], pending = 0;
            uint32_t pend_bar[kSt];
            const int n_micro_k = sw ? 1 : g.n_micro;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = sw ? t.m : mi;
                const CUtensorMap* tw = sw ? &maps.w1[m] : &maps.w2[m];
                const CUtensorMap* tsc = sw ? &maps.s1[m] : &maps.s2[m];  // MXFP8 scales
                const CUtensorMap* tx = sw ? &maps.x1 : &maps.x2;
                const int wrow = t.g * g.b_rows_per_group + t.nt * (sw ? 64 : kM);
                constexpr int kK = F8 ? kF8K : kTcBK;                      // K per stage
                const int kbn = F8 ? f8_stages(g.k_blocks) : g.k_blocks;  // stages per micro
                // the token rows of a stage: one 64-K tile (four with MXFP8 weights)
                auto load_rows = [&](int st, int kx, uint32_t bar) {
                    const uint32_t sb = ptx::smem_u32(stage_b(st));
                    if (F8)
                        ptx::tma_load_3d(sb, tx, 0, t.row0, kx / kTcBK, bar);  // four 64-K tiles (brows rows each)
                    else
                        ptx::tma_load_2d(sb, tx, kx, t.row0, bar);
                };
                for (int kb = 0; kb < kbn; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, g.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(stage_a(stage));
                    // MXFP8: codes and scales complete the barrier of the stage's dequant
                    // set, the token rows that of its MMA issuer
                    const int dset = gs & 1, iss = (mi * kbn + kb) & 1;
                    const uint32_t fb = ptx::smem_u32(F8 ? &c.fullD[dset][stage] : &c.full[stage]);
                    const uint32_t fbb = F8 ? ptx::smem_u32(&c.fullB[iss][stage]) : fb;
                    if (F8) {
                        last_d[stage] = fb;
                        last_b[stage] = fbb;
                        last_dpar = (last_dpar & ~(1u << stage)) | (((arm_d[dset] >> stage) & 1u) << stage);
                        last_bpar = (last_bpar & ~(1u << stage)) | (((arm_b[iss] >> stage) & 1u) << stage);
                        arm_d[dset] ^= 1u << stage;
                        arm_b[iss] ^= 1u << stage;
                        ptx::mbar_arrive_expect_tx(fb, kF8CodeBytes + kF8ScaleBytes);
                        ptx::mbar_arrive_expect_tx(fbb, p.brows * 512);
                    } else {
                        ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                    }
                    ++gs;
                    if (F8) {
                        // codes: two 128-K chunks of the tile's rows; scales: the eight
                        // 32-blocks of those K (rows of the scale maps)
                        const int srow = t.g * 2 * g.k_blocks + 8 * kb;
                        const uint32_t ss = ptx::smem_u32(stage_s(stage));
                        if (sw) {
                            // per chunk: 64 gate rows, then the 64 matching up rows (half 2g + 1)
                            ptx::tma_load_4d_hint(sa, tw, 0, t.nt * 64, 2 * t.g, 2 * kb, fb, wpol);
                            ptx::tma_load_3d(ss, tsc, t.nt * 64, 0, srow, fb);
                        } else {
                            ptx::tma_load_3d_hint(sa, tw, 0, wrow, 2 * kb, fb, wpol);            // per chunk: 128 rows
                            ptx::tma_load_2d(ss, tsc, t.nt * kM, srow, fb);
                        }
                    } else if (sw) {
                        // 64 gate rows, then the 64 matching up rows (half 2g + 1 of the 3D map)
                        ptx::tma_load_3d_hint(sa, tw, kb * kTcBK, t.nt * 64, 2 * t.g, fb, wpol);
                    } else {
                        ptx::tma_load_2d_hint(sa, tw, kb * kTcBK, wrow, fb, wpol);            // 128 rows
                    }
                    const int kx = (sw ? 0 : m * g.a_micro_cols) + kb * kK;
                    if (rows_ready) {
                        load_rows(stage, kx, fbb);  // 16 token rows
                    } else {
                        pend_stage[pending] = stage;
                        pend_kb[pending] = kx;
                        pend_bar[pending] = fbb;
                        ++pending;
                    }
                    ++issued;
                    if (++stage == kSt) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (!rows_ready && (pending == kSt || kb + 1 == kbn)) {
                        // every free stage holds weights: wait for the rows, then
                        // complete the pending stages with their token rows
                        const uint64_t t0 = ptx::globaltimer();
                        uint32_t it = 0;
                        while (ld_acquire(gcnt) < t.row_end - t.row0) {
                            if ((++it & 15u) == 0u && (c.abort || ptx::globaltimer() - t0 > g.limit_ns)) {
                                ok = false;
                                break;
                            }
                            __nanosleep(32);
                        }
                        fence_proxy_async_global();
                        for (int q = 0; q < pending; ++q)  // completes the armed stages even on failure
                            load_rows(pend_stage[q], pend_kb[q], pend_bar[q]);
                        pending = 0;
                        rows_ready = true;
                        if (!ok) break;
                    }
                }
            }
            if (!ok) {
                // tell the consumers to stop: a -1 in the ring, or the abort flag
                c.abort = 1;
                if (MODE == kFused) produce_tile<MODE>(c, ts, total, -1, a0.limit_ns, ok);
                break;
            }
        }
        if (!ok) {
            fail(c, a0.err);
            const int n = issued < kSt ? issued : kSt;
            // slot s was last armed in this pass of the ring if s < stage, else in the previous one
            for (int s = 0; s < n; ++s) {
                if (F8) {
                    ptx::mbar_wait(last_d[s], (last_dpar >> s) & 1u, a0.limit_ns, nullptr);
                    ptx::mbar_wait(last_b[s], (last_bpar >> s) & 1u, a0.limit_ns, nullptr);
                } else {
                    ptx::mbar_wait(ptx::smem_u32(&c.full[s]), s < stage ? phase : phase ^ 1u, a0.limit_ns, nullptr);
                }
            }
        }
    } else if (MODE == kFused && warp == 3 && lane == 0) {
        // ------------------------------------------------ scheduler
        schedule_tiles(c, p, total);
    } else if (!F8 && warp == 1) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (waits and bookkeeping, so descriptors are
        // warp-uniform values) and one elected lane issues the tcgen05
        // instructions; lane 0 takes the tiles and broadcasts them.
        const bool issuer = ptx::elect_one();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        TileStream ts;
        ts.next_static = blockIdx.x;
        for (int local = 0; ok; ++local) {
            int tile = -1;
            if (lane == 0) tile = consume_tile<MODE>(c, ts, total, a0.limit_ns);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0) break;
            bool sw;
            locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            const bool drained = ptx::mbar_wait(ptx::smem_u32(&c.tempty[acc]), acc_par ^ 1u, g.limit_ns, &c.abort);
            if (!__all_sync(0xffffffffu, drained)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * kTok);
            uint32_t accumulate = 0;
            const int n_micro_k = sw ? 1 : g.n_micro;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                for (int kb = 0; kb < g.k_blocks; ++kb) {
                    const bool got = ptx::mbar_wait(ptx::smem_u32(&c.full[stage]), phase, g.limit_ns, &c.abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t adesc = ptx::sw128_desc(ptx::smem_u32(stage_a(stage)));
                    const uint64_t bdesc = ptx::sw128_desc(ptx::smem_u32(stage_b(stage)));
                    if (issuer) {
#pragma unroll
                        for (int k = 0; k < kTcBK / 16; ++k)
                            ptx::mma_bf16(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, accumulate | (uint32_t)k);
                        ptx::mma_commit(ptx::smem_u32(&c.empty[stage]));
                    }
                    __syncwarp();
                    accumulate = 1;
                    if (++stage == kSt) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok && issuer) ptx::mma_commit(ptx::smem_u32(&c.tfull[acc]));
            __syncwarp();
        }
        if (issuer) {
            if (!ok) fail(c, a0.err);
            ptx::mma_commit(ptx::smem_u32(&c.drain));
            ptx::mbar_wait(ptx::smem_u32(&c.drain), 0, a0.limit_ns, nullptr);
        }
        __syncwarp();
    } else if (F8 && (warp == 1 || warp == 2)) {
        // ------------------------------------------------ MXFP8 MMA issuers
        // Issuer j (warp 1 + j) takes the tile's stages of parity j into half j
        // of its accumulator; the epilogue adds the halves (half 0 + half 1,
        // the same order on every call). With N = 16 the stream rate is set by
        // how fast tcgen05 instructions are issued (eight MMAs and two commits
        // per stage), so two issuing warps raise it. Each runs as a whole warp
        // with one elected lane issuing, as the bf16 issuer above.
        const bool issuer = ptx::elect_one();
        const int j = warp - 1;
        int stage = 0, dq = 0, gs = 0;  // code slot, A buffer, stage number
        uint32_t fb_bits = 0, dq_bits = 0;  // phase bits of this issuer's fullB / dq_full barriers
        bool ok = true;
        TileStream ts;
        ts.next_static = blockIdx.x;
        for (int local = 0; ok; ++local) {
            int tile = -1;
            if (lane == 0) tile = consume_tile<MODE>(c, ts, total, a0.limit_ns);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0) break;
            bool sw;
            locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            // the accumulator is free once the epilogue read the tile two back
            // (waited for even without own stages: the commit to tfull below must
            // land in this tile's phase)
            const bool drained = ptx::mbar_wait(ptx::smem_u32(&c.tempty[acc]), acc_par ^ 1u, g.limit_ns, &c.abort);
            if (!__all_sync(0xffffffffu, drained)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * 2 * kTok + j * kTok);
            uint32_t accumulate = 0;
            const int nk = (sw ? 1 : g.n_micro) * f8_stages(g.k_blocks);
            for (int i = 0; i < nk; ++i) {
                if ((i & 1) == j) {
                    const bool got = ptx::mbar_wait(ptx::smem_u32(&c.fullB[j][stage]), (fb_bits >> stage) & 1u,
                                                    g.limit_ns, &c.abort) &&
                                     ptx::mbar_wait(ptx::smem_u32(&c.dq_full[j][dq]), (dq_bits >> dq) & 1u,
                                                    g.limit_ns, &c.abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    fb_bits ^= 1u << stage;
                    dq_bits ^= 1u << dq;
                    ptx::tc_fence_after();
                    // A buffer dq: 8 columns per 16 K; 64-K chunk h pairs with token tile h
                    const uint32_t at = tmem + (uint32_t)(kF8ACol + dq * kF8ABuf);
                    const uint32_t sb0 = ptx::smem_u32(stage_b(stage));
                    if (issuer) {
                        uint32_t acc_flag = accumulate;
#pragma unroll
                        for (int h = 0; h < kF8Chunks; ++h) {
                            // the second 64-K tile starts after the first one's brows rows
                            const uint64_t bd = ptx::sw128_desc(sb0 + h * p.brows * 128);
#pragma unroll
                            for (int k = 0; k < kTcBK / 16; ++k) {
                                ptx::mma_tmem_a(d, at + 32u * h + 8u * k, bd + 2u * k, kIdescF16, acc_flag);
                                acc_flag = 1;
                            }
                        }
                        ptx::mma_commit(ptx::smem_u32(&c.empty[stage]));  // the code slot (codes, scales, rows)
                        // the A buffer, for the dequant set that writes it next
                        ptx::mma_commit(ptx::smem_u32(&c.dq_empty[(gs + kF8Dq) & 1][dq]));
                    }
                    __syncwarp();
                    accumulate = 1;
                }
                ++gs;
                if (++stage == kSt) stage = 0;
                if (++dq == kF8Dq) dq = 0;
            }
            if (ok && issuer) ptx::mma_commit(ptx::smem_u32(&c.tfull[acc]));
            __syncwarp();
        }
        if (issuer) {
            if (!ok) fail(c, a0.err);
            uint64_t* dr = j ? &c.drain2 : &c.drain;
            ptx::mma_commit(ptx::smem_u32(dr));
            ptx::mbar_wait(ptx::smem_u32(dr), 0, a0.limit_ns, nullptr);
        }
        __syncwarp();
    } else if (F8 && warp >= 8) {
        // ------------------------------------------------ MXFP8 dequant
        // warp 8 + 4 j + q owns TMEM lanes 32 q .. 32 q + 31 (weight rows, one
        // per thread) of the stages of parity j: its thread reads the row's 128
        // codes and 4 scales, converts them in registers and stores the 64 f16
        // pairs into the row's lane of the A buffer
        const int q = warp & 3, par = (warp - 8) >> 2;
        const int r = q * 32 + lane;
        const uint32_t a_lanes = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)kF8ACol;
        int stage = 0, dq = 0, kseq = 0;  // code slot, A buffer, stage number
        uint32_t fd_bits = 0, de_bits = 0;  // phase bits of this set's fullD / dq_empty barriers
        bool ok = true;
        TileStream ts;
        ts.next_static = blockIdx.x;
        for (;;) {
            int tile = -1;
            if (lane == 0) tile = consume_tile<MODE>(c, ts, total, a0.limit_ns);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0) break;
            bool sw;
            locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            const int nk = (sw ? 1 : g.n_micro) * f8_stages(g.k_blocks);
            for (int i = 0; i < nk; ++i, ++kseq) {
                if ((kseq & 1) == par) {
                    // the buffer's first use needs no free signal; later ones wait for the
                    // MMAs of its previous use, committed to this set
                    const bool first_use = kseq < kF8Dq;
                    bool got = ptx::mbar_wait(ptx::smem_u32(&c.fullD[par][stage]), (fd_bits >> stage) & 1u,
                                              g.limit_ns, &c.abort) &&
                               (first_use || ptx::mbar_wait(ptx::smem_u32(&c.dq_empty[par][dq]), (de_bits >> dq) & 1u,
                                                            g.limit_ns, &c.abort));
                    fd_bits ^= 1u << stage;
                    if (!first_use) de_bits ^= 1u << dq;
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // the stage's two 128-K code chunks, one at a time (so only one
                    // chunk's codes and one half's f16 pairs are live)
#pragma unroll 1
                    for (int kc = 0; kc < kF8K / 128; ++kc) {
                        // 16-byte piece j of row r sits at piece j ^ (r % 8) (128-byte swizzle)
                        const unsigned char* row = stage_a(stage) + kc * (kM * 128) + r * 128;
                        uint4 cv[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            cv[j] = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
                        // scales [8][128 rows] (SwiGLU tiles: each block's 64 gate rows, then its 64 up rows)
                        const unsigned char* sp = stage_s(stage) + kc * 4 * kM;
                        int sc[4];
#pragma unroll
                        for (int b = 0; b < 4; ++b) sc[b] = sp[b * kM + r];
                        bool slow = false;
#pragma unroll
                        for (int b = 0; b < 4; ++b) slow |= !dequant_in_f16(sc[b]);
                        // two halves of 64 K (32 columns each)
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            uint32_t o[32];
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                dequant16_f16(cv[4 * hf + j], sc[2 * hf + (j >> 1)], o + 8 * j);
                            if (slow) {  // rare: scales that are not f16 numbers
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    if (!dequant_in_f16(sc[2 * hf + (j >> 1)]))
                                        dequant16_f32(cv[4 * hf + j], sc[2 * hf + (j >> 1)], o + 8 * j);
                            }
                            __syncwarp();
                            ptx::tmem_st32(a_lanes + (uint32_t)(dq * kF8ABuf + 64 * kc + 32 * hf), o);
                        }
                    }
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    __syncwarp();
                    // for the MMA issuer of the stage (its index in the tile picks it)
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&c.dq_full[i & 1][dq]));
                }
                if (++stage == kSt) stage = 0;
                if (++dq == kF8Dq) dq = 0;
            }
            if (!ok) break;
        }
        if (!ok && lane == 0) fail(c, a0.err);
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ epilogue
        const int q = warp - 4;            // TMEM lanes 32q .. 32q+31 = weight rows
        const int r = q * 32 + lane;
        if (MODE == kFused && p.gx != nullptr) gather_rows<F8>(c, p);
        TileStream ts;
        ts.next_static = blockIdx.x;
        for (int local = 0;; ++local) {
            int tile = -1;
            if (lane == 0) tile = consume_tile<MODE>(c, ts, total, a0.limit_ns);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0) break;
            bool sw;
            const Tile t = locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(g.out);
            const int acc = local & 1;
            const uint32_t acc_par = (uint32_t)(local >> 1) & 1u;
            bool ready = false;
            if (lane == 0) ready = ptx::mbar_wait(ptx::smem_u32(&c.tfull[acc]), acc_par, g.limit_ns, &c.abort);
            ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
            // the four epilogue warps meet at named barriers below, so they take
            // the continue-or-stop decision together
            if (lane == 0) c.ep_ok[q] = ready ? 1 : 0;
            epilogue_bar();
            ready = c.ep_ok[0] && c.ep_ok[1] && c.ep_ok[2] && c.ep_ok[3];
            if (!ready) {
                if (lane == 0) fail(c, a0.err);
                break;
            }
            ptx::tc_fence_after();
            uint32_t v[kTok];
            if (F8) {
                // two halves (the tile's even and odd stages); a tile of one stage
                // filled only half 0
                uint32_t v2[2 * kTok];
                ptx::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 2 * kTok), v2);
                const bool both = (sw ? 1 : g.n_micro) * f8_stages(g.k_blocks) >= 2;
#pragma unroll
                for (int jj = 0; jj < kTok; ++jj)
                    v[jj] = both ? __float_as_uint(__uint_as_float(v2[jj]) + __uint_as_float(v2[kTok + jj])) : v2[jj];
            } else {
                ptx::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kTok), v);
            }
            // the accumulator is in registers: hand it back to the MMA issuer
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&c.tempty[acc]));
            const int cnt = min(kTok, t.row_end - t.row0);
            if (sw) {
                if (q >= 2) {
#pragma unroll
                    for (int j = 0; j < kTok; ++j) c.up[r - 64][j] = __uint_as_float(v[j]);
                }
                epilogue_bar();
                if (q < 2) {
                    const int64_t col = (int64_t)t.m * g.out_micro_cols + t.nt * 64 + r;
                    for (int j = 0; j < cnt; ++j) {
                        const float h = silu(__uint_as_float(v[j])) * c.up[r][j];
                        if (F8)  // the down tiles' B operand is f16 when the weights are MXFP8
                            reinterpret_cast<__half*>(out)[(int64_t)(t.row0 + j) * g.out_ld + col] = __float2half_rn(h);
                        else
                            out[(int64_t)(t.row0 + j) * g.out_ld + col] = __float2bfloat16_rn(h);
                    }
                    if (MODE == kFused) fence_proxy_async_global();
                }
                epilogue_bar();
                if (MODE == kFused && threadIdx.x == 128) {
                    // every h store of this tile happened before the barrier above
                    __threadfence();
                    atomicAdd(p.done + t.g, 1);
                }
            } else {
                const int64_t col = (int64_t)t.nt * kM + r;
                for (int j = 0; j < cnt; ++j)
                    out[(int64_t)(t.row0 + j) * g.out_ld + col] = __float2bfloat16_rn(__uint_as_float(v[j]));
                if (MODE == kFused) {
                    epilogue_bar();
                    if (threadIdx.x == 128) {
                        __threadfence();
                        atomicAdd(p.done + p.g1.G + t.g, 1);
                    }
                }
            }
        }
        if (MODE == kFused && p.fin.y != nullptr) finalize_items(c, p);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        __syncwarp();  // lane 0 ran the second MMA issuer (MXFP8)
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, F8 ? kF8TmemCols : kTmemCols);
    }
}

template <int MODE, bool F8 = false>
cudaError_t launch_small(const SmallMaps& maps, const SmallParams& p, int max_tiles, int num_sms, cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    constexpr int smem = F8 ? kF8SmemBytes : kSmemBytes;
    constexpr int threads = F8 ? kF8Threads : kThreads;
    if (cudaError_t e = ensure_smem_limit<tc_small_kernel<MODE, F8>>(smem); e != cudaSuccess) return e;
    const int grid = max_tiles < num_sms ? max_tiles : num_sms;
    if (MODE == kFused) {
        // may start while the previous kernel in the stream still runs; the
        // kernel waits for its results (griddep_wait) after its own set-up
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, tc_small_kernel<MODE, F8>, maps, p);
    }
    tc_small_kernel<MODE, F8><<<grid, threads, smem, s>>>(maps, p);
    return cudaGetLastError();
}

void fill_maps(SmallMaps& m, const CUtensorMap& x, const CUtensorMap* w, int n_micro, bool swiglu) {
    for (int i = 0; i < kMaxMicro; ++i) {
        const CUtensorMap& src = w[i < n_micro ? i : 0];
        if (swiglu) {
            m.x1 = x;
            m.w1[i] = src;
        } else {
            m.x2 = x;
            m.w2[i] = src;
        }
    }
}

}  // namespace

cudaError_t launch_tc_small_swiglu(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW,
                                   int num_sms, cudaStream_t s) {
    SmallMaps maps{};
    fill_maps(maps, tmX, tmW, a.n_micro, true);
    fill_maps(maps, tmX, tmW, 1, false);  // unused slots
    SmallParams p{a, a, nullptr, FinalizeArgs{}, nullptr, nullptr, nullptr, 0, 0};
    return launch_small<kSwiGLUOnly>(maps, p, a.max_tiles, num_sms, s);
}

cudaError_t launch_tc_small_down(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW,
                                 int num_sms, cudaStream_t s) {
    SmallMaps maps{};
    fill_maps(maps, tmX, tmW, a.n_micro, false);
    fill_maps(maps, tmX, tmW, 1, true);  // unused slots
    SmallParams p{a, a, nullptr, FinalizeArgs{}, nullptr, nullptr, nullptr, 0, 0};
    return launch_small<kDownOnly>(maps, p, a.max_tiles, num_sms, s);
}

cudaError_t launch_tc_small_fused(const TcGemmArgs& g1, const CUtensorMap& tmX1, const CUtensorMap* tmW1,
                                  const TcGemmArgs& g2, const CUtensorMap& tmX2, const CUtensorMap* tmW2,
                                  const FinalizeArgs& fin, const GatherArgs& gat, int* done, int num_sms,
                                  cudaStream_t s) {
    SmallMaps maps{};
    fill_maps(maps, tmX1, tmW1, g1.n_micro, true);
    fill_maps(maps, tmX2, tmW2, g2.n_micro, false);
    SmallParams p{g1, g2, done, fin, gat.x, gat.xp, gat.perm, gat.k, (int)gat.row_bytes};
    return launch_small<kFused>(maps, p, g1.max_tiles + g2.max_tiles, num_sms, s);
}

cudaError_t launch_tc_small_fused_mxfp8(const TcGemmArgs& g1, const CUtensorMap& tmX1, const CUtensorMap* tmW1,
                                        const CUtensorMap* tmS1, const TcGemmArgs& g2, const CUtensorMap& tmX2,
                                        const CUtensorMap* tmW2, const CUtensorMap* tmS2, const FinalizeArgs& fin,
                                        const GatherArgs& gat, int brows, int* done, int num_sms,
                                        cudaStream_t s) {
    SmallMaps maps{};
    fill_maps(maps, tmX1, tmW1, g1.n_micro, true);
    fill_maps(maps, tmX2, tmW2, g2.n_micro, false);
    for (int i = 0; i < kMaxMicro; ++i) {
        maps.s1[i] = tmS1[i < g1.n_micro ? i : 0];
        maps.s2[i] = tmS2[i < g2.n_micro ? i : 0];
    }
    SmallParams p{g1, g2, done, fin, gat.x, gat.xp, gat.perm, gat.k, (int)gat.row_bytes, brows};
    return launch_small<kFused, true>(maps, p, g1.max_tiles + g2.max_tiles, num_sms, s);
}

}  // namespace moe
