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

// MXFP8 expert weights (fused mode, moe_forward_mxfp8): the block-scaled FP8
// MMA (kind::mxf8f6f4, E4M3 x E4M3, one UE8M0 scale per 32 K on each side,
// exact products, fp32 accumulation) on the weights' codes and the MXFP8 token
// rows and h. A stage covers 256 K. Ring A holds only weight bytes: the codes
// as two 128-K chunks (128 rows of 128 contiguous bytes each, 128-byte
// swizzled; a 64-byte row halves the sustained stream rate) and their eight
// scales per row, two TMA instructions per stage from the producer thread.
// Ring B holds the 16 token rows' codes (two [16][128] chunks) and scale bytes
// of the same 256 K, loaded from L2 by a second producer thread, so the
// weight stream keeps kF8StagesA x 33 KB in flight. Four scale warps copy each
// stage's scales into tensor memory in the layout the MMA reads (per 128-K
// chunk one word per row: the A row m in lane m % 32 of every lane quarter,
// column m / 32; the B row n in lane n, column 8), and one thread issues the
// stage's eight MMAs. The gather phase writes the token rows in MXFP8 and the
// SwiGLU epilogue writes h in MXFP8 (scales [R][pitch] for the token rows,
// [micro][R][pitch] for h, pitch a multiple of 16 bytes).
constexpr int kF8StagesA = 6;
constexpr int kF8StagesB = 4;
constexpr int kF8K = 256;                            // K per stage
constexpr int kF8CodeBytes = kM * kF8K;              // 32 KB of codes: two [128 rows][128 K] chunks
constexpr int kF8ScaleBytes = kM * (kF8K / 32);      // 1 KB of scales: [8 blocks][128 rows]
constexpr int kF8SlotA = kF8CodeBytes + kF8ScaleBytes;
constexpr int kF8BCodeBytes = kTok * kF8K;           // 4 KB: two [16 rows][128 K] chunks
constexpr int kF8BScaleBytes = kTok * 16;            // [16 rows][16 scale bytes] (512 K; the stage uses 8)
constexpr int kF8SlotB = 5 * 1024;
constexpr int kF8BOff = kF8StagesA * kF8SlotA;       // ring B after ring A
constexpr int kF8CtlOff = kF8BOff + kF8StagesB * kF8SlotB;
constexpr int kF8Threads = 384;                      // warps 8..11 copy scales into tensor memory
constexpr int kF8TmemCols = 256;                     // accumulators at 0..31, scale buffers from kF8SfCol
constexpr int kF8SfCol = 32;                         // ring A slot s: 32 columns, chunk c at +16 c (SFA +0, SFB +8)
constexpr int kMaxStages = kF8StagesA > kStages ? kF8StagesA : kStages;
static_assert(kF8SlotA % 1024 == 0 && kF8SlotB % 1024 == 0 && kF8BCodeBytes + kF8BScaleBytes <= kF8SlotB,
              "128-byte swizzled tiles need 1024-byte alignment");
static_assert(kF8SfCol + kF8StagesA * 32 <= kF8TmemCols, "scale buffers exceed the TMEM allocation");

// Stages of one micro's K (k_blocks 64-K blocks) with MXFP8 weights.
__device__ __forceinline__ int f8_stages(int k_blocks) { return (k_blocks + 3) / 4; }

enum Mode { kSwiGLUOnly = 0, kDownOnly = 1, kFused = 2 };

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
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
    // MXFP8: ring B (token rows) and the scale warps' signal per ring A slot
    uint64_t fullB[kF8StagesB];
    uint64_t emptyB[kF8StagesB];
    uint64_t sf_full[kF8StagesA];
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
    // MXFP8: the gathered rows' scale bytes [R][xs_pitch] (their codes at gxp,
    // [R][H]), and h's [n_micro][R][hs_pitch] (its codes at g1.out, [R][n_micro*I])
    unsigned char* xs;
    int xs_pitch;
    unsigned char* hs;
    int hs_pitch;
};

struct SmallMaps {
    CUtensorMap x1;      // SwiGLU token rows [R][H], box {64, 16} (MXFP8: codes as 3D {128, R, H/128}, box {128, 16, 2})
    CUtensorMap x2;      // down token rows (h) [R][M*I], box {64, 16} (MXFP8: codes, 3D as x1)
    CUtensorMap w1[kMaxMicro];  // w13[m] 3D {H, I, 2E}, box {64, 64, 2} (MXFP8: codes 4D {128, I, 2E, H/128}, box {128, 64, 2, 2})
    CUtensorMap w2[kMaxMicro];  // w2[m] [E*H][I], box {64, 128} (MXFP8: codes 3D {128, E*H, I/128}, box {128, 128, 2})
    CUtensorMap s1[kMaxMicro];  // MXFP8: w13[m] scales 3D {I, 2, E*H/32}, box {64, 2, 8}: [8][gate, up][64]
    CUtensorMap s2[kMaxMicro];  // MXFP8: w2[m] scales [E*I/32][H] uint8, box {128, 8}: [8][128]
    CUtensorMap xs1;     // MXFP8: token rows' scales 3D {xs_pitch, R, 1}, box {16, 16, 1}
    CUtensorMap xs2;     // MXFP8: h's scales 3D {hs_pitch, R, n_micro}, box {16, 16, 1}
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

// The gather xp[i] = x[perm[i] / k] (blog section 6.1: index_select once), as
// the fused kernel's first phase, run by the four epilogue warps: CTA b <
// kGatherCtas copies rows b, b + kGatherCtas, ... and counts each finished row
// for its expert, so a SwiGLU tile only waits for the rows of its own expert.
// With MXFP8 weights each row is written in MXFP8: its codes (one byte per
// element) and its scale bytes (per 32-block; the row's pitch past H/32 zero),
// warp q taking the 128-element stages q, q + 4, ...
template <bool F8>
__device__ __forceinline__ void gather_rows(const Ctl& c, const SmallParams& p) {
    const int tid = threadIdx.x - 128;
    const int R = c.seg[p.g1.G];
    const int nvec = p.grow_bytes / 16;
    const int gctas = (int)gridDim.x < kGatherCtas ? (int)gridDim.x : kGatherCtas;
    for (int i = blockIdx.x; i < R; i += gctas) {
        const int64_t tok = p.gperm[i] / p.gk;
        if (F8) {
            const int lane = tid & 31, q = tid >> 5;
            const int H = p.grow_bytes / 2, stages = H / 128;
            const uint2* __restrict__ src = static_cast<const uint2*>(p.gx) + tok * (H / 4);
            uint32_t* __restrict__ codes = static_cast<uint32_t*>(p.gxp) + (int64_t)i * (H / 4);
            uint32_t* __restrict__ words = reinterpret_cast<uint32_t*>(p.xs + (int64_t)i * p.xs_pitch);
            constexpr int kBatch = 8;
            for (int s0 = q; s0 < stages; s0 += 4 * kBatch) {
                uint2 raw[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (s0 + 4 * u < stages) raw[u] = src[(s0 + 4 * u) * 32 + lane];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int st = s0 + 4 * u;
                    if (st < stages) {  // warp-uniform
                        uint32_t word;
                        codes[st * 32 + lane] = mx_quantize128(raw[u], lane, word);
                        if (lane == 0) words[st] = word;
                    }
                }
            }
            for (int w = stages + tid; w < p.xs_pitch / 4; w += 128) words[w] = 0u;
        } else {
            const uint4* __restrict__ src = static_cast<const uint4*>(p.gx);
            uint4* __restrict__ dst = static_cast<uint4*>(p.gxp);
            constexpr int kBatch = 8;
            for (int v0 = tid; v0 < nvec; v0 += 128 * kBatch) {
                uint4 buf[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (v0 + u * 128 < nvec) buf[u] = src[tok * nvec + v0 + u * 128];
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (v0 + u * 128 < nvec) dst[(int64_t)i * nvec + v0 + u * 128] = buf[u];
            }
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

template <int MODE, bool F8>
__global__ void __launch_bounds__(F8 ? kF8Threads : kThreads, 1)
    tc_small_kernel(const __grid_constant__ SmallMaps maps, const SmallParams p) {
    static_assert(!F8 || MODE == kFused, "MXFP8 weights run in the fused mode only");
    constexpr int kSt = F8 ? kF8StagesA : kStages;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl& c = *reinterpret_cast<Ctl*>(smem + (F8 ? kF8CtlOff : kStages * kStageBytes));
    // stage s: the A tile (bf16 weights; MXFP8: codes, then their scales) and
    // the token-row B tile (MXFP8: slot s of ring B, codes then scale bytes)
    auto stage_a = [&](int st) { return smem + (F8 ? st * kF8SlotA : st * kStageBytes); };
    auto stage_b = [&](int st) { return smem + (F8 ? kF8BOff + st * kF8SlotB : st * kStageBytes + kABytes); };
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
            ptx::mbar_init(ptx::smem_u32(&c.tfull[b]), 1);  // the MMA issuer's commit
            ptx::mbar_init(ptx::smem_u32(&c.tempty[b]), 4);
        }
        if (F8) {
            for (int st = 0; st < kF8StagesB; ++st) {
                ptx::mbar_init(ptx::smem_u32(&c.fullB[st]), 1);   // the row producer's expect_tx arrive
                ptx::mbar_init(ptx::smem_u32(&c.emptyB[st]), 1);  // the MMA issuer's commit
            }
            for (int st = 0; st < kF8StagesA; ++st) ptx::mbar_init(ptx::smem_u32(&c.sf_full[st]), 4);  // scale warps
        }
        ptx::mbar_init(ptx::smem_u32(&c.drain), 1);
        for (int q = 0; q < 4; ++q) {
            ptx::mbar_init(ptx::smem_u32(&c.tq_full[q]), 1);
            // MMA issuer + four epilogue warps (MXFP8: also the row producer and
            // the four scale warps)
            ptx::mbar_init(ptx::smem_u32(&c.tq_empty[q]), F8 ? 10 : 5);
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

    if (!F8 && warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        const uint64_t wpol = ptx::policy_evict_first();  // each weight byte is read once per call
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
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
            const int n_micro_k = sw ? 1 : g.n_micro;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = sw ? t.m : mi;
                const CUtensorMap* tw = sw ? &maps.w1[m] : &maps.w2[m];
                const CUtensorMap* tx = sw ? &maps.x1 : &maps.x2;
                const int wrow = t.g * g.b_rows_per_group + t.nt * kM;
                for (int kb = 0; kb < g.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, g.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(stage_a(stage));
                    const uint32_t fb = ptx::smem_u32(&c.full[stage]);
                    ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                    if (sw)  // 64 gate rows, then the 64 matching up rows (half 2g + 1 of the 3D map)
                        ptx::tma_load_3d_hint(sa, tw, kb * kTcBK, t.nt * 64, 2 * t.g, fb, wpol);
                    else
                        ptx::tma_load_2d_hint(sa, tw, kb * kTcBK, wrow, fb, wpol);  // 128 rows
                    const int kx = (sw ? 0 : m * g.a_micro_cols) + kb * kTcBK;
                    if (rows_ready) {
                        ptx::tma_load_2d(ptx::smem_u32(stage_b(stage)), tx, kx, t.row0, fb);  // 16 token rows
                    } else {
                        pend_stage[pending] = stage;
                        pend_kb[pending] = kx;
                        ++pending;
                    }
                    ++issued;
                    if (++stage == kSt) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (!rows_ready && (pending == kSt || kb + 1 == g.k_blocks)) {
                        // every free stage holds weights: wait for the rows, then
                        // complete the pending stages with their token rows
                        if (!wait_count(gcnt, t.row_end - t.row0, c, g.limit_ns)) ok = false;
                        fence_proxy_async_global();
                        for (int q = 0; q < pending; ++q)  // completes the armed stages even on failure
                            ptx::tma_load_2d(ptx::smem_u32(stage_b(pend_stage[q])), tx, pend_kb[q], t.row0,
                                             ptx::smem_u32(&c.full[pend_stage[q]]));
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
        if (!ok) fail(c, a0.err);
        // no load outlives the kernel, even one that an aborted MMA never took:
        // slot s was last armed in this pass of the ring if s < stage, else in
        // the previous one (a wait on a completed phase returns at once)
        const int n = issued < kSt ? issued : kSt;
        for (int s = 0; s < n; ++s)
            ptx::mbar_wait(ptx::smem_u32(&c.full[s]), s < stage ? phase : phase ^ 1u, a0.limit_ns, nullptr);
    } else if (F8 && warp == 0 && lane == 0) {
        // ------------------------------------------------ MXFP8 weight producer (ring A)
        const uint64_t wpol = ptx::policy_evict_first();  // each weight byte is read once per call
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        TileStream ts;
        uint32_t sq_phase = 0;
        for (;;) {
            bool rows_seen = false;
            const int next = pop_scheduled(c, sq_phase, a0.limit_ns, rows_seen, ok);
            const int tile = produce_tile<MODE>(c, ts, total, next, a0.limit_ns, ok);
            if (tile < 0) break;
            bool sw;
            const Tile t = locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            const int n_micro_k = sw ? 1 : g.n_micro;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = sw ? t.m : mi;
                for (int kb = 0; kb < f8_stages(g.k_blocks); ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.empty[stage]), phase ^ 1u, g.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(stage_a(stage)), ss = sa + kF8CodeBytes;
                    const uint32_t fb = ptx::smem_u32(&c.full[stage]);
                    ptx::mbar_arrive_expect_tx(fb, kF8SlotA);
                    // codes: two 128-K chunks of the tile's rows; scales: the eight
                    // 32-blocks of those K (rows of the scale maps). A half stage
                    // (K an odd multiple of 128) reads zeros or the next block's
                    // codes past the weights, which no MMA consumes.
                    const int srow = t.g * 2 * g.k_blocks + 8 * kb;
                    if (sw) {
                        // per chunk: 64 gate rows, then the 64 matching up rows (half 2g + 1)
                        ptx::tma_load_4d_hint(sa, &maps.w1[m], 0, t.nt * 64, 2 * t.g, 2 * kb, fb, wpol);
                        ptx::tma_load_3d(ss, &maps.s1[m], t.nt * 64, 0, srow, fb);
                    } else {
                        const int wrow = t.g * g.b_rows_per_group + t.nt * kM;
                        ptx::tma_load_3d_hint(sa, &maps.w2[m], 0, wrow, 2 * kb, fb, wpol);  // per chunk: 128 rows
                        ptx::tma_load_2d(ss, &maps.s2[m], t.nt * kM, srow, fb);
                    }
                    ++issued;
                    if (++stage == kSt) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                c.abort = 1;
                produce_tile<MODE>(c, ts, total, -1, a0.limit_ns, ok);
                break;
            }
        }
        if (!ok) fail(c, a0.err);
        const int n = issued < kSt ? issued : kSt;  // as the bf16 producer
        for (int s = 0; s < n; ++s)
            ptx::mbar_wait(ptx::smem_u32(&c.full[s]), s < stage ? phase : phase ^ 1u, a0.limit_ns, nullptr);
    } else if (F8 && warp == 2 && lane == 0) {
        // ------------------------------------------------ MXFP8 token-row producer (ring B)
        // Per stage the 16 rows' codes of the stage's 256 K (3D box: two 128-K
        // chunks) and their scale bytes (16 per row: the 512 K around the
        // stage, of which it uses half). A SwiGLU tile's rows are loaded once
        // the gather phase counted all rows of its expert; a down tile's h rows
        // were complete when the scheduler handed the tile out.
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        TileStream ts;
        for (;;) {
            const int tile = consume_tile<MODE>(c, ts, total, a0.limit_ns);
            if (tile < 0) break;
            bool sw;
            const Tile t = locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            if (sw && p.gx != nullptr &&
                !wait_count(p.done + 2 * p.g1.G + 1 + t.g, t.row_end - t.row0, c, g.limit_ns)) {
                ok = false;
                break;
            }
            fence_proxy_async_global();  // the rows are read by TMA (async proxy)
            const CUtensorMap* tx = sw ? &maps.x1 : &maps.x2;
            const CUtensorMap* tsx = sw ? &maps.xs1 : &maps.xs2;
            const int n_micro_k = sw ? 1 : g.n_micro;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                const int m = sw ? 0 : mi;
                for (int kb = 0; kb < f8_stages(g.k_blocks); ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(&c.emptyB[stage]), phase ^ 1u, g.limit_ns, &c.abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = ptx::smem_u32(stage_b(stage));
                    const uint32_t fb = ptx::smem_u32(&c.fullB[stage]);
                    ptx::mbar_arrive_expect_tx(fb, kF8BCodeBytes + kF8BScaleBytes);
                    const int kx = (sw ? 0 : m * g.a_micro_cols) + kb * kF8K;
                    ptx::tma_load_3d(sb, tx, 0, t.row0, kx / 128, fb);
                    ptx::tma_load_3d(sb + kF8BCodeBytes, tsx, (8 * kb) & ~15, t.row0, m, fb);
                    ++issued;
                    if (++stage == kF8StagesB) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) break;
        }
        if (!ok) fail(c, a0.err);
        const int n = issued < kF8StagesB ? issued : kF8StagesB;  // as the bf16 producer
        for (int s = 0; s < n; ++s)
            ptx::mbar_wait(ptx::smem_u32(&c.fullB[s]), s < stage ? phase : phase ^ 1u, a0.limit_ns, nullptr);
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
    } else if (F8 && warp == 1) {
        // ------------------------------------------------ MXFP8 MMA issuer
        // Per stage: the codes and weight scales (ring A), the token rows (ring
        // B) and the stage's scales in tensor memory (the scale warps, one
        // buffer per ring A slot); per 128-K chunk four MMAs of K = 32, the
        // scale byte picked by the instruction descriptor. Whole warp in the
        // loop, one elected lane issuing, as the bf16 issuer.
        const bool issuer = ptx::elect_one();
        int sa = 0, sb = 0;
        uint32_t pa = 0, pb = 0;
        bool ok = true;
        TileStream ts;
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
                const int chunks = g.k_blocks / 2;  // 128-K chunks of a micro's K
                for (int kb = 0; kb < f8_stages(g.k_blocks); ++kb) {
                    const bool got = ptx::mbar_wait(ptx::smem_u32(&c.full[sa]), pa, g.limit_ns, &c.abort) &&
                                     ptx::mbar_wait(ptx::smem_u32(&c.fullB[sb]), pb, g.limit_ns, &c.abort) &&
                                     ptx::mbar_wait(ptx::smem_u32(&c.sf_full[sa]), pa, g.limit_ns, &c.abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const int nch = chunks - 2 * kb < 2 ? chunks - 2 * kb : 2;
                    if (issuer) {
                        for (int ch = 0; ch < nch; ++ch) {
                            const uint64_t ad = ptx::sw128_desc(ptx::smem_u32(stage_a(sa)) + ch * (kM * 128));
                            const uint64_t bd = ptx::sw128_desc(ptx::smem_u32(stage_b(sb)) + ch * (kTok * 128));
                            const uint32_t sf = tmem + (uint32_t)(kF8SfCol + 32 * sa + 16 * ch);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                ptx::mma_mx(d, ad + 2u * k, bd + 2u * k, ptx::idesc_mx(kM, kTok, k, k), sf, sf + 8u,
                                            accumulate);
                                accumulate = 1;
                            }
                        }
                        ptx::mma_commit(ptx::smem_u32(&c.empty[sa]));   // codes and weight scales
                        ptx::mma_commit(ptx::smem_u32(&c.emptyB[sb]));  // token rows
                    }
                    __syncwarp();
                    accumulate = 1;
                    if (++sa == kSt) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++sb == kF8StagesB) {
                        sb = 0;
                        pb ^= 1u;
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
    } else if (F8 && warp >= 8) {
        // ------------------------------------------------ MXFP8 scale warps
        // Warp 8 + q writes lane quarter q of the stage's scale buffer (every
        // quarter holds the same words): per 128-K chunk, the weight rows'
        // words (row lane + 32 j in column j; byte i: 32-block i of the chunk)
        // and the token rows' word (row lane in column 8; lanes past 16 zero).
        const int q = warp & 3;
        int sa = 0, sb = 0;
        uint32_t pa = 0, pb = 0;
        bool ok = true;
        TileStream ts;
        for (;;) {
            int tile = -1;
            if (lane == 0) tile = consume_tile<MODE>(c, ts, total, a0.limit_ns);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0) break;
            bool sw;
            locate<MODE>(tile, c, p, sw);
            const TcGemmArgs& g = sw ? p.g1 : p.g2;
            const int n_micro_k = sw ? 1 : g.n_micro;
            for (int mi = 0; ok && mi < n_micro_k; ++mi) {
                for (int kb = 0; kb < f8_stages(g.k_blocks); ++kb) {
                    const bool got = ptx::mbar_wait(ptx::smem_u32(&c.full[sa]), pa, g.limit_ns, &c.abort) &&
                                     ptx::mbar_wait(ptx::smem_u32(&c.fullB[sb]), pb, g.limit_ns, &c.abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    // weight scales [8 blocks][128 rows]; token-row scale bytes
                    // [16 rows][16], this stage's eight at 8 * (kb & 1)
                    const unsigned char* sp = stage_a(sa) + kF8CodeBytes;
                    const unsigned char* bp = stage_b(sb) + kF8BCodeBytes + 8 * (kb & 1);
                    ptx::tc_fence_after();
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t wa[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int r = lane + 32 * j;
                            wa[j] = (uint32_t)sp[(4 * ch) * kM + r] | ((uint32_t)sp[(4 * ch + 1) * kM + r] << 8) |
                                    ((uint32_t)sp[(4 * ch + 2) * kM + r] << 16) |
                                    ((uint32_t)sp[(4 * ch + 3) * kM + r] << 24);
                        }
                        const uint32_t wb =
                            lane < kTok ? *reinterpret_cast<const uint32_t*>(bp + 16 * lane + 4 * ch) : 0u;
                        const uint32_t col =
                            tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(kF8SfCol + 32 * sa + 16 * ch);
                        ptx::tmem_st4(col, wa[0], wa[1], wa[2], wa[3]);
                        ptx::tmem_st1(col + 8u, wb);
                    }
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&c.sf_full[sa]));
                    if (++sa == kSt) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++sb == kF8StagesB) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
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
            ptx::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kTok), v);
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
                        if (F8) {
                            // h in MXFP8 for the down tiles: warp q holds the 32-block
                            // 2 nt + q of micro m's features; the block's scale from
                            // the largest |h| taken at h's bf16 value
                            const float hb = __bfloat162float(__float2bfloat16_rn(h));
                            const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hb)));
                            const int shared = mx_shared_exp(__uint_as_float(amax));
                            const int64_t row = t.row0 + j;
                            reinterpret_cast<unsigned char*>(out)[row * g.out_ld + col] =
                                (unsigned char)e4m3x2(hb * pow2f(-shared), 0.f);
                            if (lane == 0)
                                p.hs[((int64_t)t.m * c.seg[g.G] + row) * p.hs_pitch + 2 * t.nt + q] =
                                    (unsigned char)(shared + 127);
                        } else {
                            out[(int64_t)(t.row0 + j) * g.out_ld + col] = __float2bfloat16_rn(h);
                        }
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
        __syncwarp();  // lane 0 ran the token-row producer (MXFP8)
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
    SmallParams p{a, a, nullptr, FinalizeArgs{}, nullptr, nullptr, nullptr, 0, 0, nullptr, 0, nullptr, 0};
    return launch_small<kSwiGLUOnly>(maps, p, a.max_tiles, num_sms, s);
}

cudaError_t launch_tc_small_down(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW,
                                 int num_sms, cudaStream_t s) {
    SmallMaps maps{};
    fill_maps(maps, tmX, tmW, a.n_micro, false);
    fill_maps(maps, tmX, tmW, 1, true);  // unused slots
    SmallParams p{a, a, nullptr, FinalizeArgs{}, nullptr, nullptr, nullptr, 0, 0, nullptr, 0, nullptr, 0};
    return launch_small<kDownOnly>(maps, p, a.max_tiles, num_sms, s);
}

cudaError_t launch_tc_small_fused(const TcGemmArgs& g1, const CUtensorMap& tmX1, const CUtensorMap* tmW1,
                                  const TcGemmArgs& g2, const CUtensorMap& tmX2, const CUtensorMap* tmW2,
                                  const FinalizeArgs& fin, const GatherArgs& gat, int* done, int num_sms,
                                  cudaStream_t s) {
    SmallMaps maps{};
    fill_maps(maps, tmX1, tmW1, g1.n_micro, true);
    fill_maps(maps, tmX2, tmW2, g2.n_micro, false);
    SmallParams p{g1, g2, done, fin, gat.x, gat.xp, gat.perm, gat.k, (int)gat.row_bytes, nullptr, 0, nullptr, 0};
    return launch_small<kFused>(maps, p, g1.max_tiles + g2.max_tiles, num_sms, s);
}

cudaError_t launch_tc_small_fused_mxfp8(const TcGemmArgs& g1, const CUtensorMap& tmX1, const CUtensorMap& tmXS1,
                                        const CUtensorMap* tmW1, const CUtensorMap* tmS1, const TcGemmArgs& g2,
                                        const CUtensorMap& tmX2, const CUtensorMap& tmXS2, const CUtensorMap* tmW2,
                                        const CUtensorMap* tmS2, const FinalizeArgs& fin, const GatherArgs& gat,
                                        const MxSmallActs& act, int* done, int num_sms, cudaStream_t s) {
    SmallMaps maps{};
    fill_maps(maps, tmX1, tmW1, g1.n_micro, true);
    fill_maps(maps, tmX2, tmW2, g2.n_micro, false);
    for (int i = 0; i < kMaxMicro; ++i) {
        maps.s1[i] = tmS1[i < g1.n_micro ? i : 0];
        maps.s2[i] = tmS2[i < g2.n_micro ? i : 0];
    }
    maps.xs1 = tmXS1;
    maps.xs2 = tmXS2;
    SmallParams p{g1,  g2,         done,   fin,         gat.x, gat.xp, gat.perm, gat.k, (int)gat.row_bytes,
                  act.xs, act.xs_pitch, act.hs, act.hs_pitch};
    return launch_small<kFused, true>(maps, p, g1.max_tiles + g2.max_tiles, num_sms, s);
}

}  // namespace moe
