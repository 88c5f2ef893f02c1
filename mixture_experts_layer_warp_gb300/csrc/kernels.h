// kernels.h - internal launch interfaces of the layer's kernels (not the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>

namespace moe {

// Raises the dynamic shared-memory limit of `Kernel` to `bytes` on the current
// device, once per device (the attribute is per device; a process may drive
// several GPUs). One instantiation, and so one record, per kernel.
template <auto Kernel>
inline cudaError_t ensure_smem_limit(int bytes) {
    static std::atomic<uint64_t> done{0};  // bit d: set on device d
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launches `kernel` on `s`. With `early` set, programmatic stream
// serialization: its CTAs may be placed while the previous kernel in the
// stream is still running, and the kernel executes griddepcontrol.wait (which
// returns once that grid has completed and its writes are visible) before it
// touches global memory. Without it, an ordinary launch.
template <typename... P, typename... A>
inline cudaError_t launch_kernel(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool early, A&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Bits of the device error word.
enum DeviceError : int {
    kErrTimeout = 1,  // a bounded wait ran out
    kErrCheck = 2,    // a device-side consistency check failed
};

constexpr int kMaxExperts = 64;
constexpr int kMaxTopK = 16;
constexpr int kMaxMicro = 4;

// ---------------------------------------------------------------- router
// One block routes kRouterTokens tokens (fp32 SIMT router) or kRouterTokensTc
// tokens (bf16 tensor-core router); its histogram row is blk_hist[block].
constexpr int kRouterTokens = 32;
constexpr int kRouterTokensTc = 128;
// Batches of at most kSmallTokens tokens take the small-batch kernels.
constexpr int kSmallTokens = 16;
constexpr int kRouterClusterCtas = 8;  // CTAs of the small-batch router

struct RouterArgs {
    const void* x;         // [T][H]
    const void* wr;        // [E][H]
    const float* bias;     // [E] or null
    int T, H, E, k;
    bool bf16;
    int32_t* ids;          // [T][k]
    float* w;              // [T][k]
    float* logits;         // [T][E] or null
    int32_t* blk_hist;     // [NB][E]
    int* err;
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);

struct RouterTcArgs {
    const float* bias;      // [E] or null
    int T, H, E, k;
    int32_t* ids;           // [T][k]
    float* w;               // [T][k]
    float* logits;          // [T][E] or null
    int32_t* blk_hist;      // [NB][E] (written when more than one CTA)
    // written only when a single CTA covers all T tokens:
    int32_t* offsets;       // [E+1]
    int32_t* tiles_tc;      // [E+1]
    int32_t* tiles_simt;    // [E+1]
    int32_t* shared_seg;    // [2]
    int32_t* shared_tiles_tc;    // [2]
    int32_t* shared_tiles_simt;  // [2]
    int32_t* perm;          // [T*k]
    int32_t* inv;           // [T*k]
    int32_t* zero_counters; // [zero_count] set to 0 by the single-CTA paths, or null
    int zero_count;
    int* err;
    uint64_t limit_ns;
};
// tmX: x [T][H] bf16, box {64, 128}; tmW: Wr [E][H] bf16, box {64, 64}.
cudaError_t launch_router_tc(const RouterTcArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                             cudaStream_t s);
// Mid-size batches: 4-CTA clusters per 128 tokens splitting K (tmX box {64, 128});
// same logits and the same 128-token block histograms as launch_router_tc.
cudaError_t launch_router_tc_split(const RouterTcArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                                   cudaStream_t s);
// T <= kSmallTokens: one 8-CTA cluster; tmX box {64, 16}. Same logits bit for bit.
cudaError_t launch_router_tc_small(const RouterTcArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                                   cudaStream_t s);

// --------------------------------------------------------- scan / place
struct ScanArgs {
    const int32_t* blk_hist;  // [NB][E]
    int NB, E, T, k;
    int32_t* blk_base;        // [NB][E] first sorted position of block b's expert-e routes
    int32_t* offsets;         // [E+1]
    int32_t* tiles_tc;        // [E+1] prefix of ceil(count/kTcBM)
    int32_t* tiles_simt;      // [E+1] prefix of ceil(count/kSimtBM)
    int32_t* shared_seg;      // [2] = {0, T}
    int32_t* shared_tiles_tc;   // [2] = {0, ceil(T/kTcBM)}
    int32_t* shared_tiles_simt; // [2] = {0, ceil(T/kSimtBM)}
};
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s);

struct PlaceArgs {
    const int32_t* ids;       // [T][k]
    const int32_t* blk_base;  // [NB][E]
    int T, k, E, NB;
    int tok_per_blk;          // tokens per histogram block (router block size)
    int32_t* perm;            // [T*k]
    int32_t* inv;             // [T*k]
    int* err;
};
cudaError_t launch_place(const PlaceArgs& a, cudaStream_t s);
// Both in one launch when NB * E <= kScanPlaceMaxInts (each block reads every
// histogram row to find its own bases).
constexpr int kScanPlaceMaxInts = 16384;
cudaError_t launch_scan_place(const ScanArgs& sa, const PlaceArgs& a, cudaStream_t s);

struct GatherArgs {
    const void* x;            // [T][row_bytes]
    const int32_t* perm;      // [R]
    int R, k;
    uint32_t row_bytes;       // multiple of 16
    void* xp;                 // [R][row_bytes]
    int* err;
    uint64_t limit_ns;
    int num_sms;
    const int32_t* inv;       // [R] inverse of perm (launch_gather)
    int early;                // launch while the previous kernel in the stream finishes
};
// xp[inv[t*k + j]] = x[t] for every token t and slot j: each row of x is read
// once and written to its k routes' positions.
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s);

// ------------------------------------------------------------ finalize
struct FinalizeArgs {
    const void* o;            // [R][H] expert outputs (bf16 or f32)
    const int32_t* inv;       // [R]
    const float* w;           // [T][k]
    const void* shared;       // [T][H] or null
    int T, k, H;
    bool bf16;
    void* y;                  // [T][H]
    bool accumulate;          // y += result instead of y = result
    int early;                // launch while the previous kernel in the stream finishes
    int* err;                 // device error word: kErrCheck for an inverse entry outside [0, R), or null
};
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s);

// ------------------------------------------------------- tcgen05 GEMMs
constexpr int kTcBM = 128;   // rows per tile (MMA M)
constexpr int kTcBK = 64;    // K per stage: 64 bf16 = one 128-byte swizzled row

// Grouped GEMM over row segments [seg[g], seg[g+1]) of A, one weight block per group.
//   SwiGLU form (GEMM1): out[r][m*I + n] = silu(A_r . B_m[g][n]) * (A_r . B_m[g][I + n])
//   Plain form (GEMM2):  out[r][n] = sum_m A_r[m*I:(m+1)*I] . B_m[g][n]
struct TcGemmArgs {
    const int32_t* seg;       // [G+1] row offsets, or null: one dense segment [0, dense_rows) (G = 1)
    const int32_t* tiles;     // [G+1] prefix of ceil(rows/kTcBM) (unused when seg is null)
    int G;
    int n_micro;
    int k_blocks;             // kTcBK-blocks of K per micro
    int n_tiles;              // output column tiles per (group, micro)
    int b_rows_per_group;     // rows of B per group (2I for GEMM1, H for GEMM2)
    int up_offset;            // GEMM1: I (row offset of the up rows)
    int a_micro_cols;         // GEMM2: A columns per micro (I)
    void* out;                // bf16
    int64_t out_ld;           // elements per output row
    int out_micro_cols;       // GEMM1: I (column offset of micro m in out)
    int max_tiles;            // upper bound used for the grid
    int* err;
    uint64_t limit_ns;
    int dense_rows;           // rows of the dense segment when seg is null
    int early;                // launch while the previous kernel in the stream finishes
};
// Grouped GEMMs on CTA pairs (gemm_pair.cu): weights on the MMA's M side (256
// rows over the pair), the routes of a group on N in chunks of at most 256,
// padded to a multiple of 16.
//   SwiGLU form (GEMM1): out[r][m*I + n] = silu(x_r . W_m[g][n]) * (x_r . W_m[g][I + n])
//   Plain form (GEMM2):  out[r][n] = sum_m x_r[m*I:(m+1)*I] . W_m[g][n]
struct PairGemmArgs {
    const int32_t* seg;       // [G+1] route-row offsets of the groups, or null: one dense segment [0, dense_rows)
    int G;
    int n_micro;
    int k_blocks;             // K stages per micro: 64 K (bf16 operands) or 128 K (MXFP8 codes)
    int n_ftiles;             // feature tiles per (group, micro): I/128 (SwiGLU) or H/256 (plain)
    int w_rows_per_group;     // plain form: rows of W per group (H)
    int x_micro_cols;         // plain form: columns of the token rows per micro (I)
    void* out;                // bf16 (MXFP8 SwiGLU form: the E4M3 codes of h, one byte each)
    int64_t out_ld;           // elements per output row
    int out_micro_cols;       // SwiGLU form: I (column offset of micro m in out)
    int max_tiles;            // upper bound on the tiles (sizes the grid)
    int* err;
    uint64_t limit_ns;
    int dense_rows;           // rows of the dense segment when seg is null
    int early;                // launch while the previous kernel in the stream finishes
    // MXFP8 SwiGLU form: h leaves the epilogue as MXFP8 (each 32 features of a
    // row one block, from the bf16-rounded values): codes in `out`, scale
    // bytes stage-major [out_ld/128][out_rows_pad][4] here (launch_gather_mx
    // layout), ready for the block-scaled down GEMM.
    void* out_scales;
    int64_t out_rows_pad;
    int chunk_block;          // chunks of a group taken together past every weight tile (0: all)
    int* sched;               // 2 ints, zero at launch (and left zero): the tile hand-out counter and
                              // the count of pairs done; one pair per stream at a time
    int dynamic;              // set by the launcher: tiles from the counter (else a static sequence)
};
// tmW[m]: SwiGLU form: w13_m [G][2I][K] as a 5D map {K, 16, 2, I/16, G} (strides
// of a row, of the up half, of 16 rows, of a group) with box {64, 16, 2, 4, 1};
// plain form: W_m [G*H][I] with box {64, 128}. tmX[0..3]: the token rows
// [rows][K] with boxes {64, 32}, {64, 64}, {64, 96}, {64, 128}. All 128B-swizzled.
cudaError_t launch_pair_gemm_swiglu(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                    cudaStream_t s);
cudaError_t launch_pair_gemm_down(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                  cudaStream_t s);
// The same GEMMs on block-scaled FP8 operands (tcgen05 kind::mxf8f6f4,
// E4M3 codes with one UE8M0 scale per 32 K of every weight row and token row;
// 128 K per stage, chunks of at most 208 routes). tmW / tmX as above over the
// uint8 codes with 128-byte boxes ({128, ...}). tmSA[m]: the weights' scales
// [G][K/32][rows] (rows innermost): SwiGLU form a 5D map {16, 2, I/16, K/32, G}
// with box {16, 2, 4, 4, 1} (the row order of the w13 box), plain form a 3D
// map {H, I/32, G} with box {128, 4, 1}. tmSB: the token rows' scale words,
// stage-major [n_micro * K/128][rows_pad][4] (launch_gather_mx layout) as a 3D
// map {16, rows_pad/4, n_micro * K/128} with box {16, 65, 1}, no swizzle.
cudaError_t launch_pair_gemm_swiglu_mx(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                       const CUtensorMap* tmSA, const CUtensorMap& tmSB, cudaStream_t s);
cudaError_t launch_pair_gemm_down_mx(const PairGemmArgs& a, const CUtensorMap* tmW, const CUtensorMap* tmX,
                                     const CUtensorMap* tmSA, const CUtensorMap& tmSB, cudaStream_t s);

// Swapped-operand variants for batches of at most kSmallTokens tokens (every
// expert then owns at most kSmallTokens routes): weights on the MMA M side,
// tokens on N. tmX: activations [rows][K], box {64, 16}; tmW[m]: weights,
// a 3D map {K, I, 2G} with box {64, 64, 2} (SwiGLU form: 64 gate rows and the
// matching up rows) or box {64, 128} (down form).
// n_tiles counts 64 h-columns (SwiGLU) or 128 output columns (down).
cudaError_t launch_tc_small_swiglu(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW,
                                   int num_sms, cudaStream_t s);
cudaError_t launch_tc_small_down(const TcGemmArgs& a, const CUtensorMap& tmX, const CUtensorMap* tmW,
                                 int num_sms, cudaStream_t s);
// Both GEMMs of the routed experts and the finalize in one persistent launch
// (programmatic dependent launch: it may start while the previous kernel in
// the stream runs and waits for it after its set-up): the down tiles of
// expert e start once the SwiGLU tiles of e have stored h, and a token's
// finalize once the down tiles of its k experts have stored o; its first phase
// gathers xp from x (gat.x non-null). done[fused_counter_ints(E)] must be zero
// at launch (the small-batch router zeroes it).
inline int fused_counter_ints(int E) { return 3 * E + 2; }
// The same with MXFP8 expert weights, on the block-scaled FP8 MMA: the token
// rows and h in MXFP8 too. tmX1 / tmX2 map the codes of the gathered rows
// (gat.xp, [R][H]) and of h (g1.out, [R][M*I]) as 3D maps {128, R, K/128}
// with box {128, 16, 2}; tmXS1 / tmXS2 their scale bytes act.xs [R][xs_pitch]
// and act.hs [M][R][hs_pitch] (pitches multiples of 16) as 3D maps {pitch, R,
// 1 or M} with box {16, 16, 1}; tmW1[m] the w13 codes as a 4D map {128, I, 2E,
// H/128} with box {128, 64, 2, 2} (per 128-K chunk: gate rows, then the
// matching up rows), tmW2[m] the w2 codes as a 3D map {128, E*H, I/128} with
// box {128, 128, 2}, tmS1[m] the w13 scales as a 3D map {I, 2, E*H/32} with box
// {64, 2, 8}, tmS2[m] the w2 scales [E*I/32][H] (box {128, 8}).
struct MxSmallActs {
    unsigned char* xs;
    int xs_pitch;
    unsigned char* hs;
    int hs_pitch;
};
cudaError_t launch_tc_small_fused_mxfp8(const TcGemmArgs& g1, const CUtensorMap& tmX1, const CUtensorMap& tmXS1,
                                        const CUtensorMap* tmW1, const CUtensorMap* tmS1, const TcGemmArgs& g2,
                                        const CUtensorMap& tmX2, const CUtensorMap& tmXS2, const CUtensorMap* tmW2,
                                        const CUtensorMap* tmS2, const FinalizeArgs& fin, const GatherArgs& gat,
                                        const MxSmallActs& act, int* done, int num_sms, cudaStream_t s);
cudaError_t launch_tc_small_fused(const TcGemmArgs& g1, const CUtensorMap& tmX1, const CUtensorMap* tmW1,
                                  const TcGemmArgs& g2, const CUtensorMap& tmX2, const CUtensorMap* tmW2,
                                  const FinalizeArgs& fin, const GatherArgs& gat, int* done, int num_sms,
                                  cudaStream_t s);

// ---------------------------------------------------- fp32 SIMT GEMMs
constexpr int kSimtBM = 32;

struct SimtGemmArgs {
    const float* a;           // [rows][lda]
    int64_t lda;
    const int32_t* seg;       // [G+1]
    const int32_t* tiles;     // [G+1] prefix of ceil(rows/kSimtBM)
    int G;
    int n_micro;
    const float* b[kMaxMicro];  // per micro: [G][b_rows][K]
    int K;                    // reduction length per micro (H for GEMM1, I for GEMM2)
    int N;                    // output columns per micro (I for GEMM1, H for GEMM2)
    int b_rows_per_group;     // 2I (GEMM1) or H (GEMM2)
    int a_micro_cols;         // GEMM2: A column offset per micro (I); GEMM1: 0
    float* out;
    int64_t out_ld;
    int out_micro_cols;       // GEMM1: I; GEMM2: 0
    int max_tiles;
};
cudaError_t launch_simt_gemm_swiglu(const SimtGemmArgs& a, cudaStream_t s);
cudaError_t launch_simt_gemm_down(const SimtGemmArgs& a, cudaStream_t s);



// ------------------------------------------------------------- routing
// The routing sequence shared by moe_route, moe_forward and moe_route_noalloc:
// bf16 layers use the tensor-core router (one launch when T <= 128, else
// router + scan + place), fp32 layers the SIMT router + scan + place.
struct RoutingJob {
    const void* x;
    const void* wr;
    const float* bias;
    int T, H, E, k;
    bool bf16;
    int32_t* ids;
    float* w;
    float* logits;            // or null
    int32_t* perm;
    int32_t* inv;
    int32_t* offsets;
    int32_t* tiles_tc;        // [E+1]
    int32_t* tiles_simt;      // [E+1]
    int32_t* shared_meta;     // [6]: shared seg[2], tiles_tc[2], tiles_simt[2]
    int32_t* blk_hist;        // [ceil(T/kRouterTokens)][E]
    int32_t* blk_base;        // same
    int* err;
    uint64_t limit_ns;
    int32_t* zero_counters;   // zeroed when routing runs in one CTA (T <= 128), or null
    int zero_count;           // ints of zero_counters
};

// Optional callbacks around every kernel launch (timing, counting).
struct LaunchHook {
    void* ctx;
    void (*before)(void* ctx, int slot, cudaStream_t s);
    void (*after)(void* ctx, int slot, cudaStream_t s, cudaError_t e);
};

enum KernelSlot { kSlotRouter = 0, kSlotScan, kSlotPlace, kSlotGather, kSlotGemm1, kSlotGemm2, kSlotSharedGemm1,
                  kSlotSharedGemm2, kSlotFinalize, kNumSlots };

// Returns cudaErrorInvalidValue if a tensor map cannot be encoded.
cudaError_t enqueue_routing(const RoutingJob& j, cudaStream_t s, const LaunchHook* hook);

// 2D bf16 tensor map over a row-major [rows][inner] matrix, box {64, box_rows},
// 128-byte swizzle: the K-major operand layout of the tcgen05 kernels.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_rows);
// uint8 map (MXFP8 codes and scales): box {box_inner bytes, box_rows}, unswizzled
// or with the 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)).
bool encode_u8_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128);
// 3D map (bf16 or uint8 elements): dims[0] innermost, strides in bytes of dims
// 1 and 2, box in elements; unswizzled or with the 128-byte swizzle.
bool encode_3d(CUtensorMap* m, bool bf16, const void* base, const uint64_t dims[3], const uint64_t strides[2],
               const uint32_t box[3], bool swizzle128);
// The same for any rank 1..5 (strides of dims 1..rank-1).
bool encode_nd(CUtensorMap* m, bool bf16, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box, bool swizzle128);
// MXFP8 activations for the block-scaled FP8 GEMMs (mx_act.cu): codes [rows][K]
// uint8, scales stage-major [K/128][rows_pad][4] (the four 32-block scales of a
// 128-element stage of a row in one 32-bit word).
struct MxActArgs {
    const void* src;          // bf16: x [T][K] (gather) or the rows [rows][K]
    const int32_t* inv;       // gather: [rows] inverse permutation (route t*k+j -> its row)
    int64_t rows;             // gather: R = T*k routes; else the rows of src
    int k;                    // gather: top_k
    int K;                    // elements per row, a multiple of 128
    int64_t rows_pad;         // rows of the scale array (>= rows)
    void* codes;
    void* scales;
    int* err;
    int num_sms;
    int early;                // launch while the previous kernel in the stream finishes
};
// codes[inv[t*k + j]] = MXFP8 of x[t] for every token t and slot j (x read once)
cudaError_t launch_gather_mx(const MxActArgs& a, cudaStream_t s);
// MXFP8 quantisation (mxfp8.cu): w [groups][rows][cols] bf16 -> codes [groups][rows][cols],
// scales [groups][cols/32][rows]; cols % 32 == 0.
cudaError_t launch_mx_quantize(const void* w, int64_t groups, int rows, int cols, void* codes, void* scales,
                               int num_sms, cudaStream_t s);

// ------------------------------------------------------------ self-test
cudaError_t launch_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t s);

}  // namespace moe
