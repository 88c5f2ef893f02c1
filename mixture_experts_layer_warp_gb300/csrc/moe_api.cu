// moe_api.cu - the C ABI of include/moe.h: argument checks, the workspace,
// tensor-map encoding and the launch sequence of one layer call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/moe.h"
#include "kernels.h"

using namespace moe;

static_assert(kNumSlots == MOE_PROFILE_SLOTS, "profile slots of the C ABI");

namespace {

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

}  // namespace

struct moe_handle {
    moe_config cfg;
    int device = 0;
    int num_sms = 0;
    size_t esz = 2;
    uint64_t limit_ns = kDefaultWaitLimitNs;
    cudaStream_t last_stream = nullptr;
    bool sticky = false;
    char msg[512] = {0};
    void* ws = nullptr;
    size_t ws_bytes = 0;
    // workspace views
    int* err = nullptr;
    int32_t* ids = nullptr;
    float* topw = nullptr;
    int32_t* perm = nullptr;
    int32_t* inv = nullptr;
    int32_t* offsets = nullptr;
    int32_t* tiles_tc = nullptr;
    int32_t* tiles_simt = nullptr;
    int32_t* shared_meta = nullptr;  // shared expert: seg[2], tiles_tc[2], tiles_simt[2]
    int32_t* blk_hist = nullptr;
    int32_t* blk_base = nullptr;
    int* done = nullptr;  // counters of the fused small-batch kernel (fused_counter_ints of them)
    int* sched = nullptr;  // tile hand-out counters of the pair GEMMs: [0..1] the call's stream, [2..3] the side stream
    void* xp = nullptr;
    void* hbuf = nullptr;
    void* obuf = nullptr;
    void* hs = nullptr;
    void* sbuf = nullptr;
    void* x_stage[2] = {nullptr, nullptr};  // host-buffer calls: device staging, used alternately
    void* y_stage[2] = {nullptr, nullptr};
    // host-buffer calls: x is copied in on `in`, y out on `out` (both created on
    // the first such call); events order the reuse of each staging slot
    cudaStream_t pipe_in = nullptr, pipe_out = nullptr;
    cudaEvent_t ev_h2d[2] = {nullptr, nullptr}, ev_comp[2] = {nullptr, nullptr}, ev_d2h[2] = {nullptr, nullptr};
    int pipe_slot = 0;
    // moe_set_shared_stream: bf16 layers with a shared expert and more than
    // kSmallTokens tokens run the shared expert's GEMMs on this stream
    bool shared_stream = false;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr;
    cudaEvent_t ev_join = nullptr;
    // diagnostics
    int64_t launches = 0;
    bool accumulate = false;
    bool prof_on = false;
    int prof_max = 0;
    int prof_calls = 0;
    std::vector<cudaEvent_t> prof_ev;   // [max_calls][slots][2]
    std::vector<unsigned char> prof_used;  // [max_calls][slots]
};

namespace {

moe_status set_err(moe_handle* h, moe_status st, const char* fmt, ...) {
    if (h != nullptr) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(h->msg, sizeof h->msg, fmt, ap);
        va_end(ap);
    }
    return st;
}

moe_status cuda_err(moe_handle* h, cudaError_t e, const char* what) {
    return set_err(h, MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

moe_status check_cfg(const moe_config* c, char* msg, size_t n) {
    auto bad = [&](moe_status st, const char* why) {
        snprintf(msg, n, "%s", why);
        return st;
    };
    if (c->hidden <= 0 || c->num_experts <= 0 || c->top_k <= 0 || c->inter <= 0 || c->n_micro <= 0 ||
        c->max_tokens < 0 || c->shared_inter < 0)
        return bad(MOE_ERR_INVALID_ARG, "config sizes must be positive");
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return bad(MOE_ERR_INVALID_ARG, "dtype must be MOE_F32 or MOE_BF16");
    if (c->top_k > c->num_experts) return bad(MOE_ERR_INVALID_ARG, "top_k must not exceed num_experts");
    if (c->num_experts > kMaxExperts) return bad(MOE_ERR_UNSUPPORTED, "num_experts > 64");
    if (c->top_k > kMaxTopK) return bad(MOE_ERR_UNSUPPORTED, "top_k > 16");
    if (c->n_micro > kMaxMicro) return bad(MOE_ERR_UNSUPPORTED, "n_micro > 4");
    if ((int64_t)c->max_tokens * c->top_k >= (1ll << 31)) return bad(MOE_ERR_UNSUPPORTED, "max_tokens * top_k >= 2^31");
    if (c->dtype == MOE_BF16) {
        if (c->hidden % 256) return bad(MOE_ERR_UNSUPPORTED, "bf16 path needs hidden % 256 == 0");
        if (c->inter % 128) return bad(MOE_ERR_UNSUPPORTED, "bf16 path needs inter % 128 == 0");
        if (c->shared_inter % 128) return bad(MOE_ERR_UNSUPPORTED, "bf16 path needs shared_inter % 128 == 0");
    } else {
        if (c->hidden % 64) return bad(MOE_ERR_UNSUPPORTED, "f32 path needs hidden % 64 == 0");
        if (c->inter % 64) return bad(MOE_ERR_UNSUPPORTED, "f32 path needs inter % 64 == 0");
        if (c->shared_inter % 64) return bad(MOE_ERR_UNSUPPORTED, "f32 path needs shared_inter % 64 == 0");
        if ((int64_t)c->max_tokens * c->top_k / kSimtBM + c->num_experts >= 65535)
            return bad(MOE_ERR_UNSUPPORTED, "f32 path supports max_tokens * top_k < 2M");
    }
    return MOE_OK;
}

// The small-batch GEMMs' w13 operand, one box per K stage: w13 [G][2I][H] as a
// 3D map {H, I, 2G} whose box {64, rows, 2} is `rows` gate rows and the
// matching up rows.
bool encode_w13(CUtensorMap* m, const void* w13, uint64_t H, uint64_t I, uint64_t G, uint32_t rows) {
    const uint64_t dims[3] = {H, I, 2 * G}, strides[2] = {H * 2, I * H * 2};
    const uint32_t box[3] = {(uint32_t)kTcBK, rows, 2};
    return encode_3d(m, true, w13, dims, strides, box, true);
}

// Operands of the pair GEMMs (gemm_pair.cu). Token rows [rows][K]: four maps
// with boxes of 32, 64, 96 and 128 rows (a CTA loads the smallest one that
// covers its half of a chunk). w13 [G][2I][H] as a 5D map {H, 16, 2, I/16, G}
// whose box {64, 16, 2, 4, 1} is four groups of 16 gate rows followed by the
// matching 16 up rows; w2 [G*H][I] with 128-row boxes.
bool encode_rows_pair(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows) {
    for (uint32_t b = 0; b < 4; ++b)
        if (!encode_bf16_2d(&m[b], base, K, rows, K * 2, 32 * (b + 1))) return false;
    return true;
}
bool encode_w13_pair(CUtensorMap* m, const void* w13, uint64_t H, uint64_t I, uint64_t G) {
    const uint64_t dims[5] = {H, 16, 2, I / 16, G};
    const uint64_t strides[4] = {H * 2, I * H * 2, 16 * H * 2, 2 * I * H * 2};
    const uint32_t box[5] = {(uint32_t)kTcBK, 16, 2, 4, 1};
    return encode_nd(m, true, w13, 5, dims, strides, box, true);
}
bool encode_w2_pair(CUtensorMap* m, const void* w2, uint64_t K, uint64_t rows) {
    return encode_bf16_2d(m, w2, K, rows, K * 2, 128);
}

// Chunks of a group taken together past all its weight tiles (the pair GEMMs'
// tile order): as many as keep the block's token rows within kL2RowBytes, so
// they stay in L2 while the group's weight tiles stream past them. Measured on
// the CFG workload (full size, DRAM bytes per launch, tiles assigned
// statically): the shared expert's GEMM1 6.4 GB without blocks, 1.1 GB with
// 32 MB blocks; the routed GEMM1 (32 MB of rows per expert) 17.8 vs 16.1 GB;
// 4-16 MB blocks gave 20.5-22 GB there.
constexpr int64_t kL2RowBytes = 32ll << 20;
int chunk_block(int chunk_rows, int64_t row_bytes) {
    const int64_t b = kL2RowBytes / ((int64_t)chunk_rows * row_bytes);
    return b < 1 ? 1 : (int)(b > (1 << 20) ? (1 << 20) : b);
}

// The shared expert's two GEMMs over the dense segment [0, T) on stream `ss`
// (`early`: launched behind the preceding kernel in that stream).
moe_status run_shared_pair(moe_handle* h, const void* x, const void* sw13, const void* sw2, int32_t T,
                           cudaStream_t ss, int early);

void hook_before(void* ctx, int slot, cudaStream_t s) {
    moe_handle* h = static_cast<moe_handle*>(ctx);
    if (h->prof_on && h->prof_calls < h->prof_max)
        cudaEventRecord(h->prof_ev[2 * ((size_t)h->prof_calls * MOE_PROFILE_SLOTS + slot)], s);
}

void hook_after(void* ctx, int slot, cudaStream_t s, cudaError_t e) {
    moe_handle* h = static_cast<moe_handle*>(ctx);
    if (h->prof_on && h->prof_calls < h->prof_max) {
        const size_t i = (size_t)h->prof_calls * MOE_PROFILE_SLOTS + slot;
        cudaEventRecord(h->prof_ev[2 * i + 1], s);
        h->prof_used[i] = 1;
    }
    if (e == cudaSuccess) h->launches += 1;
}

// Runs one kernel launch between the handle's hooks (counting, optional timing).
template <typename F>
cudaError_t timed(moe_handle* h, int slot, cudaStream_t s, F&& launch) {
    hook_before(h, slot, s);
    cudaError_t e = launch();
    hook_after(h, slot, s, e);
    return e;
}

void end_call(moe_handle* h) {
    if (h->prof_on && h->prof_calls < h->prof_max) h->prof_calls += 1;
}

moe_status check_call(moe_handle* h, const void* x, const void* router_w, int32_t T) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->sticky) return set_err(h, MOE_ERR_STICKY, "handle is sticky after an earlier device error");
    if (T < 0 || T > h->cfg.max_tokens)
        return set_err(h, MOE_ERR_INVALID_ARG, "T=%d outside [0, max_tokens=%d]", T, h->cfg.max_tokens);
    if (T > 0 && (x == nullptr || router_w == nullptr))
        return set_err(h, MOE_ERR_INVALID_ARG, "x and router_w must be non-null");
    if (!aligned16(x) || !aligned16(router_w))
        return set_err(h, MOE_ERR_INVALID_ARG, "x and router_w must be 16-byte aligned");
    return MOE_OK;
}

// Router, scan and placement: leaves ids, topw, offsets, tiles, perm and inv in the workspace.
moe_status run_routing(moe_handle* h, const void* x, const void* router_w, const float* bias, int32_t T,
                       float* logits, cudaStream_t s) {
    const moe_config& c = h->cfg;
    RoutingJob j{x, router_w, bias, T, c.hidden, c.num_experts, c.top_k, c.dtype == MOE_BF16, h->ids, h->topw,
                 logits, h->perm, h->inv, h->offsets, h->tiles_tc, h->tiles_simt, h->shared_meta, h->blk_hist,
                 h->blk_base, h->err, h->limit_ns, h->done, fused_counter_ints(c.num_experts)};
    LaunchHook hook{h, hook_before, hook_after};
    cudaError_t e = enqueue_routing(j, s, &hook);
    if (e == cudaErrorInvalidValue) return set_err(h, MOE_ERR_CUDA, "router tensor map encode failed");
    if (e != cudaSuccess) return cuda_err(h, e, "routing launch");
    return MOE_OK;
}

// MXFP8 expert weights (moe_forward_mxfp8): per micro, the w13 / w2 arrays
// passed to run_forward then hold E4M3 codes and these hold the E8M0 scales.
struct MxScales {
    const void* const* w13;  // [E][H/32][2I] per micro
    const void* const* w2;   // [E][I/32][H] per micro
};

// The MXFP8 form of R rows of K elements in a workspace region: the codes
// [R][K], then (256-aligned) the stage-major scale words [K/128][rows_pad][4]
// (at most half the bytes of the region's bf16 rows).
int64_t mx_rows_pad(int64_t R) { return (R + 3) / 4 * 4; }
size_t mx_scales_off(int64_t R, int64_t K) { return round_up((size_t)(R * K), 256); }

// The routed experts of a batch of more than kSmallTokens tokens with MXFP8
// expert weights: gather and quantise the token rows to MXFP8 (one pass over
// x) into the xp region, block-scaled FP8 GEMM1 + SwiGLU whose epilogue writes
// h as MXFP8 into the h region, block-scaled FP8 GEMM2 into o.
moe_status run_routed_mx(moe_handle* h, const void* x, const void* const* w13, const void* const* w2,
                         const MxScales& mx, int32_t T, cudaStream_t s, int early_gather) {
    const moe_config& c = h->cfg;
    const int H = c.hidden, E = c.num_experts, k = c.top_k, I = c.inter, M = c.n_micro;
    const int64_t R = (int64_t)T * k, rows_pad = mx_rows_pad(R), MI = (int64_t)M * I;
    const int chunk_bound = (int)(R / 208) + E;  // bound on sum over experts of ceil(count/208)
    char* q = static_cast<char*>(h->xp);
    char* hq = static_cast<char*>(h->hbuf);
    cudaError_t e;
    CUtensorMap tmW[kMaxMicro], tmS[kMaxMicro], tmX[4], tmSB;
    auto encode_rows = [&](const char* base, int64_t K) {  // MXFP8 rows at base: codes, then scale words
        for (uint32_t b = 0; b < 4; ++b)
            if (!encode_u8_2d(&tmX[b], base, K, R, K, 128, 32 * (b + 1), true)) return false;
        const uint64_t d[3] = {16, (uint64_t)rows_pad / 4, (uint64_t)K / 128}, st[2] = {16, (uint64_t)rows_pad * 4};
        const uint32_t box[3] = {16, 65, 1};
        return encode_3d(&tmSB, false, base + mx_scales_off(R, K), d, st, box, false);
    };

    MxActArgs gx{x, h->inv, R, k, H, rows_pad, q, q + mx_scales_off(R, H), h->err, h->num_sms, early_gather};
    if ((e = timed(h, kSlotGather, s, [&] { return launch_gather_mx(gx, s); })) != cudaSuccess)
        return cuda_err(h, e, "MXFP8 gather launch");
    // GEMM1 + SwiGLU: codes of w13[m] [E][2I][H] as a 5D map {H, 16, 2, I/16, E}
    // (box: 4 groups of 16 gate rows and the matching up rows, 128 K), their
    // scales [E][H/32][2I] in the same row order
    if (!encode_rows(q, H)) return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (MXFP8 token rows)");
    for (int m = 0; m < M; ++m) {
        const uint64_t cd[5] = {(uint64_t)H, 16, 2, (uint64_t)I / 16, (uint64_t)E};
        const uint64_t cs[4] = {(uint64_t)H, (uint64_t)I * H, 16 * (uint64_t)H, 2 * (uint64_t)I * H};
        const uint32_t cb[5] = {128, 16, 2, 4, 1};
        const uint64_t sd[5] = {16, 2, (uint64_t)I / 16, (uint64_t)H / 32, (uint64_t)E};
        const uint64_t ss[4] = {(uint64_t)I, 16, 2 * (uint64_t)I, (uint64_t)H / 32 * 2 * I};
        const uint32_t sb[5] = {16, 2, 4, 4, 1};
        if (!encode_nd(&tmW[m], false, w13[m], 5, cd, cs, cb, true) ||
            !encode_nd(&tmS[m], false, mx.w13[m], 5, sd, ss, sb, false))
            return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (MXFP8 w13[%d])", m);
    }
    PairGemmArgs g1{h->offsets, E, M, H / 128, I / 128, 0, 0, hq, MI, I,
                    M * chunk_bound * (I / 128), h->err, h->limit_ns, 0, 1,  // early: behind the gather
                    hq + mx_scales_off(R, MI), rows_pad, chunk_block(208, H), h->sched};
    if ((e = timed(h, kSlotGemm1, s, [&] { return launch_pair_gemm_swiglu_mx(g1, tmW, tmX, tmS, tmSB, s); })) !=
        cudaSuccess)
        return cuda_err(h, e, "MXFP8 GEMM1 launch");
    // GEMM2: codes of w2[m] [E*H][I] (128-row boxes), scales [E][I/32][H]
    if (!encode_rows(hq, MI)) return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (MXFP8 h)");
    for (int m = 0; m < M; ++m) {
        const uint64_t sd[3] = {(uint64_t)H, (uint64_t)I / 32, (uint64_t)E}, ss[2] = {(uint64_t)H, (uint64_t)I / 32 * H};
        const uint32_t sb[3] = {128, 4, 1};
        if (!encode_u8_2d(&tmW[m], w2[m], I, (uint64_t)E * H, I, 128, 128, true) ||
            !encode_3d(&tmS[m], false, mx.w2[m], sd, ss, sb, false))
            return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (MXFP8 w2[%d])", m);
    }
    PairGemmArgs g2{h->offsets, E, M, I / 128, H / 256, H, I, h->obuf, (int64_t)H, 0,
                    chunk_bound * (H / 256), h->err, h->limit_ns, 0, 1,  // early: behind GEMM1
                    nullptr, 0, chunk_block(208, MI), h->sched};
    if ((e = timed(h, kSlotGemm2, s, [&] { return launch_pair_gemm_down_mx(g2, tmW, tmX, tmS, tmSB, s); })) !=
        cudaSuccess)
        return cuda_err(h, e, "MXFP8 GEMM2 launch");
    return MOE_OK;
}

moe_status run_forward(moe_handle* h, const void* x, const void* router_w, const float* bias,
                       const void* const* w13, const void* const* w2, const void* sw13, const void* sw2, int32_t T,
                       void* y, cudaStream_t s, const MxScales* mx = nullptr) {
    const moe_config& c = h->cfg;
    const int H = c.hidden, E = c.num_experts, k = c.top_k, I = c.inter, M = c.n_micro, Is = c.shared_inter;
    const int64_t R = (int64_t)T * k;
    cudaError_t e;
    const bool small_bf16 = c.dtype == MOE_BF16 && T <= kSmallTokens;
    // the shared expert depends on x only: fork it onto the side stream once
    // routing is done (its persistent CTAs would otherwise hold the SMs the
    // routing kernels need), so it overlaps the gather; join before the finalize
    const bool fork = h->shared_stream && c.dtype == MOE_BF16 && !small_bf16 && Is > 0 && T > 0;
    moe_status st = run_routing(h, x, router_w, bias, T, nullptr, s);
    if (st != MOE_OK) return st;
    if (fork && ((e = cudaEventRecord(h->ev_fork, s)) != cudaSuccess ||
                 (e = cudaStreamWaitEvent(h->side, h->ev_fork, 0)) != cudaSuccess))
        return cuda_err(h, e, "shared-expert fork");
    if (fork) {
        const cudaStream_t ss = h->side;
        if ((st = run_shared_pair(h, x, sw13, sw2, T, ss, 0)) != MOE_OK) return st;
        if ((e = cudaEventRecord(h->ev_join, ss)) != cudaSuccess) return cuda_err(h, e, "shared-expert join");
    }

    if (!small_bf16 && mx == nullptr) {  // small bf16 batches gather inside the fused GEMM launch
        // launched early behind the placement kernel (not behind the fork's event record)
        GatherArgs ga{x,      h->perm,        (int)R, k, (uint32_t)(H * h->esz), h->xp, h->err, h->limit_ns,
                      h->num_sms, h->inv, fork ? 0 : 1};
        if ((e = timed(h, kSlotGather, s, [&] { return launch_gather(ga, s); })) != cudaSuccess)
            return cuda_err(h, e, "gather launch");
    }

    if (c.dtype == MOE_BF16 && T <= kSmallTokens) {
        // swapped operands: weights on the MMA M side, the <= 16 tokens on N
        CUtensorMap tmX, tmW[kMaxMicro];
        const int active = (int)(R < E ? R : E);  // experts that can own routes
        if (!encode_bf16_2d(&tmX, h->xp, H, R, (uint64_t)H * 2, kSmallTokens))
            return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (xp)");
        for (int m = 0; m < M && mx == nullptr; ++m)
            if (!encode_w13(&tmW[m], w13[m], H, I, E, 64))
                return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (w13[%d])", m);
        TcGemmArgs g1{h->offsets, h->tiles_tc, E, M, H / kTcBK, I / 64, 2 * I, I, 0,
                      h->hbuf, (int64_t)M * I, I, active * M * (I / 64), h->err, h->limit_ns};
        CUtensorMap tmX2, tmW2[kMaxMicro];
        if (!encode_bf16_2d(&tmX2, h->hbuf, (uint64_t)M * I, R, (uint64_t)M * I * 2, kSmallTokens))
            return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (h)");
        for (int m = 0; m < M && mx == nullptr; ++m)
            if (!encode_bf16_2d(&tmW2[m], w2[m], I, (uint64_t)E * H, (uint64_t)I * 2, 128))
                return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (w2[%d])", m);
        TcGemmArgs g2{h->offsets, h->tiles_tc, E, M, I / kTcBK, H / 128, H, 0, I,
                      h->obuf, (int64_t)H, 0, active * (H / 128), h->err, h->limit_ns};
        if (Is > 0) {
            CUtensorMap sX, sW[1];
            if (!encode_bf16_2d(&sX, x, H, T, (uint64_t)H * 2, kSmallTokens) ||
                !encode_w13(&sW[0], sw13, H, Is, 1, 64))
                return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (shared GEMM1)");
            TcGemmArgs s1{h->shared_meta, h->shared_meta + 2, 1, 1, H / kTcBK, Is / 64, 2 * Is, Is, 0,
                          h->hs, (int64_t)Is, 0, Is / 64, h->err, h->limit_ns};
            if ((e = timed(h, kSlotSharedGemm1, s,
                           [&] { return launch_tc_small_swiglu(s1, sX, sW, h->num_sms, s); })) != cudaSuccess)
                return cuda_err(h, e, "shared GEMM1 launch");
            if (!encode_bf16_2d(&sX, h->hs, Is, T, (uint64_t)Is * 2, kSmallTokens) ||
                !encode_bf16_2d(&sW[0], sw2, Is, H, (uint64_t)Is * 2, 128))
                return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (shared GEMM2)");
            TcGemmArgs s2{h->shared_meta, h->shared_meta + 2, 1, 1, Is / kTcBK, H / 128, H, 0, Is,
                          h->sbuf, (int64_t)H, 0, H / 128, h->err, h->limit_ns};
            if ((e = timed(h, kSlotSharedGemm2, s,
                           [&] { return launch_tc_small_down(s2, sX, sW, h->num_sms, s); })) != cudaSuccess)
                return cuda_err(h, e, "shared GEMM2 launch");
        }
        // gather, both GEMMs and the finalize in one launch (the
        // router zeroed h->done); the shared expert's GEMMs ran first
        FinalizeArgs fin{h->obuf, h->inv, h->topw, Is > 0 ? h->sbuf : nullptr, T, k, H, true, y, h->accumulate};
        if (mx != nullptr) {
            // MXFP8: the block-scaled FP8 MMA on MXFP8 token rows and h. The
            // gather phase writes the rows' codes [R][H] at xp and their scale
            // bytes [R][xs_pitch] after them; the SwiGLU epilogue writes h's
            // codes [R][M*I] at hbuf and its scale bytes [M][R][hs_pitch] after
            // them. A 256-K stage is one box per operand: w13 codes as a 4D map
            // {128, I, 2E, H/128} (per 128-K chunk: 64 gate rows, then the
            // matching up rows), w2 codes as a 3D map {128, E*H, I/128}, their
            // scales (eight 32-blocks), the 16 token rows' codes (two 128-K
            // chunks) and their scale bytes (16 per row).
            CUtensorMap c1[kMaxMicro], c2[kMaxMicro], s1[kMaxMicro], s2[kMaxMicro], mX, mX2, mXS, mHS;
            const int xs_pitch = (int)round_up((size_t)H / 32, 16), hs_pitch = (int)round_up((size_t)I / 32, 16);
            unsigned char* xq = static_cast<unsigned char*>(h->xp);
            unsigned char* hq = static_cast<unsigned char*>(h->hbuf);
            unsigned char* xs = xq + mx_scales_off(R, H);
            unsigned char* hsc = hq + mx_scales_off(R, (int64_t)M * I);
            const uint64_t xd[3] = {128, (uint64_t)R, (uint64_t)H / 128}, xst[2] = {(uint64_t)H, 128};
            const uint64_t hd[3] = {128, (uint64_t)R, (uint64_t)M * I / 128}, hst[2] = {(uint64_t)M * I, 128};
            const uint32_t xb[3] = {128, (uint32_t)kSmallTokens, 2};
            const uint64_t xsd[3] = {(uint64_t)xs_pitch, (uint64_t)R, 1}, xss[2] = {(uint64_t)xs_pitch, (uint64_t)R * xs_pitch};
            const uint64_t hsd[3] = {(uint64_t)hs_pitch, (uint64_t)R, (uint64_t)M},
                           hss[2] = {(uint64_t)hs_pitch, (uint64_t)R * hs_pitch};
            const uint32_t sbx[3] = {16, (uint32_t)kSmallTokens, 1};
            if (!encode_3d(&mX, false, xq, xd, xst, xb, true) || !encode_3d(&mX2, false, hq, hd, hst, xb, true) ||
                !encode_3d(&mXS, false, xs, xsd, xss, sbx, false) || !encode_3d(&mHS, false, hsc, hsd, hss, sbx, false))
                return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (MXFP8 token rows)");
            const uint64_t cd[4] = {128, (uint64_t)I, 2 * (uint64_t)E, (uint64_t)H / 128};
            const uint64_t cs[3] = {(uint64_t)H, (uint64_t)I * H, 128};
            const uint32_t cb[4] = {128, 64, 2, 2};
            const uint64_t dd[3] = {128, (uint64_t)E * H, (uint64_t)I / 128}, ds[2] = {(uint64_t)I, 128};
            const uint32_t db[3] = {128, 128, 2};
            const uint64_t sd[3] = {(uint64_t)I, 2, (uint64_t)E * (H / 32)}, ss[2] = {(uint64_t)I, 2 * (uint64_t)I};
            const uint32_t sb[3] = {64, 2, 8};
            for (int m = 0; m < M; ++m)
                if (!encode_nd(&c1[m], false, w13[m], 4, cd, cs, cb, true) ||
                    !encode_nd(&c2[m], false, w2[m], 3, dd, ds, db, true) ||
                    !encode_3d(&s1[m], false, mx->w13[m], sd, ss, sb, false) ||
                    !encode_u8_2d(&s2[m], mx->w2[m], H, (uint64_t)E * (I / 32), (uint64_t)H, 128, 8, false))
                    return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (MXFP8 weights, micro %d)", m);
            if ((e = timed(h, kSlotGemm1, s, [&] {
                     GatherArgs gat{x, h->perm, (int)R, k, (uint32_t)(H * 2), xq, h->err, h->limit_ns, h->num_sms};
                     const MxSmallActs act{xs, xs_pitch, hsc, hs_pitch};
                     return launch_tc_small_fused_mxfp8(g1, mX, mXS, c1, s1, g2, mX2, mHS, c2, s2, fin, gat, act,
                                                        h->done, h->num_sms, s);
                 })) != cudaSuccess)
                return cuda_err(h, e, "fused MXFP8 GEMM launch");
            return MOE_OK;
        }
        if ((e = timed(h, kSlotGemm1, s, [&] {
                 GatherArgs gat{x, h->perm, (int)R, k, (uint32_t)(H * 2), h->xp, h->err, h->limit_ns, h->num_sms};
                 return launch_tc_small_fused(g1, tmX, tmW, g2, tmX2, tmW2, fin, gat, h->done, h->num_sms, s);
             })) != cudaSuccess)
            return cuda_err(h, e, "fused GEMM launch");
    } else if (mx != nullptr) {
        if ((st = run_routed_mx(h, x, w13, w2, *mx, T, s, fork ? 0 : 1)) != MOE_OK) return st;
        if (Is > 0 && !fork && (st = run_shared_pair(h, x, sw13, sw2, T, s, 1)) != MOE_OK) return st;
    } else if (c.dtype == MOE_BF16) {
        CUtensorMap tmW[kMaxMicro], tmX[4];
        const int chunk_bound = (int)(R / 256) + E;  // bound on sum over experts of ceil(count/256)
        // GEMM1 + SwiGLU: xp [R][H] x w13[m] [E][2I][H] -> h [R][M*I]
        if (!encode_rows_pair(tmX, h->xp, H, R)) return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (xp)");
        for (int m = 0; m < M; ++m)
            if (!encode_w13_pair(&tmW[m], w13[m], H, I, E))
                return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (w13[%d])", m);
        PairGemmArgs g1{h->offsets, E, M, H / kTcBK, I / 128, 0, 0, h->hbuf, (int64_t)M * I, I,
                        M * chunk_bound * (I / 128), h->err, h->limit_ns, 0, 1,  // early: behind the gather
                        nullptr, 0, chunk_block(256, (int64_t)H * 2), h->sched};
        if ((e = timed(h, kSlotGemm1, s, [&] { return launch_pair_gemm_swiglu(g1, tmW, tmX, s); })) != cudaSuccess)
            return cuda_err(h, e, "GEMM1 launch");
        // GEMM2: h [R][M*I] x w2[m] [E*H][I], summed over m -> o [R][H]
        if (!encode_rows_pair(tmX, h->hbuf, (uint64_t)M * I, R))
            return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (h)");
        for (int m = 0; m < M; ++m)
            if (!encode_w2_pair(&tmW[m], w2[m], I, (uint64_t)E * H))
                return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (w2[%d])", m);
        PairGemmArgs g2{h->offsets, E, M, I / kTcBK, H / 256, H, I, h->obuf, (int64_t)H, 0,
                        chunk_bound * (H / 256), h->err, h->limit_ns, 0, 1,  // early: behind GEMM1
                        nullptr, 0, chunk_block(256, (int64_t)M * I * 2), h->sched};
        if ((e = timed(h, kSlotGemm2, s, [&] { return launch_pair_gemm_down(g2, tmW, tmX, s); })) != cudaSuccess)
            return cuda_err(h, e, "GEMM2 launch");
        if (Is > 0 && !fork && (st = run_shared_pair(h, x, sw13, sw2, T, s, 1)) != MOE_OK) return st;
    } else {
        const int routed_tiles = (int)(R / kSimtBM) + E;
        SimtGemmArgs g1{};
        g1.a = static_cast<const float*>(h->xp);
        g1.lda = H;
        g1.seg = h->offsets;
        g1.tiles = h->tiles_simt;
        g1.G = E;
        g1.n_micro = M;
        for (int m = 0; m < M; ++m) g1.b[m] = static_cast<const float*>(w13[m]);
        g1.K = H;
        g1.N = I;
        g1.b_rows_per_group = 2 * I;
        g1.a_micro_cols = 0;
        g1.out = static_cast<float*>(h->hbuf);
        g1.out_ld = (int64_t)M * I;
        g1.out_micro_cols = I;
        g1.max_tiles = routed_tiles;
        if ((e = timed(h, kSlotGemm1, s, [&] { return launch_simt_gemm_swiglu(g1, s); })) != cudaSuccess) return cuda_err(h, e, "f32 GEMM1 launch");
        SimtGemmArgs g2 = g1;
        g2.a = static_cast<const float*>(h->hbuf);
        g2.lda = (int64_t)M * I;
        for (int m = 0; m < M; ++m) g2.b[m] = static_cast<const float*>(w2[m]);
        g2.K = I;
        g2.N = H;
        g2.b_rows_per_group = H;
        g2.a_micro_cols = I;
        g2.out = static_cast<float*>(h->obuf);
        g2.out_ld = H;
        g2.out_micro_cols = 0;
        if ((e = timed(h, kSlotGemm2, s, [&] { return launch_simt_gemm_down(g2, s); })) != cudaSuccess) return cuda_err(h, e, "f32 GEMM2 launch");
        if (Is > 0) {
            SimtGemmArgs s1{};
            s1.a = static_cast<const float*>(x);
            s1.lda = H;
            s1.seg = h->shared_meta;
            s1.tiles = h->shared_meta + 4;
            s1.G = 1;
            s1.n_micro = 1;
            s1.b[0] = static_cast<const float*>(sw13);
            s1.K = H;
            s1.N = Is;
            s1.b_rows_per_group = 2 * Is;
            s1.out = static_cast<float*>(h->hs);
            s1.out_ld = Is;
            s1.max_tiles = (T + kSimtBM - 1) / kSimtBM;
            if ((e = timed(h, kSlotSharedGemm1, s, [&] { return launch_simt_gemm_swiglu(s1, s); })) != cudaSuccess) return cuda_err(h, e, "f32 shared GEMM1");
            SimtGemmArgs s2 = s1;
            s2.a = static_cast<const float*>(h->hs);
            s2.lda = Is;
            s2.b[0] = static_cast<const float*>(sw2);
            s2.K = Is;
            s2.N = H;
            s2.b_rows_per_group = H;
            s2.a_micro_cols = Is;
            s2.out = static_cast<float*>(h->sbuf);
            s2.out_ld = H;
            if ((e = timed(h, kSlotSharedGemm2, s, [&] { return launch_simt_gemm_down(s2, s); })) != cudaSuccess) return cuda_err(h, e, "f32 shared GEMM2");
        }
    }
    if (fork && (e = cudaStreamWaitEvent(s, h->ev_join, 0)) != cudaSuccess) return cuda_err(h, e, "shared-expert join");
    if (!small_bf16) {  // small bf16 batches finalize inside the fused GEMM launch
        // launched early behind the last GEMM (not behind the join's event wait)
        FinalizeArgs fa{h->obuf, h->inv, h->topw, Is > 0 ? h->sbuf : nullptr, T, k, H, c.dtype == MOE_BF16, y,
                        h->accumulate, fork ? 0 : 1, h->err};
        if ((e = timed(h, kSlotFinalize, s, [&] { return launch_finalize(fa, s); })) != cudaSuccess)
            return cuda_err(h, e, "finalize launch");
    }
    return MOE_OK;
}

moe_status run_shared_pair(moe_handle* h, const void* x, const void* sw13, const void* sw2, int32_t T,
                           cudaStream_t ss, int early) {
    const int H = h->cfg.hidden, Is = h->cfg.shared_inter;
    const int chunks = (T + 255) / 256;
    int* sched = ss == h->side && ss != nullptr ? h->sched + 2 : h->sched;  // the side stream's own counters
    CUtensorMap tmW[1], tmX[4];
    cudaError_t e;
    if (!encode_rows_pair(tmX, x, H, T) || !encode_w13_pair(&tmW[0], sw13, H, Is, 1))
        return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (shared GEMM1)");
    // one dense segment of many chunks: chunk by chunk past every weight tile
    // (chunk blocks of 1), so the shared weights (50 MB at Is = 3072) stay in
    // L2 while x streams once (CFG, DRAM bytes per launch: GEMM1 1.00 -> 0.83 GB,
    // GEMM2 0.66 -> 0.47 GB against 32 MB blocks of rows)
    PairGemmArgs s1{nullptr, 1, 1, H / kTcBK, Is / 128, 0, 0, h->hs, (int64_t)Is, 0, chunks * (Is / 128), h->err,
                    h->limit_ns, T, early, nullptr, 0, 1, sched};
    if ((e = timed(h, kSlotSharedGemm1, ss, [&] { return launch_pair_gemm_swiglu(s1, tmW, tmX, ss); })) != cudaSuccess)
        return cuda_err(h, e, "shared GEMM1 launch");
    if (!encode_rows_pair(tmX, h->hs, Is, T) || !encode_w2_pair(&tmW[0], sw2, Is, H))
        return set_err(h, MOE_ERR_CUDA, "tensor map encode failed (shared GEMM2)");
    PairGemmArgs s2{nullptr, 1, 1, Is / kTcBK, H / 256, H, Is, h->sbuf, (int64_t)H, 0, chunks * (H / 256), h->err,
                    h->limit_ns, T, early, nullptr, 0, 1, sched};
    if ((e = timed(h, kSlotSharedGemm2, ss, [&] { return launch_pair_gemm_down(s2, tmW, tmX, ss); })) != cudaSuccess)
        return cuda_err(h, e, "shared GEMM2 launch");
    return MOE_OK;
}

moe_status check_weights(moe_handle* h, const void* const* w13, const void* const* w2, int32_t n_micro,
                         int32_t top_k, const void* sw13, const void* sw2, const void* y) {
    const moe_config& c = h->cfg;
    if (n_micro != c.n_micro) return set_err(h, MOE_ERR_INVALID_ARG, "n_micro=%d != config %d", n_micro, c.n_micro);
    if (top_k != c.top_k) return set_err(h, MOE_ERR_INVALID_ARG, "top_k=%d != config %d", top_k, c.top_k);
    if (w13 == nullptr || w2 == nullptr) return set_err(h, MOE_ERR_INVALID_ARG, "w13 and w2 arrays must be non-null");
    for (int m = 0; m < n_micro; ++m)
        if (w13[m] == nullptr || w2[m] == nullptr || !aligned16(w13[m]) || !aligned16(w2[m]))
            return set_err(h, MOE_ERR_INVALID_ARG, "micro %d weights null or not 16-byte aligned", m);
    const bool has_shared = c.shared_inter > 0;
    if (has_shared != (sw13 != nullptr) || has_shared != (sw2 != nullptr))
        return set_err(h, MOE_ERR_INVALID_ARG, "shared expert weights must be given iff shared_inter > 0");
    if (!aligned16(sw13) || !aligned16(sw2)) return set_err(h, MOE_ERR_INVALID_ARG, "shared weights not 16-byte aligned");
    if (y == nullptr || !aligned16(y)) return set_err(h, MOE_ERR_INVALID_ARG, "y null or not 16-byte aligned");
    return MOE_OK;
}

// Host-buffer calls (moe_forward_host and the _async entry points). Call n
// uses staging slot n % 2: x is copied in on pipe_in once the compute of call
// n-2 has read the slot (and, when y is accumulated, its copy-out of y is
// done); the layer runs on the caller's stream once the copy-in is done (and
// the slot's y was copied out); y is copied out on pipe_out once the compute is
// done. So call n+1's copy-in and call n-1's copy-out overlap call n.
moe_status ensure_pipe(moe_handle* h) {
    if (h->pipe_out != nullptr) return MOE_OK;
    bool ok = cudaStreamCreateWithFlags(&h->pipe_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h->pipe_out, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
        ok = cudaEventCreateWithFlags(&h->ev_h2d[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->ev_comp[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->ev_d2h[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return set_err(h, MOE_ERR_CUDA, "could not create the host-copy streams");
    }
    return MOE_OK;
}

template <typename Run>
moe_status host_call(moe_handle* h, const void* x_host, int32_t T, void* y_host, cudaStream_t s, Run&& run) {
    moe_status st = ensure_pipe(h);
    if (st != MOE_OK) return st;
    const int b = h->pipe_slot;
    h->pipe_slot ^= 1;
    const size_t bytes = (size_t)T * h->cfg.hidden * h->esz;
    cudaError_t e;
    if ((e = cudaStreamWaitEvent(h->pipe_in, h->ev_comp[b], 0)) != cudaSuccess ||
        (h->accumulate && (e = cudaStreamWaitEvent(h->pipe_in, h->ev_d2h[b], 0)) != cudaSuccess) ||
        (e = cudaMemcpyAsync(h->x_stage[b], x_host, bytes, cudaMemcpyHostToDevice, h->pipe_in)) != cudaSuccess ||
        (h->accumulate &&
         (e = cudaMemcpyAsync(h->y_stage[b], y_host, bytes, cudaMemcpyHostToDevice, h->pipe_in)) != cudaSuccess) ||
        (e = cudaEventRecord(h->ev_h2d[b], h->pipe_in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, h->ev_h2d[b], 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, h->ev_d2h[b], 0)) != cudaSuccess)
        return cuda_err(h, e, "copy x to device");
    st = run(h->x_stage[b], h->y_stage[b]);
    end_call(h);
    // recorded whatever run enqueued, so that the slot's next use waits for it
    if ((e = cudaEventRecord(h->ev_comp[b], s)) != cudaSuccess) return cuda_err(h, e, "record compute event");
    if (st != MOE_OK) return st;
    if ((e = cudaStreamWaitEvent(h->pipe_out, h->ev_comp[b], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(y_host, h->y_stage[b], bytes, cudaMemcpyDeviceToHost, h->pipe_out)) != cudaSuccess ||
        (e = cudaEventRecord(h->ev_d2h[b], h->pipe_out)) != cudaSuccess)
        return cuda_err(h, e, "copy y to host");
    return MOE_OK;
}

moe_status check_mxfp8(moe_handle* h, const void* const* w13_codes, const void* const* w13_scales,
                       const void* const* w2_codes, const void* const* w2_scales, int32_t n_micro, int32_t top_k,
                       const void* shared_w13, const void* shared_w2, const void* y) {
    if (h->cfg.dtype != MOE_BF16) return set_err(h, MOE_ERR_UNSUPPORTED, "MXFP8 expert weights need a bf16 layer");
    moe_status st = check_weights(h, w13_codes, w2_codes, n_micro, top_k, shared_w13, shared_w2, y);
    if (st != MOE_OK) return st;
    if (w13_scales == nullptr || w2_scales == nullptr)
        return set_err(h, MOE_ERR_INVALID_ARG, "w13 and w2 scale arrays must be non-null");
    for (int m = 0; m < n_micro; ++m)
        if (w13_scales[m] == nullptr || w2_scales[m] == nullptr || !aligned16(w13_scales[m]) ||
            !aligned16(w2_scales[m]))
            return set_err(h, MOE_ERR_INVALID_ARG, "micro %d scales null or not 16-byte aligned", m);
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_create(const moe_config* cfg, moe_handle** out) {
    if (cfg == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    char why[256];
    moe_status st = check_cfg(cfg, why, sizeof why);
    if (st != MOE_OK) {
        fprintf(stderr, "moe_create: %s\n", why);
        return st;
    }
    moe_handle* h = new (std::nothrow) moe_handle();
    if (h == nullptr) return MOE_ERR_OOM;
    h->cfg = *cfg;
    h->esz = cfg->dtype == MOE_BF16 ? 2 : 4;
    if (const char* v = getenv("MOE_WAIT_LIMIT_MS")) {
        const long long ms = atoll(v);
        if (ms > 0) h->limit_ns = (uint64_t)ms * 1000000ull;
    }
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        delete h;
        return MOE_ERR_CUDA;
    }
    if (cfg->dtype == MOE_BF16) {
        int major = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
        if (major != 10) {
            delete h;
            return MOE_ERR_UNSUPPORTED;
        }
    }
    const int64_t T = cfg->max_tokens, k = cfg->top_k, E = cfg->num_experts, H = cfg->hidden;
    const int64_t R = T * k, NB = (T + kRouterTokens - 1) / kRouterTokens;
    const int64_t M = cfg->n_micro, I = cfg->inter, Is = cfg->shared_inter;
    const size_t esz = h->esz;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = round_up(off + (bytes ? bytes : 1), 256);
        return o;
    };
    const size_t o_err = take(sizeof(int));
    const size_t o_ids = take(R * 4), o_topw = take(R * 4), o_perm = take(R * 4), o_inv = take(R * 4);
    const size_t o_off = take((E + 1) * 4), o_ttc = take((E + 1) * 4), o_tsi = take((E + 1) * 4);
    const size_t o_smeta = take(6 * 4);
    const size_t o_hist = take(NB * E * 4), o_base = take(NB * E * 4), o_done = take(fused_counter_ints((int)E) * 4);
    const size_t o_sched = take(4 * 4);
    // the xp and h regions also hold the MXFP8 rows of a call with MXFP8
    // weights: codes, then (256-aligned) scale bytes of at most K/32 + 16 per
    // row and micro; the end grows with the call's R, so R's bound suffices
    auto rows_region = [&](size_t K, size_t micros) {
        const size_t mx = mx_scales_off(R, (int64_t)K) + R * micros * round_up(K / micros / 32, 16);
        return R * K * esz > mx ? R * K * esz : mx;
    };
    const size_t o_xp = take(rows_region(H, 1)), o_h = take(rows_region(M * I, M)), o_o = take(R * H * esz);
    const size_t o_hs = take(T * Is * esz), o_s = take(Is ? T * H * esz : 0);
    const size_t o_xst0 = take(T * H * esz), o_xst1 = take(T * H * esz);
    const size_t o_yst0 = take(T * H * esz), o_yst1 = take(T * H * esz);
    h->ws_bytes = off;
    if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return MOE_ERR_OOM;
    }
    char* b = static_cast<char*>(h->ws);
    h->err = reinterpret_cast<int*>(b + o_err);
    h->ids = reinterpret_cast<int32_t*>(b + o_ids);
    h->topw = reinterpret_cast<float*>(b + o_topw);
    h->perm = reinterpret_cast<int32_t*>(b + o_perm);
    h->inv = reinterpret_cast<int32_t*>(b + o_inv);
    h->offsets = reinterpret_cast<int32_t*>(b + o_off);
    h->tiles_tc = reinterpret_cast<int32_t*>(b + o_ttc);
    h->tiles_simt = reinterpret_cast<int32_t*>(b + o_tsi);
    h->shared_meta = reinterpret_cast<int32_t*>(b + o_smeta);
    h->blk_hist = reinterpret_cast<int32_t*>(b + o_hist);
    h->blk_base = reinterpret_cast<int32_t*>(b + o_base);
    h->done = reinterpret_cast<int*>(b + o_done);
    h->sched = reinterpret_cast<int*>(b + o_sched);
    h->xp = b + o_xp;
    h->hbuf = b + o_h;
    h->obuf = b + o_o;
    h->hs = b + o_hs;
    h->sbuf = b + o_s;
    h->x_stage[0] = b + o_xst0;
    h->x_stage[1] = b + o_xst1;
    h->y_stage[0] = b + o_yst0;
    h->y_stage[1] = b + o_yst1;
    if (cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess || cudaMemset(h->sched, 0, 4 * sizeof(int)) != cudaSuccess) {
        cudaFree(h->ws);
        delete h;
        return MOE_ERR_CUDA;
    }
    *out = h;
    return MOE_OK;
}

void moe_destroy(moe_handle* h) {
    if (h == nullptr) return;
    cudaDeviceSynchronize();
    for (cudaEvent_t ev : h->prof_ev) cudaEventDestroy(ev);
    for (int i = 0; i < 2; ++i) {
        if (h->ev_h2d[i] != nullptr) cudaEventDestroy(h->ev_h2d[i]);
        if (h->ev_comp[i] != nullptr) cudaEventDestroy(h->ev_comp[i]);
        if (h->ev_d2h[i] != nullptr) cudaEventDestroy(h->ev_d2h[i]);
    }
    if (h->pipe_in != nullptr) cudaStreamDestroy(h->pipe_in);
    if (h->pipe_out != nullptr) cudaStreamDestroy(h->pipe_out);
    if (h->ev_fork != nullptr) cudaEventDestroy(h->ev_fork);
    if (h->ev_join != nullptr) cudaEventDestroy(h->ev_join);
    if (h->side != nullptr) cudaStreamDestroy(h->side);
    cudaFree(h->ws);
    delete h;
}

moe_status moe_route(moe_handle* h, const void* x, const void* router_w, const float* router_bias, int32_t T,
                     int32_t* topk_ids, float* topk_w, int32_t* perm, int32_t* offsets, float* logits,
                     void* stream) {
    moe_status st = check_call(h, x, router_w, T);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->last_stream = s;
    const moe_config& c = h->cfg;
    const size_t nE1 = (size_t)(c.num_experts + 1) * 4;
    if (T == 0) {
        if (offsets != nullptr && cudaMemsetAsync(offsets, 0, nE1, s) != cudaSuccess)
            return set_err(h, MOE_ERR_CUDA, "memset offsets failed");
        return MOE_OK;
    }
    st = run_routing(h, x, router_w, router_bias, T, logits, s);
    end_call(h);
    if (st != MOE_OK) return st;
    const size_t R = (size_t)T * c.top_k;
    cudaError_t e = cudaSuccess;
    if (topk_ids && e == cudaSuccess) e = cudaMemcpyAsync(topk_ids, h->ids, R * 4, cudaMemcpyDeviceToDevice, s);
    if (topk_w && e == cudaSuccess) e = cudaMemcpyAsync(topk_w, h->topw, R * 4, cudaMemcpyDeviceToDevice, s);
    if (perm && e == cudaSuccess) e = cudaMemcpyAsync(perm, h->perm, R * 4, cudaMemcpyDeviceToDevice, s);
    if (offsets && e == cudaSuccess) e = cudaMemcpyAsync(offsets, h->offsets, nE1, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_err(h, e, "copy routing outputs");
    return MOE_OK;
}

moe_status moe_forward(moe_handle* h, const void* x, const void* router_w, const float* router_bias,
                       const void* const* w13, const void* const* w2, int32_t n_micro, int32_t top_k,
                       const void* shared_w13, const void* shared_w2, int32_t T, void* y, void* stream) {
    moe_status st = check_call(h, x, router_w, T);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    st = check_weights(h, w13, w2, n_micro, top_k, shared_w13, shared_w2, y);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->last_stream = s;
    st = run_forward(h, x, router_w, router_bias, w13, w2, shared_w13, shared_w2, T, y, s);
    end_call(h);
    return st;
}

moe_status moe_forward_mxfp8(moe_handle* h, const void* x, const void* router_w, const float* router_bias,
                             const void* const* w13_codes, const void* const* w13_scales,
                             const void* const* w2_codes, const void* const* w2_scales, int32_t n_micro,
                             int32_t top_k, const void* shared_w13, const void* shared_w2, int32_t T, void* y,
                             void* stream) {
    moe_status st = check_call(h, x, router_w, T);
    if (st != MOE_OK) return st;
    if (h->cfg.dtype != MOE_BF16) return set_err(h, MOE_ERR_UNSUPPORTED, "MXFP8 expert weights need a bf16 layer");
    if (T == 0) return MOE_OK;
    st = check_mxfp8(h, w13_codes, w13_scales, w2_codes, w2_scales, n_micro, top_k, shared_w13, shared_w2, y);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->last_stream = s;
    const MxScales mx{w13_scales, w2_scales};
    st = run_forward(h, x, router_w, router_bias, w13_codes, w2_codes, shared_w13, shared_w2, T, y, s, &mx);
    end_call(h);
    return st;
}

moe_status moe_forward_mxfp8_host_async(moe_handle* h, const void* x_host, const void* router_w,
                                        const float* router_bias, const void* const* w13_codes,
                                        const void* const* w13_scales, const void* const* w2_codes,
                                        const void* const* w2_scales, int32_t n_micro, int32_t top_k,
                                        const void* shared_w13, const void* shared_w2, int32_t T, void* y_host,
                                        void* stream) {
    moe_status st = check_call(h, h ? h->x_stage[0] : nullptr, router_w, T);
    if (st != MOE_OK) return st;
    if (h->cfg.dtype != MOE_BF16) return set_err(h, MOE_ERR_UNSUPPORTED, "MXFP8 expert weights need a bf16 layer");
    if (T == 0) return MOE_OK;
    if (x_host == nullptr || y_host == nullptr) return set_err(h, MOE_ERR_INVALID_ARG, "host x and y must be non-null");
    st = check_mxfp8(h, w13_codes, w13_scales, w2_codes, w2_scales, n_micro, top_k, shared_w13, shared_w2,
                     h->y_stage[0]);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->last_stream = s;
    const MxScales mx{w13_scales, w2_scales};
    return host_call(h, x_host, T, y_host, s, [&](const void* xd, void* yd) {
        return run_forward(h, xd, router_w, router_bias, w13_codes, w2_codes, shared_w13, shared_w2, T, yd, s, &mx);
    });
}

moe_status moe_quantize_mxfp8(const void* w, int64_t groups, int32_t rows, int32_t cols, void* codes,
                              void* scales, void* stream) {
    if (groups < 0 || rows < 0 || cols <= 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
    if ((groups > 0 && rows > 0) && (w == nullptr || codes == nullptr || scales == nullptr)) return MOE_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_mx_quantize(w, groups, rows, cols, codes, scales, sms, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

moe_status moe_forward_host_async(moe_handle* h, const void* x_host, const void* router_w,
                                  const float* router_bias, const void* const* w13, const void* const* w2,
                                  int32_t n_micro, int32_t top_k, const void* shared_w13, const void* shared_w2,
                                  int32_t T, void* y_host, void* stream) {
    moe_status st = check_call(h, h ? h->x_stage[0] : nullptr, router_w, T);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (x_host == nullptr || y_host == nullptr) return set_err(h, MOE_ERR_INVALID_ARG, "host x and y must be non-null");
    st = check_weights(h, w13, w2, n_micro, top_k, shared_w13, shared_w2, h->y_stage[0]);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->last_stream = s;
    return host_call(h, x_host, T, y_host, s, [&](const void* xd, void* yd) {
        return run_forward(h, xd, router_w, router_bias, w13, w2, shared_w13, shared_w2, T, yd, s);
    });
}

moe_status moe_forward_host(moe_handle* h, const void* x_host, const void* router_w, const float* router_bias,
                            const void* const* w13, const void* const* w2, int32_t n_micro, int32_t top_k,
                            const void* shared_w13, const void* shared_w2, int32_t T, void* y_host,
                            void* stream) {
    moe_status st = moe_forward_host_async(h, x_host, router_w, router_bias, w13, w2, n_micro, top_k, shared_w13,
                                           shared_w2, T, y_host, stream);
    if (st != MOE_OK || T == 0) return st;
    cudaError_t e = cudaStreamSynchronize(h->pipe_out);
    if (e != cudaSuccess) return cuda_err(h, e, "stream synchronize");
    return MOE_OK;
}

moe_status moe_sync(moe_handle* h) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (h->sticky) return set_err(h, MOE_ERR_STICKY, "handle is sticky after an earlier device error");
    cudaError_t e = cudaStreamSynchronize(h->last_stream);
    if (e == cudaSuccess && h->pipe_out != nullptr) e = cudaStreamSynchronize(h->pipe_out);
    if (e == cudaSuccess && h->pipe_in != nullptr) e = cudaStreamSynchronize(h->pipe_in);
    if (e != cudaSuccess) return cuda_err(h, e, "stream synchronize");
    int word = 0;
    if ((e = cudaMemcpy(&word, h->err, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_err(h, e, "read device error word");
    if (word & kErrTimeout) {
        h->sticky = true;
        return set_err(h, MOE_ERR_TIMEOUT, "a bounded device wait ran out (error word %d)", word);
    }
    if (word & kErrCheck) {
        h->sticky = true;
        return set_err(h, MOE_ERR_DEVICE_CHECK, "a device-side check failed (error word %d)", word);
    }
    return MOE_OK;
}

const char* moe_last_error(const moe_handle* h) { return h ? h->msg : "null handle"; }

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_OOM: return "MOE_ERR_OOM";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
        case MOE_ERR_STICKY: return "MOE_ERR_STICKY";
    }
    return "unknown moe_status";
}

void* moe_workspace_ptr(const moe_handle* h, int32_t which) {
    if (h == nullptr) return nullptr;
    switch (which) {
        case 0: return h->xp;
        case 1: return h->hbuf;
        case 2: return h->obuf;
        case 3: return h->inv;
        case 4: return h->err;
        default: return nullptr;
    }
}

moe_status moe_profile_begin(moe_handle* h, int32_t max_calls) {
    if (h == nullptr || max_calls <= 0) return MOE_ERR_INVALID_ARG;
    for (cudaEvent_t ev : h->prof_ev) cudaEventDestroy(ev);
    h->prof_ev.assign((size_t)max_calls * MOE_PROFILE_SLOTS * 2, nullptr);
    h->prof_used.assign((size_t)max_calls * MOE_PROFILE_SLOTS, 0);
    for (auto& ev : h->prof_ev) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) return cuda_err(h, e, "event create");
    }
    h->prof_max = max_calls;
    h->prof_calls = 0;
    h->prof_on = true;
    return MOE_OK;
}

moe_status moe_profile_end(moe_handle* h, float* ms, int32_t* launches) {
    if (h == nullptr || !h->prof_on) return MOE_ERR_INVALID_ARG;
    h->prof_on = false;
    for (int k = 0; k < MOE_PROFILE_SLOTS; ++k) {
        if (ms) ms[k] = 0.f;
        if (launches) launches[k] = 0;
    }
    for (int c = 0; c < h->prof_calls; ++c)
        for (int k = 0; k < MOE_PROFILE_SLOTS; ++k) {
            const size_t i = (size_t)c * MOE_PROFILE_SLOTS + k;
            if (!h->prof_used[i]) continue;
            cudaError_t e = cudaEventSynchronize(h->prof_ev[2 * i + 1]);
            float t = 0.f;
            if (e == cudaSuccess) e = cudaEventElapsedTime(&t, h->prof_ev[2 * i], h->prof_ev[2 * i + 1]);
            if (e != cudaSuccess) return cuda_err(h, e, "event elapsed time");
            if (ms) ms[k] += t;
            if (launches) launches[k] += 1;
        }
    return MOE_OK;
}

int64_t moe_launch_count(const moe_handle* h) { return h ? h->launches : 0; }

moe_status moe_set_accumulate(moe_handle* h, int32_t on) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    h->accumulate = on != 0;
    return MOE_OK;
}

moe_status moe_set_shared_stream(moe_handle* h, int32_t on) {
    if (h == nullptr) return MOE_ERR_INVALID_ARG;
    if (on && h->side == nullptr) {
        if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return set_err(h, MOE_ERR_CUDA, "could not create the shared-expert stream");
        }
    }
    h->shared_stream = on != 0;
    return MOE_OK;
}

moe_status moe_selftest_wait_timeout(int32_t timeout_us, void* stream) {
    if (timeout_us <= 0) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* d = nullptr;
    if (cudaMalloc(&d, sizeof(int)) != cudaSuccess) return MOE_ERR_OOM;
    int word = 0;
    cudaError_t e = cudaMemsetAsync(d, 0, sizeof(int), s);
    if (e == cudaSuccess) e = launch_wait_selftest(d, (uint64_t)timeout_us * 1000ull, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&word, d, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(d);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return (word & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_OK;
}

}  // extern "C"
