/*
 * moe.h - C ABI of the GB300 (sm_103a) routed mixture-of-experts FFN layer.
 *
 * The layer is the denoise/AR MoE feed-forward of "HunyuanImage3 Hybrid
 * Parallelism" (LightX2V blog), section 6: a router scores every token
 * against E experts, keeps the top-k, sorts the routes by expert, runs the
 * selected SwiGLU experts as grouped GEMMs and reduces each token's k expert
 * outputs with its routing scales. The multi-micro-shard form of section 6.1
 * is built in: n_micro weight shards of every expert share one routing, one
 * permutation, one set of offsets and one finalize.
 *
 * Conventions for every entry point
 *   - Tensors are plain device pointers (host pointers only where a name says
 *     so), row-major, dense, owned by the caller and 16-byte aligned. They
 *     must stay valid until the work enqueued on the stream has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls enqueue asynchronously and never synchronise, except
 *     moe_sync and moe_forward_host as documented. Work is ordered exactly as
 *     stream order: the library's kernels use programmatic dependent launch
 *     (a kernel may be placed on SMs while the previous kernel in the stream
 *     finishes), but each waits for that kernel to complete before it touches
 *     global memory. A kernel launched after a call sees all its results; if
 *     it uses programmatic dependent launch itself, it must wait likewise
 *     (griddepcontrol.wait) before reading them.
 *   - After moe_create, no call allocates device memory: the handle owns a
 *     workspace sized for cfg.max_tokens.
 *   - Errors are returned, never raised or aborted. A kernel-side failure
 *     (bounded wait that ran out, failed device check) is recorded in the
 *     handle's device error word; the next moe_sync reports it and the handle
 *     turns sticky: every later call returns MOE_ERR_STICKY until
 *     moe_destroy. moe_last_error gives a one-line description.
 *   - Calls on one handle must not overlap on the GPU (they share the
 *     workspace): issue them on one stream, or order the streams.
 */
#ifndef MOE_H
#define MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, size out of range, mismatch with cfg */
    MOE_ERR_UNSUPPORTED = 2,  /* shape the kernels do not cover (see moe_create) */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    MOE_ERR_OOM = 4,          /* workspace allocation failed in moe_create */
    MOE_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
    MOE_ERR_DEVICE_CHECK = 6, /* a device-side consistency check failed */
    MOE_ERR_STICKY = 7        /* an earlier device error poisoned this handle */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/*
 * Layer configuration. Names follow the pages: hidden H, experts E, top_k k,
 * inter I (intermediate size of ONE micro-shard; the blog's W2 [2][64][4096][768]
 * has I = 768 per micro), n_micro micro-shards per expert (section 5), and an
 * optional dense shared expert of intermediate size shared_inter (Ascend
 * Hunyuan Image 3.0 guide, section 3.1).
 *
 * Supported: 1 <= E <= 64, 1 <= k <= E (k <= 16), 1 <= n_micro <= 4,
 * max_tokens * k < 2^31.
 *   bf16 (tcgen05 path): H % 256 == 0, I % 128 == 0, shared_inter % 128 == 0.
 *   f32  (exact-fp32 SIMT path): H % 64 == 0, I % 64 == 0, shared_inter % 64 == 0.
 */
typedef struct {
    int32_t hidden;       /* H */
    int32_t num_experts;  /* E */
    int32_t top_k;        /* k */
    int32_t inter;        /* I per micro-shard */
    int32_t n_micro;      /* micro-shards per expert */
    int32_t max_tokens;   /* workspace capacity (tokens per call) */
    int32_t shared_inter; /* Is; 0 = no shared expert */
    int32_t dtype;        /* moe_dtype of x, weights and y */
} moe_config;

typedef struct moe_handle moe_handle;

/*
 * Validate cfg, allocate the workspace for cfg.max_tokens on the current
 * device and return a handle in *out. This is the only call that allocates.
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a bad cfg, MOE_ERR_OOM
 * if the workspace cannot be allocated, MOE_ERR_CUDA if no device is usable.
 */
moe_status moe_create(const moe_config *cfg, moe_handle **out);

/* Free the workspace and the handle (synchronises the device). NULL is a no-op. */
void moe_destroy(moe_handle *h);

/*
 * Routing only: router logits, softmax gate, top-k and renormalised scales,
 * expert offsets and the route permutation.
 *   blog section 6.1: ids and scores [num_tokens, top_k]; flatten the ids and
 *   sort them by expert -> permuted_to_expanded; bincount(...).cumsum(...) ->
 *   offsets; Ascend guide section 5.2: the gate is computed in fp32.
 * Inputs:  x [T][H] and router_w [E][H] in cfg.dtype; router_bias fp32 [E] or NULL.
 * Outputs (device, any may be NULL to skip):
 *   topk_ids [T][k] int32   experts by descending logit, ties -> lower index
 *   topk_w   [T][k] fp32    softmax over all E, restricted to the k and renormalised
 *   perm     [T*k]  int32   permuted_to_expanded: route r = t*k + j at its sorted
 *                           position; stable, so r ascends inside an expert
 *   offsets  [E+1]  int32   offsets[e] = first sorted position of expert e, offsets[E] = T*k
 *   logits   [T][E] fp32    the fp32 logits the decision was taken on
 * 0 <= T <= cfg.max_tokens; T == 0 writes offsets (all zero) and nothing else.
 */
moe_status moe_route(moe_handle *h, const void *x, const void *router_w,
                     const float *router_bias, int32_t T, int32_t *topk_ids,
                     float *topk_w, int32_t *perm, int32_t *offsets, float *logits,
                     void *stream);

/*
 * The whole layer (blog section 6.1 and 6.2):
 *   y[t] = sum_j topk_w[t][j] * sum_m down_m,e(silu(gate_m,e x_t) * up_m,e x_t)
 *          (+ shared_down(silu(shared_gate x_t) * shared_up x_t))
 * with e = topk_ids[t][j]. Steps, all ordered on `stream`: router + histogram,
 * scan -> offsets, stable placement -> permutation, one gather of x, grouped
 * GEMM1 with the SwiGLU epilogue for every micro, grouped GEMM2 accumulating
 * all micros of a route in one fp32 accumulator, (shared expert GEMMs),
 * finalize (see moe_set_shared_stream for running the shared expert's GEMMs
 * on a second stream).
 * Inputs (device):
 *   x          [T][H]
 *   router_w   [E][H], router_bias fp32 [E] or NULL
 *   w13        host array of n_micro device pointers; w13[m] -> [E][2I][H], rows
 *              0..I-1 of an expert are its gate rows and I..2I-1 its up rows
 *              (blog section 4.4 [gate_micro, up_micro]; Ascend guide section 2.2).
 *              A micro-major pack W1[n_micro][E][2I][H] is passed as
 *              w13[m] = W1 + m*E*2I*H without repacking (blog section 5).
 *   w2         host array of n_micro device pointers; w2[m] -> [E][H][I]
 *   n_micro, top_k   must equal cfg.n_micro and cfg.top_k
 *   shared_w13 [2Is][H] and shared_w2 [H][Is], both NULL iff cfg.shared_inter == 0
 * Output: y [T][H] in cfg.dtype (fp32 accumulation, one rounding at the end).
 */
moe_status moe_forward(moe_handle *h, const void *x, const void *router_w,
                       const float *router_bias, const void *const *w13,
                       const void *const *w2, int32_t n_micro, int32_t top_k,
                       const void *shared_w13, const void *shared_w2, int32_t T,
                       void *y, void *stream);

/*
 * moe_forward with x and y in HOST memory (pinned memory gives the fastest
 * copies, and only pinned memory lets the copies overlap the layer): copies x
 * to one of the handle's two device staging buffers, runs the layer on
 * `stream` and copies y back, then waits until y is in y_host. Weights and the
 * router are device pointers as in moe_forward. The copies run on two streams
 * the handle creates on its first host-buffer call (MOE_ERR_CUDA if it cannot),
 * ordered against the layer by events.
 */
moe_status moe_forward_host(moe_handle *h, const void *x_host, const void *router_w,
                            const float *router_bias, const void *const *w13,
                            const void *const *w2, int32_t n_micro, int32_t top_k,
                            const void *shared_w13, const void *shared_w2, int32_t T,
                            void *y_host, void *stream);

/*
 * moe_forward_host without the wait: enqueues the copy of x, the layer and the
 * copy of y, and returns. Consecutive calls alternate between the two staging
 * buffers, so the copy of x of call n+1 and the copy of y of call n-1 overlap
 * the layer of call n (the serving loop's host I/O hides behind the GPU work).
 * x_host must stay unchanged, and y_host unread, until moe_sync returns (which
 * waits for every copy); with accumulation on (moe_set_accumulate), y_host is
 * also read, so calls in flight together need distinct y_host buffers.
 */
moe_status moe_forward_host_async(moe_handle *h, const void *x_host, const void *router_w,
                                  const float *router_bias, const void *const *w13,
                                  const void *const *w2, int32_t n_micro, int32_t top_k,
                                  const void *shared_w13, const void *shared_w2, int32_t T,
                                  void *y_host, void *stream);

/*
 * Block-scaled FP8 expert weights (the pages list FP8 among the precision
 * choices of the runtime: vflash architecture page, "Layered execution
 * model"; they fix no format). The reading taken is the OCP Microscaling
 * MXFP8 format: each expert weight is an FP8 E4M3 code (OCP E4M3FN, largest
 * 448) with one E8M0 power-of-two scale per 32 consecutive elements along K;
 * the layer computes with w = code * 2^(S-127). Every batch size runs the
 * tensor cores' block-scaled FP8 MMA: the gathered token rows and h (taken at
 * its bf16 value) are quantised to MXFP8 by the same rule as the weights
 * (along H and along each micro's I), and each GEMM multiplies the codes with
 * their scales exactly, accumulating in fp32; the router, the shared expert
 * (its weights stay bf16) and y keep the layer's bf16.
 *
 * Quantisation of bf16 weights w [groups][rows][cols] along cols (cols % 32
 * == 0): codes [groups][rows][cols] uint8 and scales [groups][cols/32][rows]
 * uint8. Per block: shared = floor(log2(max |v|)) - 8, clamped to
 * [-127, 127] (0 for an all-zero block); code = E4M3 of v / 2^shared,
 * nearest, ties to even, saturating at +-448; S = shared + 127. Device
 * pointers; enqueued on `stream`; needs no handle. Returns MOE_ERR_INVALID_ARG
 * for bad sizes or null pointers, MOE_ERR_CUDA on a launch failure.
 * An expert's w13[m] [E][2I][H] is quantised with groups = E, rows = 2I,
 * cols = H (scales [E][H/32][2I]); w2[m] [E][H][I] with rows = H, cols = I
 * (scales [E][I/32][H]).
 */
moe_status moe_quantize_mxfp8(const void *w, int64_t groups, int32_t rows, int32_t cols,
                              void *codes, void *scales, void *stream);

/*
 * moe_forward with MXFP8 routed-expert weights: w13_codes[m] / w13_scales[m]
 * and w2_codes[m] / w2_scales[m] as produced by moe_quantize_mxfp8 (device
 * pointers, 16-byte aligned). Supported for bf16 layers (whose hidden and
 * inter sizes, multiples of 256 and 128, fill its 128-deep K stages). Other
 * arguments, ownership, the accumulate switch and errors as for moe_forward.
 */
moe_status moe_forward_mxfp8(moe_handle *h, const void *x, const void *router_w,
                             const float *router_bias, const void *const *w13_codes,
                             const void *const *w13_scales, const void *const *w2_codes,
                             const void *const *w2_scales, int32_t n_micro, int32_t top_k,
                             const void *shared_w13, const void *shared_w2, int32_t T,
                             void *y, void *stream);

/* moe_forward_mxfp8 with x and y in host memory, as moe_forward_host_async. */
moe_status moe_forward_mxfp8_host_async(moe_handle *h, const void *x_host, const void *router_w,
                                        const float *router_bias, const void *const *w13_codes,
                                        const void *const *w13_scales, const void *const *w2_codes,
                                        const void *const *w2_scales, int32_t n_micro, int32_t top_k,
                                        const void *shared_w13, const void *shared_w2, int32_t T,
                                        void *y_host, void *stream);

/*
 * Output accumulation. With `on` non-zero, later moe_forward / moe_forward_host
 * calls on this handle add the layer's output into y (y += layer(x)): the
 * finalize reads y, adds it in fp32 and rounds once. It serves a residual add,
 * and the pages' two-dispatch form of a multi-micro layer (blog section 10.3:
 * one full layer call per micro-shard, outputs added), which is two calls of
 * single-micro handles, the second with accumulation on. Default off.
 */
moe_status moe_set_accumulate(moe_handle *h, int32_t on);

/*
 * Shared expert on a second stream (Ascend guide section 3.1, multi-stream
 * overlap): when on, a bf16 layer with a shared expert runs the shared
 * expert's two GEMMs, for calls with T > 16, on a stream the handle creates
 * (on the first call of this function with on != 0), forked from the call's
 * stream after routing and joined back before the finalize; the call still
 * completes in `stream` order and its result is bit-identical. Default off:
 * on one GPU the routed and shared GEMMs both fill every SM, so running them
 * concurrently does not shorten the layer (it only overlaps the gather).
 * Returns MOE_ERR_CUDA if the stream or its events cannot be created.
 */
moe_status moe_set_shared_stream(moe_handle *h, int32_t on);

/*
 * Synchronise the stream of the handle's last call (and the host-copy streams
 * of the host-buffer calls) and read its device error word. Returns MOE_OK, or
 * MOE_ERR_TIMEOUT / MOE_ERR_DEVICE_CHECK (and makes the handle sticky), or
 * MOE_ERR_CUDA.
 */
moe_status moe_sync(moe_handle *h);

/* One-line description of the handle's last error ("" if none). Never NULL. */
const char *moe_last_error(const moe_handle *h);

/* Static name of a status code. */
const char *moe_status_string(moe_status s);

/*
 * Diagnostics for tests: device address of a workspace buffer of the last
 * call. which: 0 = gathered input xp [T*k][H], 1 = SwiGLU output h [T*k][n_micro*I],
 * 2 = expert outputs o [T*k][H], 3 = inverse permutation [T*k] int32,
 * 4 = device error word (int32). Returns NULL for an unknown `which`. After a
 * moe_forward_mxfp8 call with T > 16, regions 0 and 1 hold the MXFP8 codes
 * (uint8) of xp [T*k][H] and of h [T*k][n_micro*I].
 */
void *moe_workspace_ptr(const moe_handle *h, int32_t which);

/*
 * Diagnostics: per-kernel timing with CUDA events. Between moe_profile_begin
 * and moe_profile_end, the first `max_calls` calls of moe_forward /
 * moe_forward_host / moe_route record an event pair around every kernel they
 * launch, on the call's stream. moe_profile_end synchronises those events and
 * writes, per kernel slot, the summed duration in milliseconds and the number
 * of launches. Slots: 0 router, 1 scan, 2 place, 3 gather (with MXFP8 expert
 * weights and T > 16: gather and MXFP8 quantisation of the token rows),
 * 4 GEMM1 (+SwiGLU; with MXFP8 expert weights and T > 16 also the MXFP8
 * quantisation of h), 5 GEMM2, 6 shared-expert GEMM1, 7 shared-expert GEMM2,
 * 8 finalize.
 */
#define MOE_PROFILE_SLOTS 9
moe_status moe_profile_begin(moe_handle *h, int32_t max_calls);
moe_status moe_profile_end(moe_handle *h, float *ms /* [MOE_PROFILE_SLOTS] */,
                           int32_t *launches /* [MOE_PROFILE_SLOTS] */);

/* Number of kernels this handle has launched since moe_create. */
int64_t moe_launch_count(const moe_handle *h);

/*
 * Routing for callers that cannot allocate device memory. The pages have no
 * counterpart to this entry point: it exists for programs whose device heap
 * belongs to a pooling allocator with a fixed budget, or whose hot path must
 * not take the implicit device synchronisation of cudaMalloc. It computes the
 * same topk_ids, topk_w, perm and offsets as moe_route (same kernels, same
 * bits) without a handle: its intermediate data lives in one file-scope
 * device array of the library (about 1.3 MB, held on every GPU that loads the
 * library until the process exits). It calls no cudaMalloc/cudaFree.
 *   x [T][hidden], router_w [num_experts][hidden] in `dtype`; router_bias fp32
 *   [num_experts] or NULL; outputs as in moe_route (all four required; logits
 *   are not produced).
 *   0 <= T <= MOE_ROUTE_NOALLOC_MAX_TOKENS, hidden % 64 == 0 (bf16) or % 32 (fp32),
 *   1 <= num_experts <= 64, 1 <= top_k <= min(num_experts, 16); anything else,
 *   or a null or misaligned pointer, returns MOE_ERR_INVALID_ARG.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. The cached address belongs to the device's primary context: a
 * process that resets the device (cudaDeviceReset) must not call it again.
 * Every call shares the array and overwrites what the previous call left
 * there, so calls that overlap on the GPU race: order them (one stream).
 * The call is asynchronous: a bounded device wait that ran out or a failed
 * device-side check is recorded in the array's error word (cleared at the
 * start of every call), which moe_route_noalloc_status reads back.
 */
#define MOE_ROUTE_NOALLOC_MAX_TOKENS 16384
moe_status moe_route_noalloc(const void *x, const void *router_w, const float *router_bias,
                             int32_t T, int32_t hidden, int32_t num_experts, int32_t top_k,
                             int32_t dtype, int32_t *topk_ids, float *topk_w, int32_t *perm,
                             int32_t *offsets, void *stream);

/*
 * Outcome of the last moe_route_noalloc call on the current device, for the
 * same allocation-free callers (no counterpart on the pages either):
 * synchronises `stream` (the stream that call used), copies the error word of
 * the file-scope array to the host (no allocation) and returns MOE_OK,
 * MOE_ERR_TIMEOUT (a bounded device wait ran out: the outputs are incomplete)
 * or MOE_ERR_DEVICE_CHECK (a device-side consistency check failed: perm and
 * offsets must not be used); MOE_ERR_CUDA if the stream or the copy failed.
 * The word is not sticky: the next moe_route_noalloc call clears it.
 */
moe_status moe_route_noalloc_status(void *stream);

/*
 * Self-test of the bounded device-side wait: launches one block whose thread
 * waits on an mbarrier that nothing completes, with a limit of `timeout_us`
 * microseconds, then returns the status the kernel reported (expected:
 * MOE_ERR_TIMEOUT). Synchronises the stream. Does not touch any handle.
 */
moe_status moe_selftest_wait_timeout(int32_t timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
