/*
 * moe_oracle.c - plain, slow fp64 CPU oracle of the routed mixture-of-experts
 * feed-forward layer, including the multi-micro-shard variant.
 *
 * TEST INFRASTRUCTURE ONLY. This file is loaded by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg, and by nothing else. It shares
 * no code, header, table or helper with the CUDA path; the two meet only in the
 * seeded input generator, which holds none of the layer's arithmetic.
 *
 * What it computes, and where the pages define it:
 *   - "HunyuanImage3 Hybrid Parallelism" (LightX2V blog), section 5: the
 *     micro-major MoE pack, W1[micro][expert][2I][H] and W2[micro][expert][H][I];
 *     section 4.4: each micro's fused gate/up block is [gate_micro; up_micro];
 *     section 6.1: router ids and scores of shape [num_tokens, top_k], route
 *     sort by expert giving permuted_to_expanded, bincount+cumsum offsets, one
 *     gather of the input, per micro grouped GEMM1 -> SwiGLU -> grouped GEMM2,
 *     inverse permutation, and the finalize
 *         output[token] = sum over routes of scale[token, route] *
 *                         (micro0_partial + micro1_partial).
 *   - CANN/Ascend Hunyuan Image 3.0 guide, section 2.2: the expert is
 *     down(SiLU(gate(x)) * up(x)) with w13 = concat(gate, up) and the fused
 *     activation SiLU(x[0]) * x[1]; section 3.1: a shared expert beside the
 *     routed ones; section 5.2: the gate (router) is computed in fp32.
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - gate = softmax over all experts, then the top-k, then the k weights are
 *     renormalised to sum to one;
 *   - the top-k decision is taken on fp32 logits (the gate's precision in the
 *     Ascend guide, section 5.2): each logit is formed in fp64 from the exact
 *     input values and rounded once to fp32; ties go to the lower expert index
 *     and the k slots are ordered by descending logit, ties by lower index;
 *   - the route sort is stable in the flattened route index r = t*k + j;
 *   - offsets has E+1 entries, offsets[E] = T*k;
 *   - the shared expert's output is added unscaled.
 *
 * All floating-point arithmetic is fp64. Inputs are read as fp32, as bf16 bit
 * patterns (uint16) or as fp64, and widened exactly to fp64.
 *
 * Quantised expert weights (the block-scaled FP8 variant of the experts; the
 * pages name no format, the reading taken is the OCP Microscaling (MX) MXFP8
 * format): codes are FP8 E4M3 (OCP E4M3FN: 4 exponent bits, bias 7, 3 mantissa
 * bits, no infinities, largest 448), one shared power-of-two scale (E8M0 code
 * S, value 2^(S-127)) per block of 32 consecutive elements along K; the value
 * of a weight is exactly code * scale (the MX definition), formed in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 2

/* Exact widening of one stored element to fp64. */
static double elem(const void *p, int dtype, int64_t i)
{
    if (dtype == ORC_F64)
        return ((const double *)p)[i];
    if (dtype == ORC_F32)
        return (double)((const float *)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static size_t elem_size(int dtype) { return dtype == ORC_F64 ? 8u : (dtype == ORC_F32 ? 4u : 2u); }

/* Pointer to element i of a typed buffer (used to address expert blocks). */
static const void *elem_ptr(const void *p, int dtype, int64_t i)
{
    return (const char *)p + (size_t)i * elem_size(dtype);
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

static void mx_round_vec(double *v, int64_t n);
static double bf16_round(double v);

static int max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int thread_id(void)
{
#ifdef _OPENMP
    return omp_get_thread_num();
#else
    return 0;
#endif
}

/*
 * Router logits (blog section 6.1, "the router produces ... routing scores";
 * Ascend guide section 5.2, gate linear):
 *     logits[t][e] = sum_h x[t][h] * Wr[e][h]  (+ bias[e])
 * x is [T][H], Wr is [E][H], bias is fp32 [E] or NULL. Output fp64 [T][E].
 */
int orc_logits(const void *x, const void *wr, int dtype, const float *bias,
               int64_t T, int64_t H, int64_t E, double *logits)
{
    if (T < 0 || H <= 0 || E <= 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            double s = 0.0;
            for (int64_t h = 0; h < H; ++h)
                s += elem(x, dtype, t * H + h) * elem(wr, dtype, e * H + h);
            if (bias)
                s += (double)bias[e];
            logits[t * E + e] = s;
        }
    }
    return 0;
}

/*
 * Softmax gate, top-k and renormalisation (blog section 6.1: ids and scores of
 * shape [num_tokens, top_k]; Ascend guide section 2.3: GatingTopK).
 *   1. l[e] = fp32 rounding of logits[t][e]   (gate precision)
 *   2. p = softmax(l) over all E experts     (row max subtracted)
 *   3. k rounds: take the not-yet-taken expert with the largest l;
 *      on equal l the lower index wins (strict '>' while scanning upward)
 *   4. w_j = p[id_j] / sum_j' p[id_j']
 * ids [T][k] int32, w [T][k] fp64; probs [T][E] (the full softmax) if non-NULL.
 */
int orc_route(const double *logits, int64_t T, int64_t E, int64_t k,
              int32_t *ids, double *w, double *probs)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E)
        return -1;
    int nt = max_threads();
    double *lbuf = (double *)malloc(sizeof(double) * (size_t)(E * nt));
    double *pbuf = (double *)malloc(sizeof(double) * (size_t)(E * nt));
    char *tbuf = (char *)malloc((size_t)(E * nt));
    if (!lbuf || !pbuf || !tbuf) {
        free(lbuf);
        free(pbuf);
        free(tbuf);
        return -2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double *l = lbuf + (int64_t)thread_id() * E;
        double *p = pbuf + (int64_t)thread_id() * E;
        char *taken = tbuf + (int64_t)thread_id() * E;
        double mx = -INFINITY;
        for (int64_t e = 0; e < E; ++e) {
            l[e] = (double)(float)logits[t * E + e];
            if (l[e] > mx)
                mx = l[e];
        }
        double z = 0.0;
        for (int64_t e = 0; e < E; ++e) {
            p[e] = exp(l[e] - mx);
            z += p[e];
        }
        for (int64_t e = 0; e < E; ++e) {
            p[e] /= z;
            if (probs)
                probs[t * E + e] = p[e];
            taken[e] = 0;
        }
        double sel = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best]))
                    best = e;
            taken[best] = 1;
            ids[t * k + j] = (int32_t)best;
            sel += p[best];
        }
        for (int64_t j = 0; j < k; ++j)
            w[t * k + j] = p[ids[t * k + j]] / sel;
    }
    free(lbuf);
    free(pbuf);
    free(tbuf);
    return 0;
}

/*
 * Route sort and expert offsets (blog section 6.1: flatten the ids, sort them
 * by expert -> permuted_to_expanded; bincount(...).cumsum(...) -> offsets;
 * section 6.2: permutation inverse).
 *   counts[e]   = number of routes r = t*k+j with ids[r] == e
 *   offsets[0]  = 0, offsets[e+1] = offsets[e] + counts[e]
 *   perm        = stable counting sort of r by ids[r] (r ascending inside an expert)
 *   inv[perm[i]] = i
 * Returns -1 if an id is out of [0, E).
 */
int orc_permute(const int32_t *ids, int64_t T, int64_t k, int64_t E,
                int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv)
{
    int64_t R = T * k;
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t r = 0; r < R; ++r) {
        if (ids[r] < 0 || ids[r] >= E)
            return -1;
        counts[ids[r]] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    if (!fill)
        return -2;
    for (int64_t e = 0; e < E; ++e)
        fill[e] = offsets[e];
    for (int64_t r = 0; r < R; ++r)
        perm[fill[ids[r]]++] = (int32_t)r;
    for (int64_t i = 0; i < R; ++i)
        inv[perm[i]] = (int32_t)i;
    free(fill);
    return 0;
}

/*
 * One SwiGLU expert applied to one row, accumulated with a scale
 * (Ascend guide section 2.2: down(SiLU(gate(x)) * up(x)); blog section 4.4:
 * a micro's w13 block is [gate rows (I); up rows (I)]):
 *     g_i = sum_h w13[i][h]   * x[h]        i in [0, I)
 *     u_i = sum_h w13[I+i][h] * x[h]
 *     a_i = silu(g_i) * u_i,   silu(z) = z / (1 + exp(-z))
 *     acc[h] += scale * sum_i w2[h][i] * a_i
 * w13 is [2I][H], w2 is [H][I]; a is caller scratch of length I. With mx_act
 * set, a is the layer's bf16 activation (each a_i rounded to bf16, nearest,
 * ties to even: the precision h is stored in between the GEMMs) and is
 * replaced by its MXFP8 value (blocks of 32 along I) before the down
 * projection: the activation input of a block-scaled FP8 GEMM2.
 */
static void swiglu_expert_acc(const double *xv, int64_t H, int64_t I,
                              const void *w13, const void *w2, int dtype,
                              double scale, double *acc, double *a, int mx_act)
{
    for (int64_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            g += elem(w13, dtype, i * H + h) * xv[h];
            u += elem(w13, dtype, (I + i) * H + h) * xv[h];
        }
        a[i] = silu(g) * u;
    }
    if (mx_act) {
        for (int64_t i = 0; i < I; ++i)
            a[i] = bf16_round(a[i]);
        mx_round_vec(a, I);
    }
    for (int64_t h = 0; h < H; ++h) {
        double s = 0.0;
        for (int64_t i = 0; i < I; ++i)
            s += elem(w2, dtype, h * I + i) * a[i];
        acc[h] += scale * s;
    }
}

/*
 * The layer's plain per-token definition, evaluated on a list of tokens:
 *     y[t] = sum_j w[t][j] * sum_m FFN_{m, ids[t][j]}(x[t])  (+ FFN_shared(x[t]))
 * where FFN_{m,e} is the SwiGLU expert built from micro m's blocks of expert e:
 * w13[m] + e*2I*H and w2[m] + e*H*I (blog section 5, micro-major pack).
 * The shared expert (Ascend guide section 3.1) is the same SwiGLU form with
 * intermediate size Is, sw13 [2Is][H] and sw2 [H][Is]; pass NULL for none.
 * ids/w are the routing of ALL tokens ([T][k]); tokens[] selects which rows to
 * evaluate; y is [n_tokens][H].
 */
int orc_forward_tokens_typed(const void *x, int dtype, int w_dtype, int s_dtype, int64_t H, int64_t E,
                             int64_t k, int64_t I, int64_t n_micro,
                             const void *const *w13, const void *const *w2,
                             const void *sw13, const void *sw2, int64_t Is,
                             const int32_t *ids, const double *w,
                             const int64_t *tokens, int64_t n_tokens, double *y, int mx_act)
{
    if (H <= 0 || E <= 0 || k <= 0 || I <= 0 || n_micro <= 0 || n_tokens < 0)
        return -1;
    if (mx_act && (H % 32 != 0 || I % 32 != 0))
        return -1;
    int nt = max_threads();
    int64_t scratch = I > Is ? I : Is;
    double *xbuf = (double *)malloc(sizeof(double) * (size_t)(2 * H * nt));
    double *abuf = (double *)malloc(sizeof(double) * (size_t)(scratch * nt));
    if (!xbuf || !abuf) {
        free(xbuf);
        free(abuf);
        return -2;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < n_tokens; ++n) {
        double *xv = xbuf + (int64_t)thread_id() * 2 * H;
        double *xq = xv + H;  /* the routed experts' input: x, or its MXFP8 value */
        double *a = abuf + (int64_t)thread_id() * scratch;
        int64_t t = tokens[n];
        double *acc = y + n * H;
        for (int64_t h = 0; h < H; ++h) {
            xv[h] = elem(x, dtype, t * H + h);
            xq[h] = xv[h];
            acc[h] = 0.0;
        }
        if (mx_act)
            mx_round_vec(xq, H);
        for (int64_t j = 0; j < k; ++j) {
            int64_t e = ids[t * k + j];
            for (int64_t m = 0; m < n_micro; ++m)
                swiglu_expert_acc(xq, H, I,
                                  elem_ptr(w13[m], w_dtype, e * 2 * I * H),
                                  elem_ptr(w2[m], w_dtype, e * H * I),
                                  w_dtype, w[t * k + j], acc, a, mx_act);
        }
        if (sw13 && sw2 && Is > 0)
            swiglu_expert_acc(xv, H, Is, sw13, sw2, s_dtype, 1.0, acc, a, 0);
    }
    free(xbuf);
    free(abuf);
    return 0;
}

/* orc_forward_tokens_typed with the routed and shared weights in x's dtype. */
int orc_forward_tokens(const void *x, int dtype, int64_t H, int64_t E, int64_t k,
                       int64_t I, int64_t n_micro,
                       const void *const *w13, const void *const *w2,
                       const void *sw13, const void *sw2, int64_t Is,
                       const int32_t *ids, const double *w,
                       const int64_t *tokens, int64_t n_tokens, double *y)
{
    return orc_forward_tokens_typed(x, dtype, dtype, dtype, H, E, k, I, n_micro, w13, w2, sw13, sw2,
                                    Is, ids, w, tokens, n_tokens, y, 0);
}

/*
 * The same layer evaluated the way the multi-micro method organises it
 * (blog section 6.1), for cross-checking the permutation and the finalize:
 *   xp[i]   = x[perm[i] / k]                    one gather, shared by all micros
 *   o[i]    = sum_m FFN_{m,e}(xp[i])            e = the expert whose segment
 *                                               [offsets[e], offsets[e+1]) holds i
 *   y[t]    = sum_j w[t][j] * o[inv[t*k + j]]   (+ FFN_shared(x[t]))
 * y is [T][H]. Memory: R*H*2 doubles, so small shapes only.
 */
int orc_forward_permuted(const void *x, int dtype, int64_t T, int64_t H, int64_t E,
                         int64_t k, int64_t I, int64_t n_micro,
                         const void *const *w13, const void *const *w2,
                         const void *sw13, const void *sw2, int64_t Is,
                         const double *w, const int32_t *offsets,
                         const int32_t *perm, const int32_t *inv, double *y)
{
    int64_t R = T * k;
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || I <= 0 || n_micro <= 0)
        return -1;
    if (offsets[0] != 0 || offsets[E] != R)
        return -1;
    int nt = max_threads();
    int64_t scratch = I > Is ? I : Is;
    double *xp = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R * H : 1));
    double *o = (double *)calloc((size_t)(R > 0 ? R * H : 1), sizeof(double));
    double *xbuf = (double *)malloc(sizeof(double) * (size_t)(H * nt));
    double *abuf = (double *)malloc(sizeof(double) * (size_t)(scratch * nt));
    int rc = 0;
    if (!xp || !o || !xbuf || !abuf) {
        rc = -2;
        goto done;
    }
    /* one gather, shared by every micro */
    for (int64_t i = 0; i < R; ++i) {
        int64_t t = perm[i] / k;
        for (int64_t h = 0; h < H; ++h)
            xp[i * H + h] = elem(x, dtype, t * H + h);
    }
    /* grouped GEMM1 -> SwiGLU -> grouped GEMM2, summed over micros, per segment */
    for (int64_t e = 0; e < E; ++e) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = offsets[e]; i < offsets[e + 1]; ++i) {
            double *a = abuf + (int64_t)thread_id() * scratch;
            for (int64_t m = 0; m < n_micro; ++m)
                swiglu_expert_acc(xp + i * H, H, I,
                                  elem_ptr(w13[m], dtype, e * 2 * I * H),
                                  elem_ptr(w2[m], dtype, e * H * I),
                                  dtype, 1.0, o + i * H, a, 0);
        }
    }
    /* finalize: routing scale applied once, top-k reduced once */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double *xv = xbuf + (int64_t)thread_id() * H;
        double *a = abuf + (int64_t)thread_id() * scratch;
        double *acc = y + t * H;
        for (int64_t h = 0; h < H; ++h)
            acc[h] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            const double *row = o + (int64_t)inv[t * k + j] * H;
            for (int64_t h = 0; h < H; ++h)
                acc[h] += w[t * k + j] * row[h];
        }
        if (sw13 && sw2 && Is > 0) {
            for (int64_t h = 0; h < H; ++h)
                xv[h] = elem(x, dtype, t * H + h);
            swiglu_expert_acc(xv, H, Is, sw13, sw2, dtype, 1.0, acc, a, 0);
        }
    }
done:
    free(xp);
    free(o);
    free(xbuf);
    free(abuf);
    return rc;
}

/*
 * ---------------------------------------------------------------- MXFP8
 * Value of an E4M3 code (OCP E4M3FN): sign, 4-bit exponent e (bias 7), 3-bit
 * mantissa m; e == 0 is subnormal m * 2^-9; the code S.1111.111 is NaN (never
 * produced by the quantiser below).
 */
static double e4m3_value(uint8_t c)
{
    int e = (c >> 3) & 0xF, m = c & 7;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    if (e == 15 && m == 7)
        v = NAN;
    return (c & 0x80) ? -v : v;
}

/*
 * Magnitude code (0 .. 0x7E) of the E4M3 value nearest to u >= 0, ties to the
 * even mantissa, saturating at 448: u is split into an exponent and a 3-bit
 * mantissa (the subnormal range keeps the exponent of 2^-6) and the scaled
 * mantissa is rounded half to even.
 */
static uint8_t e4m3_round_mag(double u)
{
    if (!(u < 448.0))
        return 0x7E;
    int e;
    if (u < ldexp(1.0, -6)) {
        e = -6;  /* subnormal: steps of 2^-9 */
    } else {
        int ex;
        frexp(u, &ex);  /* u = f * 2^ex, f in [0.5, 1) */
        e = ex - 1;
    }
    double scaled = ldexp(u, 3 - e);  /* u / 2^(e-3): the mantissa in units of 1/8 */
    double q = nearbyint(scaled);     /* default rounding: to nearest, ties to even */
    int64_t qi = (int64_t)q;
    if (u < ldexp(1.0, -6))
        return (uint8_t)qi;           /* 0..8; 8 is the normal 2^-6 (code 0x08) */
    if (qi == 16) {                   /* mantissa overflowed: next binade */
        qi = 8;
        e += 1;
    }
    int code = ((e + 7) << 3) | (int)(qi - 8);
    return code > 0x7E ? 0x7E : (uint8_t)code;
}

/*
 * v rounded to bfloat16 (1 sign, 8 exponent and 7 fraction bits: 8 significant
 * bits, smallest normal 2^-126, subnormal steps of 2^-133, largest finite
 * (2 - 2^-7) * 2^127), nearest with ties to even; beyond the largest finite
 * value after rounding: infinity. Exact in fp64: scaling by powers of two.
 */
static double bf16_round(double v)
{
    double u = fabs(v);
    if (u == 0.0 || isnan(u) || isinf(u))
        return v;
    int e;
    if (u < ldexp(1.0, -126)) {
        e = -126;  /* subnormal: the step of the smallest normal binade */
    } else {
        int ex;
        frexp(u, &ex);  /* u = f * 2^ex, f in [0.5, 1) */
        e = ex - 1;
    }
    double q = ldexp(nearbyint(ldexp(u, 7 - e)), e - 7);  /* 128 steps per binade; 256 carries into the next */
    if (q > ldexp(255.0, 120))  /* (2 - 2^-7) * 2^127 */
        q = INFINITY;
    return signbit(v) ? -q : q;
}

/* bf16_round of n values (for tests of the rounding rule). */
int orc_bf16_round(const double *v, int64_t n, double *out)
{
    if (n < 0)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_round(v[i]);
    return 0;
}

/*
 * The MXFP8 value of a vector v[0..n) (n % 32 == 0), in place: each block of
 * 32 consecutive elements takes the shared exponent floor(log2(max |v|)) - 8
 * (clamped to [-127, 127]; 0 for an all-zero block) and every element becomes
 * its E4M3 code (nearest, ties to even, saturating at 448) times 2^shared --
 * the same rule as orc_mx_quantize, applied to activations.
 */
static void mx_round_vec(double *v, int64_t n)
{
    for (int64_t b = 0; b < n; b += 32) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i)
            if (fabs(v[b + i]) > amax)
                amax = fabs(v[b + i]);
        int shared = 0;
        if (amax > 0.0) {
            int ex;
            frexp(amax, &ex);
            shared = (ex - 1) - 8;
            if (shared < -127)
                shared = -127;
            if (shared > 127)
                shared = 127;
        }
        for (int i = 0; i < 32; ++i) {
            double q = ldexp(e4m3_value(e4m3_round_mag(ldexp(fabs(v[b + i]), -shared))), shared);
            v[b + i] = signbit(v[b + i]) ? -q : q;
        }
    }
}

/*
 * MXFP8 quantisation of w [groups][rows][cols] along cols, in blocks of 32
 * (OCP Microscaling: shared exponent = floor(log2(max |v|)) - 8, 8 being the
 * largest exponent of E4M3; codes = E4M3 of v / 2^shared, nearest, ties to
 * even, saturating): codes [groups][rows][cols], scales [groups][cols/32][rows]
 * as E8M0 codes S = shared + 127 (shared clamped to [-127, 127]; an all-zero
 * block gets S = 127). The sign bit of a code is the sign bit of v.
 */
int orc_mx_quantize(const void *w, int dtype, int64_t groups, int64_t rows, int64_t cols,
                    uint8_t *codes, uint8_t *scales)
{
    if (groups < 0 || rows < 0 || cols <= 0 || cols % 32 != 0)
        return -1;
    const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t gr = 0; gr < groups * rows; ++gr) {
        const int64_t g = gr / rows, r = gr % rows;
        for (int64_t b = 0; b < nb; ++b) {
            const int64_t base = gr * cols + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double v = fabs(elem(w, dtype, base + i));
                if (v > amax)
                    amax = v;
            }
            int shared = 0;
            if (amax > 0.0) {
                int ex;
                frexp(amax, &ex);
                shared = (ex - 1) - 8;
                if (shared < -127)
                    shared = -127;
                if (shared > 127)
                    shared = 127;
            }
            scales[(g * nb + b) * rows + r] = (uint8_t)(shared + 127);
            for (int i = 0; i < 32; ++i) {
                double v = elem(w, dtype, base + i);
                uint8_t mag = e4m3_round_mag(ldexp(fabs(v), -shared));
                codes[base + i] = (uint8_t)(signbit(v) ? (0x80 | mag) : mag);
            }
        }
    }
    return 0;
}

/*
 * The value of MXFP8 weights (OCP Microscaling: element value = the E4M3
 * code's value times the block's E8M0 scale 2^(S - 127), exact in fp64 for
 * every code and every finite scale), for codes [groups][rows][cols] and
 * scales [groups][cols/32][rows]; out [groups][rows][cols] fp64.
 */
int orc_mx_dequant(const uint8_t *codes, const uint8_t *scales, int64_t groups, int64_t rows,
                   int64_t cols, double *out)
{
    if (groups < 0 || rows < 0 || cols <= 0 || cols % 32 != 0)
        return -1;
    const int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t gr = 0; gr < groups * rows; ++gr) {
        const int64_t g = gr / rows, r = gr % rows;
        for (int64_t c = 0; c < cols; ++c) {
            int S = scales[(g * nb + c / 32) * rows + r];
            out[gr * cols + c] = ldexp(e4m3_value(codes[gr * cols + c]), S - 127);
        }
    }
    return 0;
}

/* Number of OpenMP threads the oracle uses (reported beside its timings). */
int orc_num_threads(void) { return max_threads(); }

/* Sets the number of OpenMP threads of later calls from this thread (n >= 1;
 * used to time the oracle on one core beside all cores); returns the number
 * now in effect. */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#endif
    return max_threads();
}
