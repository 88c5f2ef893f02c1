"""Checks that pin the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an oracle library handle (``None`` = the real
oracle; the mutation test passes builds of the oracle with a planted mistake)
and raises ``AssertionError`` when the oracle disagrees with what the pages or
the mathematics fix:

* hand-derived worked examples with closed-form values (``tests/golden``);
* brute force over all k-subsets for the top-k selection;
* library routines for special cases: ``scipy.special.softmax`` for k = E,
  ``np.argsort(kind="stable")`` for the route sort, ``np.bincount`` +
  ``np.cumsum`` for the offsets;
* identities the pages state: concatenated micro-shards equal the unsharded
  expert ("HunyuanImage3 Hybrid Parallelism" section 5), two single-micro
  dispatches summed equal the multi-micro call (section 10.3), the
  per-token definition equals the gather/segment/finalize organisation
  (section 6.1);
* invariants: Sum_j w = 1, distinct ids, bijective permutation.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f32(a):
    return np.asarray(a, dtype=np.float32)


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / den)


# ---------------------------------------------------------------- routing pins
def pin_routing_worked_example(lib=None):
    g = _golden("routing_worked_example.json")
    lg = oracle.logits(_f32(g["x"]), _f32(g["router_w"]), _f32(g["router_bias"]), lib=lib)
    ids, w, probs = oracle.route(lg, g["k"], return_probs=True, lib=lib)
    assert ids.tolist() == g["expect_ids"], (ids.tolist(), g["expect_ids"])
    assert np.allclose(w, g["expect_w"], rtol=0, atol=1e-7), w
    assert np.allclose(probs[2], g["expect_probs_token2"], rtol=0, atol=1e-7), probs[2]


def pin_fp32_gate_decision(lib=None):
    g = _golden("fp32_gate_decision.json")
    lg = oracle.logits(_f32(g["x"]), _f32(g["router_w"]), lib=lib)
    ids1, _ = oracle.route(lg, 1, lib=lib)
    ids2, w2 = oracle.route(lg, 2, lib=lib)
    assert ids1.tolist() == g["expect_ids_k1"], ids1
    assert ids2.tolist() == g["expect_ids_k2"], ids2
    assert np.allclose(w2, g["expect_w_k2"], rtol=0, atol=1e-12), w2


def _brute_topk(l, k):
    """The unique k-subset S with every member ranked above every non-member
    under (larger logit, then lower index), listed in that rank order."""
    E = len(l)
    key = lambda e: (-l[e], e)  # noqa: E731
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(key(a) < key(b) for a in S for b in rest):
            found.append(sorted(S, key=key))
    assert len(found) == 1
    return found[0]


def pin_topk_brute_force(lib=None):
    rng = np.random.default_rng(11)
    for trial in range(60):
        T = int(rng.integers(1, 7))
        E = int(rng.integers(1, 7))
        k = int(rng.integers(1, min(E, 3) + 1))
        H = int(rng.integers(1, 5))
        if trial % 2:  # integer grid: exact ties are common
            x = _f32(rng.integers(-2, 3, (T, H)))
            wr = _f32(rng.integers(-1, 2, (E, H)))
        else:
            x = _f32(rng.standard_normal((T, H)))
            wr = _f32(rng.standard_normal((E, H)))
        lg = oracle.logits(x, wr, lib=lib)
        ids, w = oracle.route(lg, k, lib=lib)
        lf = lg.astype(np.float32).astype(np.float64)
        for t in range(T):
            want = _brute_topk(lf[t], k)
            assert ids[t].tolist() == want, (t, ids[t], want, lf[t])
            # renormalised softmax of the chosen subset: k = 1 gives 1; a pair
            # with logit gap d gives sigma(d) and 1 - sigma(d)
            if k == 1:
                assert abs(w[t, 0] - 1.0) < 1e-15
            if k == 2:
                d = lf[t, want[0]] - lf[t, want[1]]
                assert abs(w[t, 0] - scipy.special.expit(d)) < 1e-12
            assert abs(w[t].sum() - 1.0) < 1e-12


def pin_k_equals_E_is_softmax(lib=None):
    rng = np.random.default_rng(5)
    x = _f32(rng.standard_normal((9, 7)))
    wr = _f32(rng.standard_normal((5, 7)))
    b = _f32(rng.standard_normal(5))
    lg = oracle.logits(x, wr, b, lib=lib)
    ids, w = oracle.route(lg, 5, lib=lib)
    lf = lg.astype(np.float32).astype(np.float64)
    ref = scipy.special.softmax(lf, axis=1)
    got = np.zeros_like(ref)
    for t in range(9):
        got[t, ids[t]] = w[t]
    assert _rel(got, ref) < 1e-12
    # the logits themselves: a library matmul of the widened inputs plus bias
    assert _rel(lg, x.astype(np.float64) @ wr.astype(np.float64).T + b) < 1e-12


# ------------------------------------------------------------ permutation pins
def pin_permutation_library(lib=None):
    rng = np.random.default_rng(3)
    for T, k, E in [(1, 1, 1), (7, 2, 5), (33, 8, 64), (100, 3, 4), (0, 2, 3)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) \
            if T else np.zeros((0, k), np.int32)
        counts, offsets, perm, inv = oracle.permute(ids, E, lib=lib)
        flat = ids.ravel()
        assert counts.tolist() == np.bincount(flat, minlength=E).tolist()
        assert offsets.tolist() == [0] + np.cumsum(np.bincount(flat, minlength=E)).tolist()
        assert perm.tolist() == np.argsort(flat, kind="stable").tolist()
        assert np.array_equal(inv[perm], np.arange(T * k))
        assert sorted(perm.tolist()) == list(range(T * k))


# -------------------------------------------------------------------- FFN pins
def pin_swiglu_worked_example(lib=None):
    g = _golden("swiglu_expert_worked_example.json")
    x = _f32(g["x"])
    ids = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1))
    y = oracle.forward_tokens(x, ids, w, [_f32(g["w13"])], [_f32(g["w2"])], lib=lib)
    assert _rel(y, g["expect_y"]) < 1e-12, y
    ym = oracle.forward_tokens(x, ids, w, [_f32(a) for a in g["micro_w13"]],
                               [_f32(a) for a in g["micro_w2"]], lib=lib)
    assert _rel(ym, g["expect_y"]) < 1e-12, ym


def pin_layer_worked_example(lib=None):
    g = _golden("layer_worked_example.json")
    out = oracle.layer(_f32(g["x"]), _f32(g["router_w"]), None, [_f32(g["w13"])],
                       [_f32(g["w2"])], g["k"], lib=lib)
    assert out["ids"].tolist() == g["expect_ids"], out["ids"]
    assert _rel(out["y"], g["expect_y"]) < 1e-12, out["y"]
    yp = oracle.forward_permuted(_f32(g["x"]), out["w"], out["offsets"], out["perm"],
                                 out["inv"], [_f32(g["w13"])], [_f32(g["w2"])], lib=lib)
    assert _rel(yp, g["expect_y"]) < 1e-12, yp


def _rand_layer(rng, T, H, E, k, I, M, Is=0):
    x = _f32(rng.standard_normal((T, H)))
    wr = _f32(rng.standard_normal((E, H)) / math.sqrt(H))
    w13 = [_f32(rng.standard_normal((E, 2 * I, H)) / math.sqrt(H)) for _ in range(M)]
    w2 = [_f32(rng.standard_normal((E, H, I)) / math.sqrt(I)) for _ in range(M)]
    sw13 = _f32(rng.standard_normal((2 * Is, H)) / math.sqrt(H)) if Is else None
    sw2 = _f32(rng.standard_normal((H, Is)) / math.sqrt(Is)) if Is else None
    return x, wr, w13, w2, sw13, sw2


def pin_per_token_equals_permuted(lib=None):
    rng = np.random.default_rng(21)
    x, wr, w13, w2, sw13, sw2 = _rand_layer(rng, 23, 16, 6, 3, 8, 2, Is=12)
    out = oracle.layer(x, wr, None, w13, w2, 3, sw13, sw2, lib=lib)
    yp = oracle.forward_permuted(x, out["w"], out["offsets"], out["perm"], out["inv"],
                                 w13, w2, sw13, sw2, lib=lib)
    assert _rel(yp, out["y"]) < 1e-12


def pin_micro_concat_identity(lib=None):
    """Two micro-shards equal one unsharded expert with I_full = 2I (blog section 5:
    the micro-major pack holds the expert's intermediate dimension split in two)."""
    rng = np.random.default_rng(8)
    T, H, E, k, I = 11, 12, 4, 2, 5
    x, wr, w13, w2, _, _ = _rand_layer(rng, T, H, E, k, I, 2)
    full13 = np.concatenate([w13[0][:, :I], w13[1][:, :I], w13[0][:, I:], w13[1][:, I:]], axis=1)
    full2 = np.concatenate([w2[0], w2[1]], axis=2)
    a = oracle.layer(x, wr, None, w13, w2, k, lib=lib)
    b = oracle.layer(x, wr, None, [full13], [full2], k, lib=lib)
    assert np.array_equal(a["ids"], b["ids"])
    assert _rel(a["y"], b["y"]) < 1e-12


def pin_two_dispatch_identity(lib=None):
    """Summing two single-micro layer calls equals one multi-micro call (blog
    section 10.3, the two-dispatch path adds the two outputs)."""
    rng = np.random.default_rng(9)
    x, wr, w13, w2, _, _ = _rand_layer(rng, 13, 10, 5, 2, 6, 2)
    both = oracle.layer(x, wr, None, w13, w2, 2, lib=lib)["y"]
    one = oracle.layer(x, wr, None, w13[:1], w2[:1], 2, lib=lib)["y"]
    two = oracle.layer(x, wr, None, w13[1:], w2[1:], 2, lib=lib)["y"]
    assert _rel(one + two, both) < 1e-12


def pin_degenerate_experts(lib=None):
    rng = np.random.default_rng(10)
    T, H, E, k, I = 9, 8, 4, 2, 6
    x, wr, w13, w2, _, _ = _rand_layer(rng, T, H, E, k, I, 1)
    # gate rows zero -> silu(0) = 0 -> y = 0; up rows zero -> y = 0
    for half in (slice(0, I), slice(I, 2 * I)):
        z = w13[0].copy()
        z[:, half] = 0
        y = oracle.layer(x, wr, None, [z], w2, k, lib=lib)["y"]
        assert np.abs(y).max() == 0.0
    # every expert identical -> routing weights sum to one -> y = the single expert
    same13 = np.repeat(w13[0][:1], E, axis=0)
    same2 = np.repeat(w2[0][:1], E, axis=0)
    y = oracle.layer(x, wr, None, [same13], [same2], k, lib=lib)["y"]
    y1 = oracle.forward_tokens(x, np.zeros((T, 1), np.int32), np.ones((T, 1)),
                               [same13], [same2], lib=lib)
    assert _rel(y, y1) < 1e-12


def pin_textbook_glu(lib=None):
    """k = 1 and E = 1 reduce the layer to a two-layer GLU MLP, evaluated here
    with library matmuls and scipy's logistic function."""
    rng = np.random.default_rng(12)
    T, H, I = 6, 10, 7
    x, wr, w13, w2, _, _ = _rand_layer(rng, T, H, 1, 1, I, 1)
    y = oracle.layer(x, wr, None, w13, w2, 1, lib=lib)["y"]
    X = x.astype(np.float64)
    G = w13[0][0, :I].astype(np.float64)
    U = w13[0][0, I:].astype(np.float64)
    D = w2[0][0].astype(np.float64)
    gx = X @ G.T
    ref = ((gx * scipy.special.expit(gx)) * (X @ U.T)) @ D.T
    assert _rel(y, ref) < 1e-12


def pin_shared_expert_added_unscaled(lib=None):
    rng = np.random.default_rng(13)
    T, H, E, k, I, Is = 8, 10, 4, 2, 5, 9
    x, wr, w13, w2, sw13, sw2 = _rand_layer(rng, T, H, E, k, I, 1, Is)
    with_s = oracle.layer(x, wr, None, w13, w2, k, sw13, sw2, lib=lib)["y"]
    without = oracle.layer(x, wr, None, w13, w2, k, lib=lib)["y"]
    X = x.astype(np.float64)
    gx = X @ sw13[:Is].astype(np.float64).T
    s = ((gx * scipy.special.expit(gx)) * (X @ sw13[Is:].astype(np.float64).T)) @ \
        sw2.astype(np.float64).T
    assert _rel(with_s - without, s) < 1e-10


def pin_bf16_widening(lib=None):
    """bf16 inputs are widened exactly: the same values given as fp32 and as
    bf16 bit patterns produce identical results."""
    rng = np.random.default_rng(14)
    x, wr, w13, w2, _, _ = _rand_layer(rng, 5, 8, 3, 2, 4, 1)

    def bits(a):
        u = np.ascontiguousarray(a, np.float32).view(np.uint32)
        return (u >> 16).astype(np.uint16)

    def back(b):
        return (b.astype(np.uint32) << 16).view(np.float32)

    xb, wrb = bits(x), bits(wr)
    w13b, w2b = [bits(w13[0])], [bits(w2[0])]
    a = oracle.layer(xb, wrb, None, w13b, w2b, 2, lib=lib)
    b = oracle.layer(back(xb), back(wrb), None, [back(w13b[0])], [back(w2b[0])], 2, lib=lib)
    assert np.array_equal(a["ids"], b["ids"])
    assert np.array_equal(a["y"], b["y"])


# ------------------------------------------------------------ MXFP8 weights
# The block-scaled FP8 expert weights follow the OCP Microscaling (MX) MXFP8
# format; the pins below hold the oracle's quantiser and dequantiser to torch's
# float8_e4m3fn conversions and numpy's ldexp (library routines), and to
# closed-form values of the shared-exponent rule.

def _e4m3_torch_codes(v):
    import torch
    return torch.tensor(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_torch_values():
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def _blocks_at_unit_scale(vals):
    """Blocks of 32 whose first element (256) fixes the shared exponent at 0."""
    vals = np.asarray(vals, np.float32)
    n = -(-vals.size // 31)
    w = np.zeros((n, 32), np.float32)
    w[:, 0] = 256.0
    w[:, 1:].flat[:vals.size] = vals
    return w


def pin_mx_e4m3_rounding_matches_torch(lib=None):
    rng = np.random.default_rng(7)
    rep = _e4m3_torch_values()[:127]                      # the non-negative finite values
    mids = (rep[:-1] + rep[1:]) / 2                       # exact ties
    vals = np.concatenate([rep, mids, rng.uniform(0, 448, 2000), rng.uniform(0, 2.0 ** -6, 500),
                           np.array([448.0, 455.0, 463.9])]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    w = _blocks_at_unit_scale(vals)
    codes, scales = oracle.mx_quantize(w, lib=lib)
    assert (scales == 127).all(), "the leading 256 must fix the scale at 2^0"
    got = codes[:, 1:].reshape(-1)[:vals.size]
    assert np.array_equal(got, _e4m3_torch_codes(vals)), "E4M3 rounding differs from torch's"
    sat = np.array([470.0, 500.0, 511.0, -480.0], np.float32)
    c2, _ = oracle.mx_quantize(_blocks_at_unit_scale(sat), lib=lib)
    assert list(c2[0, 1:5]) == [0x7E, 0x7E, 0x7E, 0xFE], "values above 448 must saturate"


def pin_mx_e4m3_decode_matches_torch(lib=None):
    codes = np.arange(256, dtype=np.uint8)
    finite = codes[(codes & 0x7F) != 0x7F]
    c = np.zeros((1, 1, 256), np.uint8)
    c[0, 0, :finite.size] = finite
    s = np.full((1, 8, 1), 127, np.uint8)
    got = oracle.mx_dequant(c, s, lib=lib)[0, 0, :finite.size]
    want = _e4m3_torch_values()[finite]
    assert np.array_equal(got, want), "E4M3 decoding differs from torch's"


def pin_mx_dequant_is_the_exact_product(lib=None):
    """A dequantised weight is exactly the E4M3 code's value (torch's
    float8_e4m3fn decode) times 2^(S-127) (numpy's ldexp), the MX definition,
    for every finite code under every finite E8M0 scale S = 0..254, including
    the extremes 2^-127 and 2^127 where no 16-bit float could hold the product;
    plus two values written out: the largest code 0x7E at S = 127 is 448, the
    smallest subnormal code 0x01 at S = 0 is 2^-9 * 2^-127."""
    val = _e4m3_torch_values()
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    Ss = np.arange(0, 255)
    c = np.zeros((1, 1, 256 * Ss.size), np.uint8)
    s = np.zeros((1, 8 * Ss.size, 1), np.uint8)
    for b, S in enumerate(Ss):
        c[0, 0, 256 * b:256 * b + finite.size] = finite
        s[0, 8 * b:8 * b + 8, 0] = S
    got = oracle.mx_dequant(c, s, lib=lib)[0, 0]
    for b, S in enumerate(Ss):
        want = np.ldexp(val[finite], int(S) - 127)
        g = got[256 * b:256 * b + finite.size]
        assert np.array_equal(g, want), f"dequantised value is not code * 2^(S-127) at S={S}"
    one = lambda code, S: oracle.mx_dequant(np.full((1, 32), code, np.uint8), np.full((1, 1), S, np.uint8),  # noqa: E731
                                            lib=lib)[0, 0]
    assert one(0x7E, 127) == 448.0 and one(0xFE, 127) == -448.0
    assert one(0x01, 0) == 2.0 ** -136


def pin_mx_shared_exponent_rule(lib=None):
    """Closed forms of the MX rule: shared = floor(log2 amax) - 8 (E4M3's largest
    exponent), clamped to [-127, 127]; an all-zero block gets S = 127; scales are
    laid out [G][C/32][R]."""
    cases = [(1.0, 119), (0.75, 118), (448.0, 127), (511.0, 127), (512.0, 128), (2.0 ** -130, 0),
             (3.0e38, 246)]
    w = np.zeros((len(cases) + 1, 32), np.float32)
    for i, (amax, _) in enumerate(cases):
        w[i, 5] = -amax
        w[i, 9] = amax / 4
    codes, scales = oracle.mx_quantize(w, lib=lib)
    for i, (amax, S) in enumerate(cases):
        assert scales[0, i] == S, f"amax {amax}: S {scales[0, i]} != {S}"
    assert scales[0, -1] == 127 and not codes[-1].any(), "an all-zero block: S = 127, codes 0"
    # layout: a distinct amax at (g, r, block) must land in scales[g, block, r]
    G, R, C = 2, 3, 96
    w3 = np.full((G, R, C), 1.0, np.float32)
    w3[1, 2, 64 + 7] = 8.0
    _, s3 = oracle.mx_quantize(w3, lib=lib)
    assert s3.shape == (G, C // 32, R)
    assert s3[1, 2, 2] == 122 and (np.delete(s3.reshape(-1), (1 * 3 + 2) * 3 + 2) == 119).all()


def pin_mx_roundtrip_error_bound(lib=None):
    """|dequant(quant(w)) - w| is within half an E4M3 step of w, except
    saturated elements, which become +-448 * 2^shared exactly."""
    rng = np.random.default_rng(3)
    w = _f32(rng.normal(0, 0.02, (4, 64, 256))).astype(np.float32)
    codes, scales = oracle.mx_quantize(w, lib=lib)
    deq = oracle.mx_dequant(codes, scales, lib=lib)
    shared = np.repeat(scales.astype(np.int64) - 127, 32, axis=1).transpose(0, 2, 1)  # [G][R][C]
    unit = np.ldexp(1.0, shared)
    u = np.abs(w.astype(np.float64)) / unit
    sat = u >= 448.0
    step = np.where(u < 2.0 ** -6, 2.0 ** -9, np.ldexp(1.0, np.floor(np.log2(np.maximum(u, 2.0 ** -6))).astype(int) - 3))
    bound = (step / 2) * unit
    err = np.abs(deq - w.astype(np.float64))
    assert (err[~sat] <= bound[~sat]).all(), "quantisation error beyond half a step"
    assert np.array_equal(np.abs(deq[sat]), 448.0 * unit[sat])


def _mx_value_torch(v):
    """MXFP8 value of v along its last axis (blocks of 32) from library
    routines: numpy frexp for the shared exponent, torch's float8_e4m3fn cast
    (nearest, ties to even) for the code, saturated at 448."""
    import torch
    v = np.asarray(v, np.float64)
    b = v.reshape(-1, 32)
    amax = np.abs(b).max(axis=1)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    shared = np.clip(np.where(amax > 0, ex - 1 - 8, 0), -127, 127)[:, None]
    u = np.minimum(np.abs(b) * np.ldexp(1.0, -shared), 448.0)
    q = torch.tensor(u).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return (np.sign(b) * q * np.ldexp(1.0, shared)).reshape(v.shape)


def _bf16_value_torch(v):
    """bf16 value of fp64 v from torch's cast. torch converts fp64 through fp32,
    which equals the direct rounding unless the fp32 value is itself a bf16
    tie (low 16 bits 0x8000); the caller's values are checked to hold none."""
    import torch
    v = np.asarray(v, np.float64)
    bits = v.astype(np.float32).view(np.uint32)
    assert not ((bits & 0xFFFF) == 0x8000).any(), "an fp32 tie: torch's cast would round twice"
    return torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()


def pin_bf16_rounding(lib=None):
    """bf16_round against the format's closed forms (8 significant bits,
    ties to even, subnormal step 2^-133, overflow past (2 - 2^-7) 2^127) and
    torch's cast on random values of every magnitude."""
    t = 2.0 ** -8
    cases = {
        1.0 + t: 1.0,                      # a tie: to the even neighbour 1
        1.0 + 3 * t: 1.0 + 4 * t,          # a tie: to the even neighbour 1 + 2^-6
        1.0 + t + 2.0 ** -30: 1.0 + 2 * t,  # just past the tie (lost in fp32)
        -(1.0 + t + 2.0 ** -30): -(1.0 + 2 * t),
        255.5: 256.0,                      # 8 significant bits: 255.5 is a tie, 256 even
        254.5: 254.0,
        2.0 ** -133 * 0.5: 0.0,            # half the smallest subnormal: tie to 0
        2.0 ** -133 * 0.75: 2.0 ** -133,
        2.0 ** -133 * 3.5: 2.0 ** -131,     # 3.5 steps: tie to 4
        (2.0 - 2.0 ** -7) * 2.0 ** 127: (2.0 - 2.0 ** -7) * 2.0 ** 127,
        (2.0 - 2.0 ** -9) * 2.0 ** 127: np.inf,  # rounds up past the largest finite value
        0.0: 0.0,
    }
    got = oracle.bf16_round(np.array(list(cases)), lib=lib)
    assert np.array_equal(got, np.array(list(cases.values()))), f"bf16 closed forms: {got}"
    rng = np.random.default_rng(5)
    v = rng.normal(0, 1, 4000) * np.ldexp(1.0, rng.integers(-140, 120, 4000))
    v = v[np.abs(v) >= 2.0 ** -126]
    v = v[(v.astype(np.float32).view(np.uint32) & 0xFFFF) != 0x8000]  # where torch's cast rounds once
    assert np.array_equal(oracle.bf16_round(v, lib=lib), _bf16_value_torch(v)), "bf16 rounding differs from torch"


def pin_mx_activation_forward_matches_library_rounding(lib=None):
    """forward_tokens_mx: each token's routed input replaced by its MXFP8 value
    along H, each expert's SwiGLU output rounded to bf16 and then replaced by
    its MXFP8 value along I (per micro), the shared expert on the unrounded
    input; checked against the same layer built from library routines
    (torch's bf16 and E4M3 casts for every rounding)."""
    rng = np.random.default_rng(21)
    T, H, E, k, I, M, Is = 5, 64, 3, 2, 64, 2, 32
    x = _f32(rng.normal(0, 1.0, (T, H))).astype(np.float32)
    w13 = [rng.normal(0, 0.2, (E, 2 * I, H)) for _ in range(M)]
    w2 = [rng.normal(0, 0.2, (E, H, I)) for _ in range(M)]
    sw13 = _f32(rng.normal(0, 0.2, (2 * Is, H))).astype(np.float32)
    sw2 = _f32(rng.normal(0, 0.2, (H, Is))).astype(np.float32)
    ids = np.array([[0, 2], [1, 0], [2, 1], [0, 1], [2, 0]], np.int32)
    w = rng.uniform(0.2, 0.8, (T, k))
    got = oracle.forward_tokens_mx(x, ids, w, w13, w2, None, sw13, sw2, lib=lib)
    silu = lambda z: z / (1.0 + np.exp(-z))  # noqa: E731
    xs = x.astype(np.float64)
    want = np.zeros((T, H))
    for t in range(T):
        xq = _mx_value_torch(xs[t])
        for j in range(k):
            e = ids[t, j]
            for m in range(M):
                g = w13[m][e, :I] @ xq
                u = w13[m][e, I:] @ xq
                want[t] += w[t, j] * (w2[m][e] @ _mx_value_torch(_bf16_value_torch(silu(g) * u)))
        gs = sw13[:Is].astype(np.float64) @ xs[t]
        us = sw13[Is:].astype(np.float64) @ xs[t]
        want[t] += sw2.astype(np.float64) @ (silu(gs) * us)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max()), "MX activation forward differs"
    # rounding to MX values is idempotent: inputs already on the grid are unchanged
    xg = _mx_value_torch(xs).astype(np.float32)
    assert np.array_equal(_mx_value_torch(xg.astype(np.float64)), xg.astype(np.float64))
    plain = oracle.forward_tokens(xg, ids, w, w13, w2, None, None, None, lib=lib)
    mxv = oracle.forward_tokens_mx(xg, ids, w, w13, w2, None, None, None, lib=lib)
    assert not np.allclose(plain, mxv, rtol=1e-6), "the SwiGLU outputs must be rounded too"


def pin_forward_accepts_fp64_weights(lib=None):
    """The fp64 weight path (used with dequantised weights) equals the fp32 path
    on the same values."""
    rng = np.random.default_rng(11)
    x, wr, w13, w2, sw13, sw2 = _rand_layer(rng, 6, 64, 4, 2, 32, 2, Is=32)
    lg = oracle.logits(x, wr, None, lib=lib)
    ids, w = oracle.route(lg, 2, lib=lib)
    y32 = oracle.forward_tokens(x, ids, w, w13, w2, None, sw13, sw2, lib=lib)
    y64 = oracle.forward_tokens(x, ids, w, [a.astype(np.float64) for a in w13], [a.astype(np.float64) for a in w2],
                                None, sw13, sw2, lib=lib)
    assert np.array_equal(y32, y64)


ALL_PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_")]
