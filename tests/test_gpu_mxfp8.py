"""Block-scaled FP8 (MXFP8) expert weights on the GPU against the oracle.

The quantiser must reproduce the oracle's codes and scales bit for bit (an
integer decision taken on the same bf16 inputs); the layer run on MXFP8
weights must match the oracle evaluated on the exact value of those weights
(code * 2^(S-127), the MX definition, in fp64) within the bf16 layer
tolerance.

Every batch size runs the tensor cores' block-scaled FP8 MMA on MXFP8 token
rows and h, so the oracle takes the MXFP8 values of each token's input and of
each SwiGLU output too (``forward_tokens_mx``), both taking h's codes on its
bf16 value (the kernel rounds its fp32 accumulator, the oracle the fp64 h:
they differ where the two roundings do, which the tolerance covers).
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from mixture_experts_layer_warp_gb300 import binding
from mixture_experts_layer_warp_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TAU = 4e-6


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _special_weights(G=3, R=40, C=256, seed=5):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn((G, R, C), generator=g) * 0.02
    w[0, 0, :32] = 0.0                                   # an all-zero block
    w[0, 1, :32] = -0.0
    w[0, 2, :32] = 2.0 ** -130                           # bf16 subnormals
    w[0, 3, :32] = torch.linspace(-1e30, 1e30, 32)       # huge values
    w[0, 4, :32] = 256.0                                 # scale 2^0 ...
    w[0, 4, 1:32] = torch.tensor([1.0625, 1.1875, 2.125, 3.25, -1.0625, 448.0, 460.0, 464.0, 470.0, 500.0,
                                  2.0 ** -9, 3 * 2.0 ** -10, 2.0 ** -10, -(2.0 ** -10), 0.015625, 17.0,
                                  18.0, 19.0, 200.0, 208.0, 216.0, -500.0, 0.0, -0.0, 1e-3, 5e-4, 7e-4,
                                  300.0, 320.0, 352.0, 1.0])  # ... with ties and saturation
    return w.to(torch.bfloat16)


def test_quantizer_matches_the_oracle_bit_for_bit():
    w = _special_weights()
    codes, scales = binding.quantize_mxfp8(w.cuda())
    torch.cuda.synchronize()
    oc, os_ = oracle.mx_quantize(_bits(w))
    assert np.array_equal(scales.cpu().numpy(), os_), "scales differ"
    gc = codes.cpu().numpy()
    bad = np.argwhere(gc != oc)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}: {gc[tuple(bad[0])]} vs {oc[tuple(bad[0])]}"


def _quantize_experts(dev):
    w13 = [binding.quantize_mxfp8(t) for t in dev["w13"]]
    w2 = [binding.quantize_mxfp8(t) for t in dev["w2"]]
    return w13, w2


def _dequant(q):
    return [oracle.mx_dequant(c.cpu().numpy(), s.cpu().numpy()) for c, s in q]


def _check(wl, inp, y, w13_q, w2_q, rows=None, cover=False):
    host = parity.to_host_numpy(inp)
    orc = parity.oracle_routing(host, wl.k)
    set_ok, _ = parity.decided(orc["lf"], orc["ids"], TAU)
    T = host["x"].shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    if cover:
        rows = np.union1d(rows, parity.covering_tokens(orc, T, wl.k))
    rows = rows[set_ok[rows]]
    ref = oracle.forward_tokens_mx(host["x"], orc["ids"], orc["w"], _dequant(w13_q), _dequant(w2_q), rows,
              host["shared_w13"], host["shared_w2"])
    err = parity.y_error(y, ref, rows)
    assert err <= parity.Y_TOL["bf16"], f"{wl.name}: rel err {err:.3e}"
    return err


SMALL = [
    W.Workload("mx_two_micro", 8, 512, 16, 4, 256, 2),
    W.Workload("mx_shared", 13, 512, 16, 4, 128, 1, shared_inter=256),
    W.Workload("mx_one_token", 1, 256, 8, 2, 128, 1),
    W.Workload("mx_e64_k8", 16, 1024, 64, 8, 256, 1),
    # H/32 = 24 scale bytes per row (a 32-byte pitch), I = 384: the down
    # projection's last 256-K stage is half a stage, in each of two micros
    W.Workload("mx_h768_i384", 12, 768, 16, 4, 384, 2),
    # four micros of I = 128: h's scale map four deep, a half stage per micro
    W.Workload("mx_four_micro_small", 5, 256, 8, 2, 128, 4),
    # every token to the same 4 of 16 experts (12 experts untouched)
    W.Workload("mx_hot_experts_small", 12, 512, 16, 4, 128, 2, router_bias="hot"),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_mxfp8_layer_matches_the_oracle_on_dequantised_weights(wl):
    inp = W.make_inputs(wl, seed=3)
    dev = parity.to_device(inp)
    w13_q, w2_q = _quantize_experts(dev)
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=wl.T, shared_inter=wl.shared_inter)
    y = layer.forward_mxfp8(dev["x"], dev["router_w"], dev["router_bias"], w13_q, w2_q, dev["shared_w13"],
                            dev["shared_w2"])
    layer.sync()
    y2 = layer.forward_mxfp8(dev["x"], dev["router_w"], dev["router_bias"], w13_q, w2_q, dev["shared_w13"],
                             dev["shared_w2"])
    layer.sync()
    assert torch.equal(y, y2), "MXFP8 layer is not deterministic across calls"
    layer.close()
    _check(wl, inp, y, w13_q, w2_q)


def test_mxfp8_decode_workload_matches_the_oracle():
    wl = W.WORKLOADS["decode"]
    inp = W.make_inputs(wl, seed=0, device="cuda")
    w13_q, w2_q = _quantize_experts(inp)
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=wl.T)
    y = layer.forward_mxfp8(inp["x"], inp["router_w"], inp["router_bias"], w13_q, w2_q)
    layer.sync()
    layer.close()
    _check(wl, inp, y, w13_q, w2_q)


# Batches above 16 tokens: block-scaled FP8 MMA on MXFP8 token rows and h.
# Ragged expert segments, chunks split at 240 routes (an expert with ~300
# routes), every micro count, a shared expert, E = 64 with k = 8.
LARGE = [
    W.Workload("mx_large_17", 17, 256, 8, 2, 128, 1),
    W.Workload("mx_large_two_micro", 200, 512, 16, 4, 256, 2),
    W.Workload("mx_large_shared", 37, 256, 8, 2, 128, 1, shared_inter=256),
    W.Workload("mx_large_long_chunks", 600, 256, 4, 2, 128, 1),
    W.Workload("mx_large_four_micro", 64, 512, 16, 4, 128, 4),
    W.Workload("mx_large_e64_k8", 300, 1024, 64, 8, 256, 1),
    W.Workload("mx_large_wide_h", 40, 256, 8, 2, 512, 2),  # n_micro * I = 4 H
    # every token to the same 4 of 16 experts: 12 empty segments, 4 of 500
    # routes (three chunks each)
    W.Workload("mx_large_hot_experts", 500, 256, 16, 4, 128, 2, router_bias="hot"),
]


@pytest.mark.parametrize("wl", LARGE, ids=lambda w: w.name)
def test_mxfp8_large_batch_matches_the_oracle_with_mxfp8_activations(wl):
    inp = W.make_inputs(wl, seed=7)
    dev = parity.to_device(inp)
    w13_q, w2_q = _quantize_experts(dev)
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=wl.T, shared_inter=wl.shared_inter)
    y = layer.forward_mxfp8(dev["x"], dev["router_w"], dev["router_bias"], w13_q, w2_q, dev["shared_w13"],
                            dev["shared_w2"])
    layer.sync()
    y2 = layer.forward_mxfp8(dev["x"], dev["router_w"], dev["router_bias"], w13_q, w2_q, dev["shared_w13"],
                             dev["shared_w2"])
    layer.sync()
    assert torch.equal(y, y2), "MXFP8 layer is not deterministic across calls"
    layer.close()
    _check(wl, inp, y, w13_q, w2_q)


@pytest.mark.parametrize("which", ["small", "large"])
def test_mxfp8_activations_are_distinguishable_from_the_plain_layer(which):
    """The MXFP8 oracle is not the plain layer on the MX weights: on the same
    inputs the MXFP8 activations move y by far more than the kernel's error
    against forward_tokens_mx, so the parity tests tell the two readings
    apart, for the small-batch kernel and the large-batch one."""
    wl = SMALL[0] if which == "small" else LARGE[1]
    inp = W.make_inputs(wl, seed=7)
    dev = parity.to_device(inp)
    w13_q, w2_q = _quantize_experts(dev)
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=wl.T)
    y = layer.forward_mxfp8(dev["x"], dev["router_w"], dev["router_bias"], w13_q, w2_q)
    layer.sync()
    layer.close()
    host = parity.to_host_numpy(inp)
    orc = parity.oracle_routing(host, wl.k)
    set_ok, _ = parity.decided(orc["lf"], orc["ids"], TAU)
    rows = np.arange(wl.T)[set_ok]
    args = (host["x"], orc["ids"], orc["w"], _dequant(w13_q), _dequant(w2_q), rows)
    e_mx = parity.y_error(y, oracle.forward_tokens_mx(*args), rows)
    e_plain = parity.y_error(y, oracle.forward_tokens(*args), rows)
    assert e_mx < e_plain / 3, f"kernel vs MX oracle {e_mx:.3e}, vs plain oracle {e_plain:.3e}"


def test_mxfp8_denoise_workload_matches_the_oracle():
    """The two-micro denoise layer (T=4096, H=4096, E=64, k=8, I=768) at full
    size, in the launch configuration the benchmark times, on the tokens that
    cover every chunk of every expert segment."""
    wl = W.WORKLOADS["denoise_multi_micro"]
    inp = W.make_inputs(wl, seed=0, device="cuda")
    w13_q, w2_q = _quantize_experts(inp)
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=wl.T)
    y = layer.forward_mxfp8(inp["x"], inp["router_w"], inp["router_bias"], w13_q, w2_q)
    layer.sync()
    layer.close()
    _check(wl, inp, y, w13_q, w2_q, rows=np.arange(0, wl.T, 512), cover=True)


def test_mxfp8_async_host_calls_match_device_calls():
    """moe_forward_mxfp8_host_async on both batch sizes, back to back on pinned
    buffers, equals moe_forward_mxfp8 on the same inputs."""
    wl = W.Workload("mx_host_async", 120, 512, 16, 4, 256, 1)
    wts = parity.to_device(W.make_inputs(wl, seed=2))
    w13_q, w2_q = _quantize_experts(wts)
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, 1, max_tokens=wl.T)
    sizes = [8, 120, 16, 70]
    xs = [W.make_inputs(wl, seed=40 + i, T=T, experts=False)["x"].pin_memory() for i, T in enumerate(sizes)]
    ys = [torch.empty_like(x).pin_memory() for x in xs]
    for x, y in zip(xs, ys):
        layer.forward_mxfp8(x, wts["router_w"], None, w13_q, w2_q, out=y, host_async=True)
    layer.sync()
    for T, x, y in zip(sizes, xs, ys):
        ref = layer.forward_mxfp8(x.cuda(), wts["router_w"], None, w13_q, w2_q)
        layer.sync()
        assert torch.equal(y, ref.cpu()), f"T={T}: async host result differs from the device call"
    layer.close()


def test_weight_scales_below_the_f16_range_are_exact():
    """w2 scaled by 2^-14: its blocks get scales near 2^-26 (below f16's
    range); the block-scaled MMA applies them exactly, so y (made by w2) must
    still match the exact MX weight values."""
    wl = W.Workload("mx_tiny_w2", 8, 512, 16, 4, 256, 1)
    inp = W.make_inputs(wl, seed=4)
    inp["w2"] = [(t.float() * 2.0 ** -14).to(torch.bfloat16) for t in inp["w2"]]
    dev = parity.to_device(inp)
    w13_q, w2_q = _quantize_experts(dev)
    assert (w2_q[0][1] < 127 - 24).float().mean() > 0.5, "the test needs scales below 2^-24"
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, 1, max_tokens=wl.T)
    y = layer.forward_mxfp8(dev["x"], dev["router_w"], None, w13_q, w2_q)
    layer.sync()
    layer.close()
    _check(wl, inp, y, w13_q, w2_q)


def test_mxfp8_and_bf16_calls_back_to_back_match_isolated_calls():
    """MXFP8 calls of both sizes interleaved with bf16 calls of both sizes on
    one handle and stream, no sync in between, equal the same calls run alone."""
    base = W.Workload("mx_mix", 200, 512, 16, 4, 256, 1)
    wts = parity.to_device(W.make_inputs(base, seed=0))
    w13_q, w2_q = _quantize_experts(wts)
    layer = binding.MoELayer(base.H, base.E, base.k, base.I, 1, max_tokens=base.T)
    plan = [("mx", 8), ("bf16", 200), ("mx", 16), ("mx", 200), ("bf16", 8), ("mx", 1), ("bf16", 200), ("mx", 150),
            ("mx", 8)]
    xs = [W.make_inputs(base, seed=60 + i, T=T, experts=False)["x"].cuda() for i, (_, T) in enumerate(plan)]

    def call(kind, x, out=None):
        if kind == "mx":
            return layer.forward_mxfp8(x, wts["router_w"], None, w13_q, w2_q, out=out)
        return layer.forward(x, wts["router_w"], None, wts["w13"], wts["w2"], out=out)

    outs = [torch.empty_like(x) for x in xs]
    for (kind, _), x, y in zip(plan, xs, outs):
        call(kind, x, y)
    layer.sync()
    for (kind, T), x, y in zip(plan, xs, outs):
        ref = call(kind, x)
        layer.sync()
        assert torch.equal(y, ref), f"{kind} T={T}: back-to-back result differs from the isolated call"
    layer.close()
