"""The whole layer (moe_forward) against the fp64 oracle.

Small shapes are compared on every token; the five workloads at full size on a
sample of tokens that puts a checked row into every 128-row block of every
expert segment (the oracle evaluates the per-token definition for those).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import parity
from mixture_experts_layer_warp_gb300 import binding
from mixture_experts_layer_warp_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TAU = 4e-6


def _layer(wl: W.Workload, T=None):
    return binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=T or wl.T,
                            shared_inter=wl.shared_inter, dtype=wl.torch_dtype)


def _forward(layer, dev):
    y = layer.forward(dev["x"], dev["router_w"], dev["router_bias"], dev["w13"], dev["w2"],
                      dev["shared_w13"], dev["shared_w2"])
    layer.sync()
    return y


def _check(wl, inp, y, rows=None, cover: bool = False):
    host = parity.to_host_numpy(inp)
    orc = parity.oracle_routing(host, wl.k)
    set_ok, _ = parity.decided(orc["lf"], orc["ids"], TAU if wl.dtype == "bf16" else 0.0)
    T = host["x"].shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    if cover:
        rows = np.union1d(rows, parity.covering_tokens(orc, T, wl.k))
    rows = rows[set_ok[rows]]
    ref = oracle.forward_tokens(host["x"], orc["ids"], orc["w"], host["w13"], host["w2"], rows,
                                host["shared_w13"], host["shared_w2"])
    err = parity.y_error(y, ref, rows)
    assert err <= parity.Y_TOL[wl.dtype], f"{wl.name}: rel err {err:.3e}"
    return err


SMALL = [
    W.Workload("bf16_two_micro", 300, 256, 8, 2, 128, 2),
    W.Workload("bf16_one_token", 1, 256, 8, 2, 128, 1),
    W.Workload("bf16_small_batch_shared", 13, 512, 16, 4, 128, 2, shared_inter=256),
    W.Workload("bf16_small_batch_e64", 16, 4096, 64, 8, 768, 1),
    W.Workload("bf16_17_tokens", 17, 512, 8, 2, 256, 2, shared_inter=128),
    W.Workload("bf16_e64_k8_ragged", 129, 512, 64, 8, 256, 1),
    W.Workload("bf16_shared", 257, 256, 16, 4, 128, 2, shared_inter=256),
    W.Workload("bf16_four_micro", 70, 512, 8, 3, 128, 4),
    W.Workload("bf16_skew_bias", 600, 256, 64, 8, 128, 1, router_bias="log_zipf"),
    # every token to the same 4 of 16 experts: 12 empty segments, 4 of 700
    # routes (three chunks each); and the same at a decode-sized batch
    W.Workload("bf16_hot_experts", 700, 256, 16, 4, 128, 2, shared_inter=128, router_bias="hot"),
    W.Workload("bf16_hot_experts_small", 12, 512, 16, 4, 128, 2, router_bias="hot"),
    # groups of more than 16 row blocks (about 3000 routes per expert; a 47-block
    # dense shared segment): the large GEMM walks their row blocks in chunks
    W.Workload("bf16_long_groups", 6000, 256, 4, 2, 128, 2, shared_inter=128),
    W.Workload("f32_tiny_multi_shared", 45, 128, 4, 2, 64, 2, shared_inter=64, dtype="f32"),
    W.WORKLOADS["tiny_fp32"],
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_small_layer_matches_oracle_on_every_token(wl):
    inp = W.make_inputs(wl, seed=1)
    layer = _layer(wl)
    y = _forward(layer, parity.to_device(inp))
    err = _check(wl, inp, y)
    print(f"{wl.name}: rel err {err:.3e}")
    layer.close()


@pytest.mark.parametrize("name", ["decode", "denoise_multi_micro", "skewed", "cfg_shared"])
def test_workload_matches_oracle_on_sampled_tokens(name):
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl, seed=0, device="cuda")
    layer = _layer(wl)
    y = _forward(layer, inp)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, wl.T - 1], rng.integers(0, wl.T, 30)]))
    layer.close()
    del layer
    err = _check(wl, inp, y, rows, cover=True)
    print(f"{name}: rel err {err:.3e}")


def test_bitwise_deterministic_across_calls():
    wl = W.Workload("det", 513, 512, 64, 8, 256, 2, shared_inter=128)
    dev = parity.to_device(W.make_inputs(wl, seed=2))
    layer = _layer(wl)
    a = _forward(layer, dev).clone()
    b = _forward(layer, dev)
    assert torch.equal(a, b)
    layer.close()


@pytest.mark.parametrize("T", [8, 200])
def test_two_dispatches_sum_to_the_multi_micro_call(T):
    """Two single-micro layer calls, the second accumulating into the first's
    output, equal one multi-micro call ("HunyuanImage3 Hybrid Parallelism",
    section 10.3), up to bf16 rounding of the intermediate y."""
    wl = W.Workload("mm", T, 256, 8, 2, 128, 2)
    dev = parity.to_device(W.make_inputs(wl, seed=3))
    both = _forward(_layer(wl), dev).float()
    one = W.Workload("m1", T, 256, 8, 2, 128, 1)
    l0, l1 = _layer(one), _layer(one)
    l1.set_accumulate(True)
    y = l0.forward(dev["x"], dev["router_w"], None, dev["w13"][:1], dev["w2"][:1])
    l1.forward(dev["x"], dev["router_w"], None, dev["w13"][1:], dev["w2"][1:], out=y)
    l1.sync()
    err = (y.float() - both).abs().max().item() / both.abs().max().item()
    assert err < 1e-2
    # and the two-dispatch output against the oracle's multi-micro layer
    _check(wl, W.make_inputs(wl, seed=3), y)


def test_two_dispatches_at_denoise_size_match_the_oracle():
    """The pages' two-dispatch form ("HunyuanImage3 Hybrid Parallelism",
    section 10.3) of the two-micro denoise workload at full size: one
    single-micro layer call per micro-shard, the second accumulating into the
    first's y, against the oracle's multi-micro layer on covering tokens."""
    wl = W.WORKLOADS["denoise_multi_micro"]
    inp = W.make_inputs(wl, seed=0, device="cuda")
    one = W.Workload("m1", wl.T, wl.H, wl.E, wl.k, wl.I, 1, router_init=wl.router_init)
    l0, l1 = _layer(one), _layer(one)
    l1.set_accumulate(True)
    y = l0.forward(inp["x"], inp["router_w"], None, inp["w13"][:1], inp["w2"][:1])
    l1.forward(inp["x"], inp["router_w"], None, inp["w13"][1:], inp["w2"][1:], out=y)
    l1.sync()
    l0.close()
    l1.close()
    err = _check(wl, inp, y, [0], cover=True)
    print(f"two dispatches, denoise: rel err {err:.3e}")


@pytest.mark.parametrize("wl", [W.Workload("acc_small", 12, 512, 16, 4, 128, 2, shared_inter=128),
                                W.Workload("acc_large", 300, 512, 16, 4, 128, 2, shared_inter=128),
                                W.Workload("acc_f32", 40, 128, 4, 2, 64, 1, dtype="f32")],
                         ids=lambda w: w.name)
def test_accumulate_adds_the_layer_output_into_y(wl):
    dev = parity.to_device(W.make_inputs(wl, seed=6))
    layer = _layer(wl)
    plain = _forward(layer, dev).float()
    g = torch.Generator(device="cuda").manual_seed(1)
    y0 = torch.randn(plain.shape, generator=g, device="cuda").to(wl.torch_dtype)
    y = y0.clone()
    layer.set_accumulate(True)
    layer.forward(dev["x"], dev["router_w"], dev["router_bias"], dev["w13"], dev["w2"], dev["shared_w13"],
                  dev["shared_w2"], out=y)
    layer.sync()
    want = y0.float() + plain
    err = (y.float() - want).abs().max().item() / want.abs().max().item()
    assert err <= (1e-2 if wl.dtype == "bf16" else 1e-5)
    # the host entry point accumulates into the host buffer the same way
    yh = y0.cpu().pin_memory()
    layer.forward_host(dev["x"].cpu().pin_memory(), dev["router_w"], dev["router_bias"], dev["w13"], dev["w2"],
                       dev["shared_w13"], dev["shared_w2"], out_host=yh)
    assert torch.equal(yh, y.cpu())
    layer.close()


def test_host_entry_point_matches_device_entry_point():
    wl = W.Workload("host", 100, 256, 8, 2, 128, 1)
    inp = W.make_inputs(wl, seed=4)
    dev = parity.to_device(inp)
    layer = _layer(wl)
    y_dev = _forward(layer, dev).cpu()
    y_host = layer.forward_host(inp["x"].pin_memory(), dev["router_w"], None, dev["w13"], dev["w2"])
    assert torch.equal(y_dev, y_host)
    layer.close()


def test_async_host_calls_overlap_and_match_device_calls():
    """moe_forward_host_async: a run of calls of mixed sizes (decode-sized and
    large, so both launch sequences), each on its own pinned buffers, issued
    back to back and read after one moe_sync, equals the same calls through
    moe_forward; a blocking host call in the middle of the run keeps the order."""
    wl = W.Workload("host_async", 300, 256, 8, 2, 128, 2, shared_inter=128)
    wts = parity.to_device(W.make_inputs(wl, seed=6))
    layer = _layer(wl)
    sizes = [8, 300, 16, 1, 200, 300, 5, 64]
    xs = [W.make_inputs(wl, seed=80 + i, T=T, experts=False)["x"].pin_memory() for i, T in enumerate(sizes)]
    ys = [torch.empty_like(x).pin_memory() for x in xs]
    args = (wts["router_w"], wts["router_bias"], wts["w13"], wts["w2"], wts["shared_w13"], wts["shared_w2"])
    for i, (x, y) in enumerate(zip(xs, ys)):
        layer.forward_host(x, *args, out_host=y, wait=(i == 4))
    layer.sync()
    for T, x, y in zip(sizes, xs, ys):
        ref = layer.forward(x.cuda(), *args)
        layer.sync()
        assert torch.equal(y, ref.cpu()), f"T={T}: async host result differs from the device call"
    layer.close()


def test_async_host_calls_accumulate_into_their_own_buffers():
    wl = W.Workload("host_async_acc", 40, 256, 8, 2, 128, 1)
    wts = parity.to_device(W.make_inputs(wl, seed=7))
    layer = _layer(wl)
    args = (wts["router_w"], None, wts["w13"], wts["w2"])
    xs = [W.make_inputs(wl, seed=90 + i, experts=False)["x"].pin_memory() for i in range(3)]
    plain = [layer.forward(x.cuda(), *args).float().cpu() for x in xs]
    layer.sync()
    g = torch.Generator().manual_seed(3)
    y0 = [torch.randn((wl.T, wl.H), generator=g).to(torch.bfloat16) for _ in xs]
    ys = [y.clone().pin_memory() for y in y0]
    layer.set_accumulate(True)
    for x, y in zip(xs, ys):
        layer.forward_host(x, *args, out_host=y, wait=False)
    layer.sync()
    for y, a, p_ in zip(ys, y0, plain):
        want = a.float() + p_
        err = (y.float() - want).abs().max().item() / want.abs().max().item()
        assert err <= 1e-2
    layer.close()


def test_invalid_arguments_are_rejected_without_poisoning_the_handle():
    wl = W.Workload("args", 16, 256, 8, 2, 128, 2)
    dev = parity.to_device(W.make_inputs(wl, seed=5))
    layer = _layer(wl)
    lib = binding.load()
    p13 = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in dev["w13"]])
    p2 = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in dev["w2"]])
    y = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = [layer._h, dev["x"].data_ptr(), dev["router_w"].data_ptr(), None, p13, p2, 2, 2, None, None, 16,
            y.data_ptr(), s]
    assert lib.moe_forward(*args) == 0
    for i, v in [(6, 1), (7, 3), (10, 17), (10, -1), (11, y.data_ptr() + 2), (1, dev["x"].data_ptr() + 8),
                 (8, dev["w13"][0].data_ptr())]:
        bad = list(args)
        bad[i] = v
        assert lib.moe_forward(*bad) == 1, (i, v)
    assert lib.moe_forward(*args) == 0
    layer.sync()
    layer.close()


def test_bounded_wait_reports_timeout_instead_of_hanging():
    assert binding.selftest_wait_timeout(2000) == "MOE_ERR_TIMEOUT"
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda")
    assert x.sum().item() == 4.0


def test_back_to_back_small_batches_reuse_the_workspace():
    """Consecutive decode-sized calls on one handle (per-call counters must be
    reset by each call) give the same result as fresh handles."""
    wl = W.Workload("b2b", 8, 512, 64, 8, 128, 1)
    inps = [parity.to_device(W.make_inputs(wl, seed=s)) for s in (31, 32, 33)]
    layer = _layer(wl)
    ys = [_forward(layer, d).clone() for d in inps + inps]
    layer.close()
    for i, d in enumerate(inps):
        fresh = _layer(wl)
        ref = _forward(fresh, d)
        fresh.close()
        assert torch.equal(ys[i], ref) and torch.equal(ys[i + 3], ref)


def test_empty_batches_return_empty_outputs_and_leave_the_handle_usable():
    """T = 0 through the device and host entry points (and the MXFP8 one) is a
    no-op that returns an empty y; the next call on the handle still matches
    the oracle."""
    wl = W.Workload("empty", 40, 512, 16, 4, 128, 2, shared_inter=128)
    inp = W.make_inputs(wl, seed=9)
    dev = parity.to_device(inp)
    args = (dev["router_w"], dev["router_bias"], dev["w13"], dev["w2"], dev["shared_w13"], dev["shared_w2"])
    layer = _layer(wl)
    x0 = torch.empty((0, wl.H), dtype=torch.bfloat16, device="cuda")
    assert layer.forward(x0, *args).shape == (0, wl.H)
    assert layer.forward_host(torch.empty((0, wl.H), dtype=torch.bfloat16), *args).shape == (0, wl.H)
    layer.sync()
    y = _forward(layer, dev)
    _check(wl, inp, y)
    layer.close()
    mx = W.Workload("empty_mx", 8, 512, 16, 4, 128, 1)
    mdev = parity.to_device(W.make_inputs(mx, seed=9))
    q13 = [binding.quantize_mxfp8(t) for t in mdev["w13"]]
    q2 = [binding.quantize_mxfp8(t) for t in mdev["w2"]]
    mlayer = binding.MoELayer(mx.H, mx.E, mx.k, mx.I, 1, max_tokens=mx.T)
    assert mlayer.forward_mxfp8(x0, mdev["router_w"], None, q13, q2).shape == (0, mx.H)
    mlayer.sync()
    mlayer.close()


def test_mixed_batch_sizes_back_to_back_match_isolated_calls():
    """Calls of different sizes issued back to back on one stream, no sync in
    between: each call's kernels may be placed while the previous kernel in the
    stream still runs (programmatic dependent launch: the fused small-batch
    kernel, the router, and the large-batch scan, placement, gather, GEMMs and
    finalize), and small and large calls share the workspace. Every result must
    equal the same call run on its own."""
    base = W.Workload("mix", 300, 512, 16, 4, 128, 2, shared_inter=128)
    wts = parity.to_device(W.make_inputs(base, seed=0))
    args = (wts["router_w"], wts["router_bias"], wts["w13"], wts["w2"], wts["shared_w13"], wts["shared_w2"])
    Ts = [300, 8, 257, 16, 1, 300, 13, 129, 8]
    xs = [W.make_inputs(base, seed=40 + i, T=T, experts=False)["x"].cuda() for i, T in enumerate(Ts)]
    layer = _layer(base)
    outs = [torch.empty_like(x) for x in xs]
    for x, y in zip(xs, outs):
        layer.forward(x, *args, out=y)
    layer.sync()
    for T, x, y in zip(Ts, xs, outs):
        ref = layer.forward(x, *args)
        layer.sync()
        assert torch.equal(y, ref), f"T={T}: back-to-back result differs from the isolated call"
    layer.close()


@pytest.mark.parametrize("wl", [W.Workload("side_17", 17, 512, 8, 2, 256, 2, shared_inter=128),
                                W.Workload("side_257", 257, 256, 16, 4, 128, 2, shared_inter=256)],
                         ids=lambda w: w.name)
def test_shared_expert_on_a_second_stream_is_bit_identical(wl):
    """moe_set_shared_stream: the shared expert's GEMMs forked onto the handle's
    stream and joined before the finalize give the same bits as the default
    single-stream order, also for back-to-back calls on one handle."""
    inps = [parity.to_device(W.make_inputs(wl, seed=s)) for s in (41, 42)]
    plain = _layer(wl)
    ref = [_forward(plain, d).clone() for d in inps]
    plain.close()
    side = _layer(wl)
    side.set_shared_stream(True)
    ys = [_forward(side, d).clone() for d in inps + inps]
    side.close()
    for i in range(2):
        assert torch.equal(ys[i], ref[i]) and torch.equal(ys[i + 2], ref[i])
    _check(wl, W.make_inputs(wl, seed=41), ys[0])
