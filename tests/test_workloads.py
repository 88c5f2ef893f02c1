"""The seeded input generator: shapes, determinism and the skewed workload's load."""
import numpy as np
import torch

import oracle
from mixture_experts_layer_warp_gb300 import workloads as W


def test_shapes_and_dtypes_small():
    wl = W.WORKLOADS["tiny_fp32"]
    inp = W.make_inputs(wl, seed=0)
    assert inp["x"].shape == (64, 256) and inp["x"].dtype == torch.float32
    assert inp["router_w"].shape == (8, 256)
    assert len(inp["w13"]) == 1 and inp["w13"][0].shape == (8, 1024, 256)
    assert inp["w2"][0].shape == (8, 256, 512)
    assert inp["router_bias"] is None and inp["shared_w13"] is None


def test_multi_micro_and_shared_shapes():
    wl = W.Workload("t", 10, 64, 4, 2, 32, 2, shared_inter=48, x_parts=2)
    inp = W.make_inputs(wl, seed=1)
    assert inp["x"].shape == (10, 64) and inp["x"].dtype == torch.bfloat16
    assert [t.shape for t in inp["w13"]] == [(4, 64, 64)] * 2
    assert [t.shape for t in inp["w2"]] == [(4, 64, 32)] * 2
    assert inp["shared_w13"].shape == (96, 64) and inp["shared_w2"].shape == (64, 48)


def test_seeded_and_independent_of_token_count():
    wl = W.Workload("t", 16, 32, 4, 2, 16, 1)
    a = W.make_inputs(wl, seed=3)
    b = W.make_inputs(wl, seed=3, T=5)
    c = W.make_inputs(wl, seed=4)
    assert torch.equal(a["w13"][0], b["w13"][0]) and torch.equal(a["router_w"], b["router_w"])
    assert not torch.equal(a["w13"][0], c["w13"][0])
    assert torch.equal(a["x"], W.make_inputs(wl, seed=3)["x"])


def test_weight_scale_follows_fan_in():
    wl = W.Workload("t", 4, 512, 2, 1, 256, 1)
    inp = W.make_inputs(wl, seed=0)
    assert abs(inp["w13"][0].float().std().item() * np.sqrt(512) - 1) < 0.02
    assert abs(inp["w2"][0].float().std().item() * np.sqrt(256) - 1) < 0.02


def test_integer_grid_is_exact_in_fp32():
    g = W.integer_grid_inputs(20, 4096, 64, seed=0)
    x = W.to_numpy(g["x"])
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert np.all(xf * 4 == np.round(xf * 4)) and np.abs(xf).max() <= 1.0


def test_skewed_load_is_about_ten_to_one():
    """The log-Zipf bias gives max/min expert load near 10 (oracle routing, seed 0)."""
    wl = W.WORKLOADS["skewed"]
    inp = W.make_inputs(wl, seed=0, experts=False)
    lg = oracle.logits(W.to_numpy(inp["x"]), W.to_numpy(inp["router_w"]),
                       inp["router_bias"].numpy())
    ids, _ = oracle.route(lg, wl.k)
    c = np.bincount(ids.ravel(), minlength=wl.E)
    assert 8.0 <= c.max() / c.min() <= 12.0, (c.max(), c.min())


def test_hot_bias_routes_every_token_to_the_same_k_experts():
    """The "hot" bias: every token's top-k is the seeded set of k experts, in
    some order, and the other experts receive no route (oracle routing)."""
    wl = W.Workload("hot", 300, 256, 16, 4, 128, 1, router_bias="hot")
    inp = W.make_inputs(wl, seed=1, experts=False)
    bias = inp["router_bias"].numpy()
    hot = np.flatnonzero(bias)
    assert len(hot) == wl.k and np.all(bias[hot] == W.HOT_BIAS)
    lg = oracle.logits(W.to_numpy(inp["x"]), W.to_numpy(inp["router_w"]), bias)
    ids, w = oracle.route(lg, wl.k)
    assert np.all(np.sort(ids, axis=1) == hot[None, :])
    assert np.allclose(w.sum(axis=1), 1.0)
    assert w.min() > 0.0
