"""Seeded synthetic inputs for the routed MoE layer.

This module draws random numbers and nothing else: it holds none of the layer's
arithmetic (no logits, no routing, no expert math), so both the CUDA path's
tests and the fp64 oracle can take their inputs from it.

The five workloads are shaped like the two phases of Hunyuan Image 3.0 that
"HunyuanImage3 Hybrid Parallelism" describes: hidden 4096, 64 experts, top-8,
and the micro-major pack W1 [2][64][1536][4096], W2 [2][64][4096][768] of one
storage-TP rank (section 5). Token counts stand in for an AR decode step and
for denoise image-token batches; there is no dataset.

Distributions: x ~ N(0, 1); router and expert weights ~ N(0, 1/fan_in) with
fan_in = H for the router and w13, and I (or Is) for w2; the "uniform" router
is U(-1/sqrt(H), 1/sqrt(H)). Weights are drawn in fp32 and rounded once to
bf16 for the bf16 workloads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# log-Zipf router bias strength for the skewed workload: b_e = -ALPHA * s * ln(rank_e)
# with s = 1.1 and rank_e a seeded permutation of 1..E. ALPHA was chosen so that
# the busiest expert receives about 10x the routes of the least busy one at
# seed 0 (checked by a CPU test on the oracle's routing).
LOG_ZIPF_S = 1.1
LOG_ZIPF_ALPHA = 0.365
# "hot" router bias: +HOT_BIAS on a seeded set of k experts, far above the
# spread of the logits x.Wr (about N(0, 1)), so every token routes to those k
# and every other expert's segment is empty (the most skewed load top-k allows)
HOT_BIAS = 16.0


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # hidden
    E: int            # routed experts
    k: int            # top_k
    I: int            # intermediate size of one micro-shard
    n_micro: int      # micro-shards per expert
    shared_inter: int = 0          # Is of the dense shared expert (0 = none)
    dtype: str = "bf16"            # "bf16" or "f32"
    router_init: str = "normal"    # "normal" N(0,1/H) or "uniform" U(+-1/sqrt(H))
    router_bias: str | None = None  # None, "log_zipf" or "hot"
    x_parts: int = 1               # x drawn as this many independent halves (CFG)
    note: str = field(default="", compare=False)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_tokens(self, T: int) -> "Workload":
        return Workload(self.name, T, self.H, self.E, self.k, self.I, self.n_micro,
                        self.shared_inter, self.dtype, self.router_init, self.router_bias,
                        self.x_parts, self.note)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 64, 256, 8, 2, 512, 1, dtype="f32",
                          note="tiny fp32 layer; the oracle runs it whole in seconds"),
    "decode": Workload("decode", 8, 4096, 64, 8, 768, 1,
                       note="AR-decode-like: 8 tokens, every touched expert streamed once"),
    "denoise_multi_micro": Workload("denoise_multi_micro", 4096, 4096, 64, 8, 768, 2,
                                    router_init="uniform",
                                    note="denoise-like, two micro-shards sharing one routing"),
    "skewed": Workload("skewed", 16384, 4096, 64, 8, 1536, 1, router_bias="log_zipf",
                       note="large denoise with log-Zipf router bias (about 10x load skew)"),
    "cfg_shared": Workload("cfg_shared", 32768, 4096, 64, 8, 1536, 2, shared_inter=3072,
                           x_parts=2,
                           note="CFG-doubled denoise, two micro-shards plus a dense shared expert"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std: float, g: torch.Generator, device, dtype: torch.dtype) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_inputs(wl: Workload, seed: int = 0, device="cpu", T: int | None = None,
                experts: bool = True) -> dict:
    """Draw the inputs of one layer call.

    Returns a dict of tensors on ``device``: ``x [T,H]``, ``router_w [E,H]``,
    ``router_bias [E] fp32 or None``, ``w13`` (list over micros of [E,2I,H]),
    ``w2`` (list of [E,H,I]), ``shared_w13 [2Is,H]`` and ``shared_w2 [H,Is]``
    (or None). Each tensor has its own generator seeded from ``seed``, so
    changing ``T`` leaves the weights unchanged. ``experts=False`` skips the
    expert and shared weights.
    """
    T = wl.T if T is None else T
    dt = wl.torch_dtype
    H, E, I = wl.H, wl.E, wl.I
    base = 1000 * seed
    out: dict = {}

    parts = []
    per = [T // wl.x_parts + (1 if p < T % wl.x_parts else 0) for p in range(wl.x_parts)]
    for p, n in enumerate(per):
        parts.append(_normal((n, H), 1.0, _gen(base + 1 + p, device), device, dt))
    out["x"] = torch.cat(parts, 0) if len(parts) > 1 else parts[0]

    g = _gen(base + 10, device)
    if wl.router_init == "uniform":
        r = torch.rand((E, H), generator=g, device=device, dtype=torch.float32)
        out["router_w"] = ((r * 2.0 - 1.0) / math.sqrt(H)).to(dt)
    else:
        out["router_w"] = _normal((E, H), 1.0 / math.sqrt(H), g, device, dt)

    if wl.router_bias == "log_zipf":
        rank = torch.randperm(E, generator=_gen(base + 11, "cpu")).to(torch.float64) + 1.0
        bias = -LOG_ZIPF_ALPHA * LOG_ZIPF_S * torch.log(rank)
        out["router_bias"] = bias.to(torch.float32).to(device)
    elif wl.router_bias == "hot":
        hot = torch.randperm(E, generator=_gen(base + 12, "cpu"))[: wl.k]
        bias = torch.zeros(E, dtype=torch.float32)
        bias[hot] = HOT_BIAS
        out["router_bias"] = bias.to(device)
    else:
        out["router_bias"] = None

    out["w13"], out["w2"] = [], []
    out["shared_w13"] = out["shared_w2"] = None
    if experts:
        for m in range(wl.n_micro):
            g13 = _gen(base + 100 + m, device)
            w13 = torch.empty((E, 2 * I, H), dtype=dt, device=device)
            for e in range(E):
                w13[e] = _normal((2 * I, H), 1.0 / math.sqrt(H), g13, device, dt)
            g2 = _gen(base + 200 + m, device)
            w2 = torch.empty((E, H, I), dtype=dt, device=device)
            for e in range(E):
                w2[e] = _normal((H, I), 1.0 / math.sqrt(I), g2, device, dt)
            out["w13"].append(w13)
            out["w2"].append(w2)
        if wl.shared_inter:
            Is = wl.shared_inter
            out["shared_w13"] = _normal((2 * Is, H), 1.0 / math.sqrt(H), _gen(base + 300, device),
                                        device, dt)
            out["shared_w2"] = _normal((H, Is), 1.0 / math.sqrt(Is), _gen(base + 301, device),
                                       device, dt)
    return out


def integer_grid_inputs(T: int, H: int, E: int, seed: int = 0, dtype=torch.bfloat16,
                        device="cpu", x_levels: int = 4, w_levels: int = 2) -> dict:
    """x and router weights on a small power-of-two grid.

    x = i / 4 with i in [-x_levels, x_levels], Wr = j / 8 with j in
    [-w_levels, w_levels]. Every product and every partial sum is a multiple of
    1/32 far below 2**24 of them, so fp32 and fp64 sums are exact in any order
    and exact ties between experts are common.
    """
    g = _gen(7000 + seed, "cpu")
    xi = torch.randint(-x_levels, x_levels + 1, (T, H), generator=g)
    wi = torch.randint(-w_levels, w_levels + 1, (E, H), generator=g)
    x = (xi.to(torch.float32) / 4.0).to(dtype).to(device)
    wr = (wi.to(torch.float32) / 8.0).to(dtype).to(device)
    return {"x": x, "router_w": wr}


def to_numpy(t: torch.Tensor | None) -> np.ndarray | None:
    """Host numpy view: fp32 as float32, bf16 as its uint16 bit pattern."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    return t.numpy()
