"""Parity checks between the CUDA path and the fp64 oracle.

Routing. Both sides take the top-k decision on fp32 logits (the gate's
precision, Ascend Hunyuan Image 3.0 guide section 5.2), but fp32 sums depend on
the summation order, so a token whose competing logits lie closer together
than the logit tolerance ``tau`` is *undecided*: either order is correct. For
decided tokens ids, slot order and weights must match the oracle exactly (ids)
or to 1e-5 (weights); for undecided ones the CUDA choice must be one the
oracle's logits allow within ``tau``. Offsets and the permutation must equal
the oracle's bit for bit when every token is decided, and must always equal
the stable counting sort of the CUDA path's own ids. On integer-grid inputs
logits are exact on both sides, so ``tau = 0`` and every token is decided:
ties are broken identically (lower expert index).

Outputs. ``max|y_gpu - y_oracle| / max|y_oracle|`` over the tokens whose
expert SET is decided must be <= 1e-2 for bf16 and <= 1e-5 for fp32.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_layer_warp_gb300 import workloads as W

Y_TOL = {"bf16": 1e-2, "f32": 1e-5}
W_TOL = 1e-5


def to_device(inp: dict, device="cuda") -> dict:
    out = {}
    for k, v in inp.items():
        if isinstance(v, list):
            out[k] = [t.to(device) for t in v]
        elif v is None:
            out[k] = None
        else:
            out[k] = v.to(device)
    return out


def to_host_numpy(inp: dict) -> dict:
    out = {}
    for k, v in inp.items():
        if isinstance(v, list):
            out[k] = [W.to_numpy(t) for t in v]
        elif v is None:
            out[k] = None
        elif k == "router_bias":
            out[k] = v.detach().cpu().numpy().astype(np.float32)
        else:
            out[k] = W.to_numpy(v)
    return out


def oracle_routing(host: dict, k: int) -> dict:
    lg = oracle.logits(host["x"], host["router_w"], host.get("router_bias"))
    ids, w = oracle.route(lg, k)
    counts, offsets, perm, inv = oracle.permute(ids, host["router_w"].shape[0])
    lf = lg.astype(np.float32).astype(np.float64)
    return dict(logits=lg, lf=lf, ids=ids, w=w, counts=counts, offsets=offsets, perm=perm, inv=inv)


def decided(lf: np.ndarray, ids: np.ndarray, tau: float):
    """(set_decided, order_decided) masks per token for logit tolerance tau."""
    T, E = lf.shape
    k = ids.shape[1]
    srt = -np.sort(-lf, axis=1)
    if k < E:
        set_ok = (srt[:, k - 1] - srt[:, k]) > 2 * tau
    else:
        set_ok = np.ones(T, bool)
    if k > 1:
        order_ok = set_ok & np.all((srt[:, : k - 1] - srt[:, 1:k]) > 2 * tau, axis=1)
    else:
        order_ok = set_ok.copy()
    if tau == 0:
        set_ok[:] = True
        order_ok[:] = True
    return set_ok, order_ok


def check_routing(gpu: dict, orc: dict, k: int, tau: float) -> dict:
    """Asserts the routing contract; returns counts of undecided tokens."""
    ids_g = gpu["ids"].cpu().numpy()
    w_g = gpu["w"].cpu().numpy().astype(np.float64)
    perm_g = gpu["perm"].cpu().numpy()
    off_g = gpu["offsets"].cpu().numpy()
    lf = orc["lf"]
    T, E = lf.shape
    if "logits" in gpu:
        lg_g = gpu["logits"].cpu().numpy().astype(np.float64)
        err = np.abs(lg_g - lf).max() if T else 0.0
        assert err <= tau, f"logit error {err:.3e} > tau {tau:.3e}"
    set_ok, order_ok = decided(lf, orc["ids"], tau)

    # decided tokens: identical ids in identical slot order
    bad = np.nonzero(order_ok & np.any(ids_g != orc["ids"], axis=1))[0]
    assert bad.size == 0, f"{bad.size} decided tokens differ, first {bad[:5]}: " \
        f"gpu {ids_g[bad[:1]]} oracle {orc['ids'][bad[:1]]}"
    # every token: distinct valid ids, consistent with the oracle's logits within tau
    assert ids_g.min() >= 0 and ids_g.max() < E
    for t in np.nonzero(~order_ok)[0]:
        s = ids_g[t]
        assert len(set(s.tolist())) == k
        rest = np.setdiff1d(np.arange(E), s)
        if rest.size:
            assert lf[t, s].min() >= lf[t, rest].max() - 2 * tau, f"token {t}: invalid set"
        assert np.all(lf[t, s[:-1]] >= lf[t, s[1:]] - 2 * tau), f"token {t}: invalid order"
    # weights, compared per expert on set-decided tokens
    if np.all(order_ok):
        d = np.abs(w_g - orc["w"]).max() if T else 0.0
    else:
        m = set_ok
        o_sorted = np.take_along_axis(orc["w"][m], np.argsort(orc["ids"][m], axis=1), axis=1)
        g_sorted = np.take_along_axis(w_g[m], np.argsort(ids_g[m], axis=1), axis=1)
        d = np.abs(o_sorted - g_sorted).max() if m.any() else 0.0
    assert d <= W_TOL, f"routing weight error {d:.3e}"
    assert np.all(np.abs(w_g.sum(1) - 1) < 1e-5)
    # offsets and permutation
    flat = ids_g.ravel()
    assert off_g.tolist() == [0] + np.cumsum(np.bincount(flat, minlength=E)).tolist()
    assert np.array_equal(perm_g, np.argsort(flat, kind="stable"))
    if np.all(set_ok):
        assert np.array_equal(off_g, orc["offsets"])
    if np.all(order_ok):
        assert np.array_equal(perm_g, orc["perm"])
    return dict(set_undecided=int((~set_ok).sum()), order_undecided=int((~order_ok).sum()))


def y_error(y_gpu: torch.Tensor, y_ref: np.ndarray, rows=None) -> float:
    g = y_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g = g[rows]
    den = np.abs(y_ref).max()
    return float(np.abs(g - y_ref).max() / den) if den > 0 else float(np.abs(g - y_ref).max())


def covering_tokens(orc: dict, T: int, k: int, stride: int = 128) -> np.ndarray:
    """Tokens such that every `stride`-row block of every expert segment of the
    sorted routes (and of the dense segment [0, T) of a shared expert) holds at
    least one of their routes, plus each segment's last row: every tile of the
    grouped GEMMs, whatever their row blocking at that granularity, then has a
    row the oracle checks."""
    off, perm = orc["offsets"], orc["perm"]
    rows = [np.arange(off[e], off[e + 1], stride) for e in range(len(off) - 1)]
    rows += [np.array([off[e + 1] - 1]) for e in range(len(off) - 1) if off[e + 1] > off[e]]
    routed = perm[np.concatenate(rows)] // k
    return np.unique(np.concatenate([routed, np.arange(0, T, stride), [T - 1]]))
