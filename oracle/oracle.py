"""ctypes wrapper of the fp64 C oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
CPU-baseline leg load this module; the CUDA path never does.

Arrays are numpy. Activations and weights are passed as ``float32``, as
``uint16`` bf16 bit patterns or (weights) as ``float64``; the C side widens them
exactly to fp64. Every function follows the steps of "HunyuanImage3 Hybrid
Parallelism" section 6.1 and the Ascend guide section 2.2, as documented in
``moe_oracle.c``; ``mx_quantize`` / ``mx_dequant`` define the block-scaled FP8
(MXFP8) expert weights.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

_F32, _BF16, _F64 = 0, 1, 2
_p = ctypes.c_void_p
_i64 = ctypes.c_int64


def build(force: bool = False, src: str = _SRC, out: str = _SO) -> str:
    """Compile ``moe_oracle.c`` with gcc -O2 -fopenmp (no fast-math)."""
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.orc_logits.argtypes = [_p, _p, ctypes.c_int, _p, _i64, _i64, _i64, _p]
    lib.orc_route.argtypes = [_p, _i64, _i64, _i64, _p, _p, _p]
    lib.orc_permute.argtypes = [_p, _i64, _i64, _i64, _p, _p, _p, _p]
    lib.orc_forward_tokens.argtypes = [
        _p, ctypes.c_int, _i64, _i64, _i64, _i64, _i64, _p, _p, _p, _p, _i64,
        _p, _p, _p, _i64, _p]
    lib.orc_forward_tokens_typed.argtypes = [
        _p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _i64, _i64, _p, _p, _p, _p,
        _i64, _p, _p, _p, _i64, _p, ctypes.c_int]
    lib.orc_mx_quantize.argtypes = [_p, ctypes.c_int, _i64, _i64, _i64, _p, _p]
    lib.orc_mx_dequant.argtypes = [_p, _p, _i64, _i64, _i64, _p]
    lib.orc_bf16_round.argtypes = [_p, _i64, _p]
    lib.orc_forward_permuted.argtypes = [
        _p, ctypes.c_int, _i64, _i64, _i64, _i64, _i64, _i64, _p, _p, _p, _p, _i64,
        _p, _p, _p, _p, _p]
    lib.orc_num_threads.argtypes = []
    lib.orc_set_threads.argtypes = [ctypes.c_int]
    for fn in ("orc_logits", "orc_route", "orc_permute", "orc_forward_tokens", "orc_forward_tokens_typed",
               "orc_forward_permuted", "orc_num_threads", "orc_set_threads", "orc_mx_quantize", "orc_mx_dequant",
               "orc_bf16_round"):
        getattr(lib, fn).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return _F32
    if a.dtype == np.uint16:
        return _BF16
    if a.dtype == np.float64:
        return _F64
    raise TypeError(f"oracle takes float32, uint16 (bf16 bits) or float64, got {a.dtype}")


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


def load_variant(src: str, out: str):
    """Compile and bind another build of the oracle source (used by the tests
    that plant a mistake in a copy of the oracle to show that a pin catches it)."""
    return _bind(build(True, src, out))


def _ptr(a) -> int | None:
    return None if a is None else a.ctypes.data


def num_threads(lib=None) -> int:
    return int((lib or _load()).orc_num_threads())


def set_threads(n: int, lib=None) -> int:
    """OpenMP threads for later oracle calls from this thread; returns the number in effect."""
    return int((lib or _load()).orc_set_threads(int(n)))


def logits(x: np.ndarray, wr: np.ndarray, bias: np.ndarray | None = None, lib=None) -> np.ndarray:
    """fp64 router logits ``x @ wr.T + bias``; x [T,H], wr [E,H], bias fp32 [E]."""
    x, wr = _c(x), _c(wr)
    dt = _dtype_code(x)
    if _dtype_code(wr) != dt:
        raise TypeError("x and router weight must share a dtype")
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float64)
    rc = (lib or _load()).orc_logits(_ptr(x), _ptr(wr), dt, _ptr(b), T, H, E, _ptr(out))
    if rc:
        raise RuntimeError(f"orc_logits failed ({rc})")
    return out


def route(lg: np.ndarray, k: int, return_probs: bool = False, lib=None):
    """Softmax gate, top-k (ties to lower index), renormalised weights.

    Returns ``(ids int32 [T,k], w float64 [T,k])`` (+ full softmax if asked).
    """
    lg = _c(lg, np.float64)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    probs = np.empty((T, E), np.float64) if return_probs else None
    rc = (lib or _load()).orc_route(_ptr(lg), T, E, k, _ptr(ids), _ptr(w), _ptr(probs))
    if rc:
        raise RuntimeError(f"orc_route failed ({rc})")
    return (ids, w, probs) if return_probs else (ids, w)


def permute(ids: np.ndarray, num_experts: int, lib=None):
    """Stable route sort by expert: ``(counts, offsets[E+1], perm, inv)``."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    E = num_experts
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    rc = (lib or _load()).orc_permute(_ptr(ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv))
    if rc:
        raise RuntimeError(f"orc_permute failed ({rc})")
    return counts, offsets, perm, inv


def _weights(w13, w2, dt):
    """Routed expert weights: x's dtype, or fp64 (e.g. dequantised MXFP8 weights)."""
    w13 = [_c(a) for a in w13]
    w2 = [_c(a) for a in w2]
    wdt = _dtype_code(w13[0]) if w13 else dt
    for a in w13 + w2:
        if _dtype_code(a) != wdt or wdt not in (dt, _F64):
            raise TypeError("routed weights must all be in the activation dtype or all fp64")
    n_micro = len(w13)
    if len(w2) != n_micro or n_micro == 0:
        raise ValueError("w13 and w2 need one entry per micro-shard")
    E, two_i, H = w13[0].shape
    I = two_i // 2
    for a, b in zip(w13, w2):
        if a.shape != (E, 2 * I, H) or b.shape != (E, H, I):
            raise ValueError(f"bad expert shapes {a.shape} / {b.shape}")
    p13 = (ctypes.c_void_p * n_micro)(*[a.ctypes.data for a in w13])
    p2 = (ctypes.c_void_p * n_micro)(*[a.ctypes.data for a in w2])
    return w13, w2, p13, p2, E, I, H, n_micro, wdt


def _shared(sw13, sw2, H, dt):
    if sw13 is None:
        return None, None, 0
    sw13, sw2 = _c(sw13), _c(sw2)
    if _dtype_code(sw13) != dt or _dtype_code(sw2) != dt:
        raise TypeError("shared expert weights must share the activation dtype")
    Is = sw13.shape[0] // 2
    if sw13.shape != (2 * Is, H) or sw2.shape != (H, Is):
        raise ValueError("bad shared expert shapes")
    return sw13, sw2, Is


def forward_tokens(x, ids, w, w13, w2, tokens=None, shared_w13=None, shared_w2=None, lib=None, mx_act=False):
    """Per-token definition ``y[t] = sum_j w_tj sum_m FFN_{m,e_j}(x_t) (+ shared)``.

    ``tokens`` selects rows to evaluate (default: all). Returns fp64 [n, H].
    """
    x = _c(x)
    dt = _dtype_code(x)
    keep = _weights(w13, w2, dt)
    _, _, p13, p2, E, I, H, n_micro, wdt = keep
    sw13, sw2, Is = _shared(shared_w13, shared_w2, H, dt)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    T, k = ids.shape
    tok = np.arange(T, dtype=np.int64) if tokens is None else _c(np.asarray(tokens), np.int64)
    if tok.size and (tok.min() < 0 or tok.max() >= T):
        raise IndexError("token index out of range")
    y = np.empty((tok.size, H), np.float64)
    rc = (lib or _load()).orc_forward_tokens_typed(
        _ptr(x), dt, wdt, dt, H, E, k, I, n_micro, p13, p2, _ptr(sw13), _ptr(sw2), Is,
        _ptr(ids), _ptr(w), _ptr(tok), tok.size, _ptr(y), 1 if mx_act else 0)
    if rc:
        raise RuntimeError(f"orc_forward_tokens failed ({rc})")
    return y


def forward_tokens_mx(x, ids, w, w13, w2, tokens=None, shared_w13=None, shared_w2=None, lib=None):
    """The layer with block-scaled FP8 arithmetic in the routed experts: as
    ``forward_tokens`` (``w13``/``w2`` typically the exact values of MXFP8
    weights, fp64), with each token's input to the routed experts replaced by
    its MXFP8 value (blocks of 32 along H) and each expert's SwiGLU output,
    rounded to bf16 (the layer's activation dtype), by its MXFP8 value (blocks
    of 32 along I) before the down projection. The shared expert takes the
    unquantised input."""
    return forward_tokens(x, ids, w, w13, w2, tokens, shared_w13, shared_w2, lib=lib, mx_act=True)


def forward_permuted(x, w, offsets, perm, inv, w13, w2, shared_w13=None, shared_w2=None,
                     lib=None):
    """The method's organisation: gather once, per-segment experts, one finalize."""
    x = _c(x)
    dt = _dtype_code(x)
    keep = _weights(w13, w2, dt)
    _, _, p13, p2, E, I, H, n_micro, wdt = keep
    if wdt != dt:
        raise TypeError("forward_permuted takes weights in the activation dtype")
    sw13, sw2, Is = _shared(shared_w13, shared_w2, H, dt)
    w = _c(w, np.float64)
    T, k = w.shape
    offsets = _c(offsets, np.int32)
    perm = _c(perm, np.int32)
    inv = _c(inv, np.int32)
    y = np.empty((T, H), np.float64)
    rc = (lib or _load()).orc_forward_permuted(
        _ptr(x), dt, T, H, E, k, I, n_micro, p13, p2, _ptr(sw13), _ptr(sw2), Is,
        _ptr(w), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(y))
    if rc:
        raise RuntimeError(f"orc_forward_permuted failed ({rc})")
    return y


def layer(x, wr, bias, w13, w2, k, shared_w13=None, shared_w2=None, tokens=None, lib=None):
    """Whole layer: logits -> route -> permute -> per-token outputs.

    Returns a dict with ``logits, ids, w, counts, offsets, perm, inv, y`` where
    ``y`` covers ``tokens`` (default: every token).
    """
    lg = logits(x, wr, bias, lib=lib)
    ids, w = route(lg, k, lib=lib)
    counts, offsets, perm, inv = permute(ids, wr.shape[0], lib=lib)
    y = forward_tokens(x, ids, w, w13, w2, tokens, shared_w13, shared_w2, lib=lib)
    return dict(logits=lg, ids=ids, w=w, counts=counts, offsets=offsets, perm=perm, inv=inv, y=y)


def mx_quantize(w: np.ndarray, lib=None):
    """MXFP8 codes and scales of ``w`` ([G][R][C] or [R][C], float32 or bf16
    bits), quantised along C in blocks of 32 (see ``orc_mx_quantize``).

    Returns ``(codes uint8 [G][R][C], scales uint8 [G][C/32][R])`` (no G axis
    for a 2-D input)."""
    w = _c(w)
    two_d = w.ndim == 2
    w3 = w[None] if two_d else w
    G, R, C = w3.shape
    codes = np.empty((G, R, C), np.uint8)
    scales = np.empty((G, C // 32, R), np.uint8)
    rc = (lib or _load()).orc_mx_quantize(_ptr(w3), _dtype_code(w3), G, R, C, _ptr(codes), _ptr(scales))
    if rc:
        raise RuntimeError(f"orc_mx_quantize failed ({rc})")
    return (codes[0], scales[0]) if two_d else (codes, scales)


def mx_dequant(codes: np.ndarray, scales: np.ndarray, lib=None) -> np.ndarray:
    """The fp64 value of MXFP8 weights: E4M3 code value times 2^(S-127), exactly."""
    two_d = codes.ndim == 2
    c3 = _c(codes[None] if two_d else codes, np.uint8)
    s3 = _c(scales[None] if two_d else scales, np.uint8)
    G, R, C = c3.shape
    if s3.shape != (G, C // 32, R):
        raise ValueError(f"scales must be [G][C/32][R], got {s3.shape}")
    out = np.empty((G, R, C), np.float64)
    rc = (lib or _load()).orc_mx_dequant(_ptr(c3), _ptr(s3), G, R, C, _ptr(out))
    if rc:
        raise RuntimeError(f"orc_mx_dequant failed ({rc})")
    return out[0] if two_d else out


def bf16_round(v, lib=None) -> np.ndarray:
    """fp64 values rounded to bfloat16 (nearest, ties to even), as fp64."""
    v = _c(np.asarray(v, np.float64).ravel(), np.float64)
    out = np.empty_like(v)
    rc = (lib or _load()).orc_bf16_round(_ptr(v), v.size, _ptr(out))
    if rc:
        raise RuntimeError(f"orc_bf16_round failed ({rc})")
    return out
