"""Python face of the C ABI in ``include/moe.h`` (ctypes; marshalling only).

Every step of the layer runs in the CUDA kernels of ``libmoe.so``; this module
checks tensor shapes, dtypes and devices, passes raw pointers and the current
CUDA stream, and turns status codes into exceptions. There is no fallback:
if the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import weakref

import torch

from . import build as _build

_lib = None

MOE_F32, MOE_BF16 = 0, 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_OOM", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_CHECK", 7: "MOE_ERR_STICKY"}
HEADER = os.path.join(_build.ROOT, "include", "moe.h")


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{self.name}: {message}")


class MoEConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("n_micro", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def declared_functions() -> list[str]:
    """Names of the functions ``include/moe.h`` declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load ``libmoe.so`` (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    p, i32 = ctypes.c_void_p, ctypes.c_int32
    st = ctypes.c_int
    sig = {
        "moe_create": (st, [ctypes.POINTER(MoEConfig), ctypes.POINTER(p)]),
        "moe_destroy": (None, [p]),
        "moe_route": (st, [p, p, p, p, i32, p, p, p, p, p, p]),
        "moe_forward": (st, [p, p, p, p, p, p, i32, i32, p, p, i32, p, p]),
        "moe_forward_host": (st, [p, p, p, p, p, p, i32, i32, p, p, i32, p, p]),
        "moe_forward_host_async": (st, [p, p, p, p, p, p, i32, i32, p, p, i32, p, p]),
        "moe_forward_mxfp8": (st, [p, p, p, p, p, p, p, p, i32, i32, p, p, i32, p, p]),
        "moe_forward_mxfp8_host_async": (st, [p, p, p, p, p, p, p, p, i32, i32, p, p, i32, p, p]),
        "moe_quantize_mxfp8": (st, [p, ctypes.c_int64, i32, i32, p, p, p]),
        "moe_sync": (st, [p]),
        "moe_last_error": (ctypes.c_char_p, [p]),
        "moe_status_string": (ctypes.c_char_p, [st]),
        "moe_workspace_ptr": (p, [p, i32]),
        "moe_selftest_wait_timeout": (st, [i32, p]),
        "moe_profile_begin": (st, [p, i32]),
        "moe_profile_end": (st, [p, p, p]),
        "moe_launch_count": (ctypes.c_int64, [p]),
        "moe_route_noalloc": (st, [p, p, p, i32, i32, i32, i32, i32, p, p, p, p, p]),
        "moe_route_noalloc_status": (st, [p]),
        "moe_set_accumulate": (st, [p, i32]),
        "moe_set_shared_stream": (st, [p, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device) -> int:
    """The raw cudaStream_t of the current stream on ``device``."""
    if _raw_stream is not None:
        if isinstance(device, torch.device):
            idx = device.index if device.index is not None else torch.cuda.current_device()
        else:
            idx = int(device)
        return _raw_stream(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def quantize_mxfp8(w: torch.Tensor):
    """``moe_quantize_mxfp8`` of a bf16 device tensor ``w`` [G, R, C] (or [R, C])
    along C: returns ``(codes uint8 [G, R, C], scales uint8 [G, C/32, R])``."""
    if w.dtype != torch.bfloat16 or not w.is_cuda or not w.is_contiguous() or w.dim() not in (2, 3):
        raise ValueError("w must be a contiguous bf16 CUDA tensor of 2 or 3 dimensions")
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    G, R, C = w3.shape
    if C % 32:
        raise ValueError("the last dimension must be a multiple of 32")
    codes = torch.empty((G, R, C), dtype=torch.uint8, device=w.device)
    scales = torch.empty((G, C // 32, R), dtype=torch.uint8, device=w.device)
    rc = load().moe_quantize_mxfp8(_ptr(w3), G, R, C, _ptr(codes), _ptr(scales), _stream(w.device))
    if rc != 0:
        raise MoEError(rc, "moe_quantize_mxfp8 failed")
    return (codes[0], scales[0]) if w.dim() == 2 else (codes, scales)


def selftest_wait_timeout(timeout_us: int = 1000) -> str:
    """Run the bounded-wait self-test kernel; returns the status name."""
    lib = load()
    return STATUS[lib.moe_selftest_wait_timeout(int(timeout_us), _stream(torch.cuda.current_device()))]


class MoELayer:
    """One routed MoE layer configuration with its device workspace.

    Weights are passed per call (they stay owned by the caller), so a resident
    micro-major pack ``W1[n_micro][E][2I][H]`` is used without repacking by
    passing ``[W1[m] for m in range(n_micro)]``.
    """

    def __init__(self, hidden: int, num_experts: int, top_k: int, inter: int, n_micro: int = 1,
                 max_tokens: int = 4096, shared_inter: int = 0, dtype: torch.dtype = torch.bfloat16,
                 device=None):
        if dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("dtype must be torch.bfloat16 or torch.float32")
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.dtype = dtype
        self.cfg = MoEConfig(hidden, num_experts, top_k, inter, n_micro, max_tokens, shared_inter,
                             MOE_BF16 if dtype == torch.bfloat16 else MOE_F32)
        self._lib = load()
        self._h = ctypes.c_void_p()
        self._wcache = None
        self._valid = {}  # argument name -> {id(tensor): (weak reference, data_ptr)} of tensors validated there
        self._stream_id = None
        with torch.cuda.device(self.device):
            rc = self._lib.moe_create(ctypes.byref(self.cfg), ctypes.byref(self._h))
        if rc != 0:
            raise MoEError(rc, "moe_create rejected the configuration")

    # -------------------------------------------------------------- helpers
    def _check(self, rc: int):
        if rc != 0:
            raise MoEError(rc, self._lib.moe_last_error(self._h).decode())

    def _tensor(self, t, name, shape, dtype=None, host=False):
        dtype = self.dtype if dtype is None else dtype
        # a tensor passed again in the same role (router matrix, output buffer,
        # a rotating set of input buffers) is not re-validated: a call's host
        # time is part of its latency
        seen = self._valid.get(name)
        memo = seen.get(id(t)) if seen is not None else None
        if memo is not None and memo[0]() is t and memo[1] == t.data_ptr() and t.shape == shape \
                and t.dtype == dtype:
            return t
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        if t.dtype != dtype:
            raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if host and t.is_cuda:
            raise ValueError(f"{name} must be in host memory")
        if not host and t.device != self.device:
            raise ValueError(f"{name} must be on {self.device}")
        seen = self._valid.setdefault(name, {})
        if len(seen) >= 16:
            seen.clear()
        seen[id(t)] = (weakref.ref(t), t.data_ptr())
        return t

    def _weights(self, w13, w2, shared_w13, shared_w2):
        # the same resident weight tensors are passed on every call: validate once
        key = (tuple(t.data_ptr() for t in w13), tuple(t.data_ptr() for t in w2),
               None if shared_w13 is None else shared_w13.data_ptr(),
               None if shared_w2 is None else shared_w2.data_ptr())
        if self._wcache is not None and self._wcache[0] == key:
            return self._wcache[1], self._wcache[2]
        c = self.cfg
        if len(w13) != c.n_micro or len(w2) != c.n_micro:
            raise ValueError(f"expected {c.n_micro} micro-shards of w13 and w2")
        for m in range(c.n_micro):
            self._tensor(w13[m], f"w13[{m}]", (c.num_experts, 2 * c.inter, c.hidden))
            self._tensor(w2[m], f"w2[{m}]", (c.num_experts, c.hidden, c.inter))
        if c.shared_inter:
            self._tensor(shared_w13, "shared_w13", (2 * c.shared_inter, c.hidden))
            self._tensor(shared_w2, "shared_w2", (c.hidden, c.shared_inter))
        elif shared_w13 is not None or shared_w2 is not None:
            raise ValueError("this layer has no shared expert")
        p13 = (ctypes.c_void_p * c.n_micro)(*[t.data_ptr() for t in w13])
        p2 = (ctypes.c_void_p * c.n_micro)(*[t.data_ptr() for t in w2])
        self._wcache = (key, p13, p2)
        return p13, p2

    def _router(self, router_w, router_bias):
        c = self.cfg
        self._tensor(router_w, "router_w", (c.num_experts, c.hidden))
        if router_bias is not None:
            self._tensor(router_bias, "router_bias", (c.num_experts,), torch.float32)
        return router_w, router_bias

    # -------------------------------------------------------------- API
    def route(self, x, router_w, router_bias=None, logits: bool = False) -> dict:
        """``moe_route``: ids, renormalised weights, permutation and offsets."""
        c = self.cfg
        T = x.shape[0]
        self._tensor(x, "x", (T, c.hidden))
        self._router(router_w, router_bias)
        dev = self.device
        out = {
            "ids": torch.empty((T, c.top_k), dtype=torch.int32, device=dev),
            "w": torch.empty((T, c.top_k), dtype=torch.float32, device=dev),
            "perm": torch.empty((T * c.top_k,), dtype=torch.int32, device=dev),
            "offsets": torch.empty((c.num_experts + 1,), dtype=torch.int32, device=dev),
        }
        if logits:
            out["logits"] = torch.empty((T, c.num_experts), dtype=torch.float32, device=dev)
        rc = self._lib.moe_route(self._h, _ptr(x), _ptr(router_w), _ptr(router_bias), T,
                                 _ptr(out["ids"]), _ptr(out["w"]), _ptr(out["perm"]), _ptr(out["offsets"]),
                                 _ptr(out.get("logits")), _stream(dev))
        self._check(rc)
        return out

    def forward(self, x, router_w, router_bias, w13, w2, shared_w13=None, shared_w2=None, out=None):
        """``moe_forward``: the whole layer on device tensors; returns y [T, H]."""
        c = self.cfg
        T = x.shape[0]
        self._tensor(x, "x", (T, c.hidden))
        self._router(router_w, router_bias)
        p13, p2 = self._weights(w13, w2, shared_w13, shared_w2)
        y = torch.empty((T, c.hidden), dtype=self.dtype, device=self.device) if out is None else \
            self._tensor(out, "out", (T, c.hidden))
        rc = self._lib.moe_forward(self._h, _ptr(x), _ptr(router_w), _ptr(router_bias), p13, p2, c.n_micro,
                                   c.top_k, _ptr(shared_w13), _ptr(shared_w2), T, _ptr(y),
                                   _stream(self.device))
        self._check(rc)
        return y

    def forward_host(self, x_host, router_w, router_bias, w13, w2, shared_w13=None, shared_w2=None,
                     out_host=None, wait=True):
        """``moe_forward_host`` (``wait=False``: ``moe_forward_host_async``, y valid
        after ``sync()``): x and y in (preferably pinned) host memory."""
        c = self.cfg
        T = x_host.shape[0]
        self._tensor(x_host, "x_host", (T, c.hidden), host=True)
        self._router(router_w, router_bias)
        p13, p2 = self._weights(w13, w2, shared_w13, shared_w2)
        y = torch.empty((T, c.hidden), dtype=self.dtype, pin_memory=True) if out_host is None else \
            self._tensor(out_host, "out_host", (T, c.hidden), host=True)
        fn = self._lib.moe_forward_host if wait else self._lib.moe_forward_host_async
        rc = fn(self._h, _ptr(x_host), _ptr(router_w), _ptr(router_bias), p13, p2, c.n_micro, c.top_k,
                _ptr(shared_w13), _ptr(shared_w2), T, _ptr(y), _stream(self.device))
        self._check(rc)
        return y

    def forward_mxfp8(self, x, router_w, router_bias, w13_q, w2_q, shared_w13=None, shared_w2=None, out=None,
                      host_async=False):
        """``moe_forward_mxfp8``: routed experts in MXFP8 (``w13_q`` / ``w2_q``: per
        micro, ``(codes, scales)`` pairs from ``quantize_mxfp8``); returns y [T, H].
        ``host_async``: x and ``out`` in host memory through
        ``moe_forward_mxfp8_host_async`` (y valid after ``sync()``)."""
        c = self.cfg
        T = x.shape[0]
        self._tensor(x, "x_host" if host_async else "x", (T, c.hidden), host=host_async)
        self._router(router_w, router_bias)
        if len(w13_q) != c.n_micro or len(w2_q) != c.n_micro:
            raise ValueError(f"expected {c.n_micro} micro-shards of w13 and w2")
        E, H, I = c.num_experts, c.hidden, c.inter
        for m in range(c.n_micro):
            self._tensor(w13_q[m][0], f"w13 codes[{m}]", (E, 2 * I, H), torch.uint8)
            self._tensor(w13_q[m][1], f"w13 scales[{m}]", (E, H // 32, 2 * I), torch.uint8)
            self._tensor(w2_q[m][0], f"w2 codes[{m}]", (E, H, I), torch.uint8)
            self._tensor(w2_q[m][1], f"w2 scales[{m}]", (E, I // 32, H), torch.uint8)
        if c.shared_inter:
            self._tensor(shared_w13, "shared_w13", (2 * c.shared_inter, H))
            self._tensor(shared_w2, "shared_w2", (H, c.shared_inter))
        arr = lambda ts: (ctypes.c_void_p * c.n_micro)(*[t.data_ptr() for t in ts])  # noqa: E731
        if host_async:
            y = torch.empty((T, H), dtype=self.dtype, pin_memory=True) if out is None else \
                self._tensor(out, "out_host", (T, H), host=True)
        else:
            y = torch.empty((T, H), dtype=self.dtype, device=self.device) if out is None else \
                self._tensor(out, "out", (T, H))
        fn = self._lib.moe_forward_mxfp8_host_async if host_async else self._lib.moe_forward_mxfp8
        rc = fn(self._h, _ptr(x), _ptr(router_w), _ptr(router_bias),
                arr([q[0] for q in w13_q]), arr([q[1] for q in w13_q]),
                arr([q[0] for q in w2_q]), arr([q[1] for q in w2_q]),
                c.n_micro, c.top_k, _ptr(shared_w13), _ptr(shared_w2), T, _ptr(y), _stream(self.device))
        self._check(rc)
        return y

    def set_accumulate(self, on: bool):
        """``moe_set_accumulate``: later forwards add into ``out`` (y += layer(x))."""
        self._check(self._lib.moe_set_accumulate(self._h, 1 if on else 0))

    def set_shared_stream(self, on: bool):
        """``moe_set_shared_stream``: the shared expert's GEMMs on a second stream."""
        self._check(self._lib.moe_set_shared_stream(self._h, 1 if on else 0))

    def sync(self):
        """``moe_sync``: wait for the last call and raise on a device-side error."""
        self._check(self._lib.moe_sync(self._h))

    PROFILE_SLOTS = ("router", "scan", "place", "gather", "gemm1_swiglu", "gemm2_down", "shared_gemm1",
                     "shared_gemm2", "finalize")

    def profile_begin(self, max_calls: int):
        """Start per-kernel event timing for the next ``max_calls`` calls."""
        self._check(self._lib.moe_profile_begin(self._h, int(max_calls)))

    def profile_end(self) -> dict:
        """Stop timing; returns {slot: (total_ms, launches)} for slots that ran."""
        n = len(self.PROFILE_SLOTS)
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int32 * n)()
        self._check(self._lib.moe_profile_end(self._h, ms, cnt))
        return {name: (float(ms[i]), int(cnt[i])) for i, name in enumerate(self.PROFILE_SLOTS) if cnt[i]}

    def launch_count(self) -> int:
        """Kernels launched by this handle since it was created."""
        return int(self._lib.moe_launch_count(self._h))

    def workspace_ptr(self, which: int) -> int:
        return self._lib.moe_workspace_ptr(self._h, which) or 0

    def close(self):
        if self._h:
            self._lib.moe_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass
