"""GB300-native routed mixture-of-experts FFN layer (sm_103a CUDA behind a C ABI).

The layer: softmax gate with renormalised top-k, a stable route permutation
with per-expert offsets, one gather, tcgen05 grouped GEMM1 with a fused SwiGLU
epilogue, a grouped down-projection GEMM that accumulates across micro-shards,
and one finalize (routing scale and top-k sum). ``MoELayer`` in ``binding`` is
the Python face of the C ABI declared in ``include/moe.h``.
"""
import importlib

__all__ = ["MoELayer", "MoEError"]


def __getattr__(name):
    if name in ("MoELayer", "MoEError"):
        return getattr(importlib.import_module(__name__ + ".binding"), name)
    raise AttributeError(name)
