"""fp64 CPU oracle of the routed MoE layer.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (``bench.py`` ``cpu_baseline`` and
``--impl reference``) may import this package. The CUDA path never imports it
and shares no code with it.
"""
from .oracle import (  # noqa: F401
    bf16_round,
    build,
    load_variant,
    forward_permuted,
    forward_tokens,
    forward_tokens_mx,
    layer,
    logits,
    mx_dequant,
    mx_quantize,
    num_threads,
    permute,
    route,
    set_threads,
)
