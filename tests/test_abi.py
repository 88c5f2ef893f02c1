"""The C-ABI library loads and exports every function its header declares.
No compute call is made: these run without a GPU."""
import ctypes

from mixture_experts_layer_warp_gb300 import binding


def test_header_declares_the_layer_entry_points():
    names = binding.declared_functions()
    for n in ("moe_create", "moe_destroy", "moe_route", "moe_forward", "moe_forward_host", "moe_forward_host_async",
              "moe_forward_mxfp8", "moe_forward_mxfp8_host_async", "moe_sync", "moe_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    missing = [n for n in binding.declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_config_rejection_need_no_device():
    lib = binding.load()
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(5) == b"MOE_ERR_TIMEOUT"
    h = ctypes.c_void_p()
    bad = [binding.MoEConfig(4096, 64, 65, 768, 1, 8, 0, 1),     # top_k > E
           binding.MoEConfig(4096, 65, 8, 768, 1, 8, 0, 1),     # E > 64
           binding.MoEConfig(4000, 64, 8, 768, 1, 8, 0, 1),     # H % 256 on bf16
           binding.MoEConfig(4096, 64, 8, 768, 5, 8, 0, 1),     # n_micro > 4
           binding.MoEConfig(0, 64, 8, 768, 1, 8, 0, 1),        # non-positive size
           binding.MoEConfig(4096, 64, 8, 768, 1, 8, 0, 7)]     # unknown dtype
    want = [1, 2, 2, 2, 1, 1]
    for cfg, w in zip(bad, want):
        assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(h)) == w
        assert not h.value
    assert lib.moe_create(None, ctypes.byref(h)) == 1
    assert lib.moe_sync(None) == 1
    assert lib.moe_last_error(None) == b"null handle"
