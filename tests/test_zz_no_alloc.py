"""moe_route_noalloc: routing for callers that cannot allocate device memory
(their device heap belongs to a fixed-budget pool, or their hot path must not
take cudaMalloc's implicit synchronisation). It keeps its intermediate data in
a file-scope device array of the library instead of a handle's workspace.

Checked through the C ABI against moe_route on two calls in a row with
different inputs (the shared array keeps the first call's contents when the
second one starts), and against its size limit. This file is collected last.
"""
import ctypes

import pytest
import torch

from mixture_experts_layer_warp_gb300 import binding
from mixture_experts_layer_warp_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(lib, x, wr, bias, k, dtype_code):
    T, H = x.shape
    E = wr.shape[0]
    out = dict(ids=torch.empty((T, k), dtype=torch.int32, device="cuda"),
               w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
               perm=torch.empty((T * k,), dtype=torch.int32, device="cuda"),
               offsets=torch.empty((E + 1,), dtype=torch.int32, device="cuda"))
    rc = lib.moe_route_noalloc(x.data_ptr(), wr.data_ptr(), None if bias is None else bias.data_ptr(), T, H, E, k,
                               dtype_code, out["ids"].data_ptr(), out["w"].data_ptr(), out["perm"].data_ptr(),
                               out["offsets"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc, out


def test_noalloc_routing_matches_moe_route_on_two_calls_in_a_row():
    lib = binding.load()
    cases = [(W.Workload("a", 3000, 4096, 64, 8, 768, 1, router_bias="log_zipf"), torch.bfloat16, 1),
             (W.Workload("b", 777, 512, 16, 4, 128, 1), torch.bfloat16, 1)]
    for call, (wl, dt, code) in enumerate(cases):
        inp = W.make_inputs(wl, seed=10 + call, device="cuda", experts=False)
        layer = binding.MoELayer(wl.H, wl.E, wl.k, 128, 1, max_tokens=wl.T, dtype=dt)
        ref = layer.route(inp["x"], inp["router_w"], inp["router_bias"])
        layer.sync()
        rc, got = _noalloc(lib, inp["x"], inp["router_w"], inp["router_bias"], wl.k, code)
        assert binding.STATUS[rc] == "MOE_OK"
        torch.cuda.synchronize()
        assert torch.equal(got["ids"], ref["ids"]), call
        assert torch.equal(got["perm"], ref["perm"]), call
        assert torch.equal(got["offsets"], ref["offsets"]), call
        assert (got["w"] - ref["w"]).abs().max().item() <= 1e-5, call
        layer.close()


def test_noalloc_rejects_sizes_beyond_its_limit():
    lib = binding.load()
    limit = 16384
    x = torch.zeros((limit + 1, 256), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    rc, _ = _noalloc(lib, x, wr, None, 2, 1)
    assert binding.STATUS[rc] == "MOE_ERR_INVALID_ARG"
    rc, _ = _noalloc(lib, x[:limit], wr, None, 2, 1)
    assert binding.STATUS[rc] == "MOE_OK"
    torch.cuda.synchronize()
