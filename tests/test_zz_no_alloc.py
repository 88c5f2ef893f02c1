"""moe_route_noalloc: routing for callers that cannot allocate device memory
(their device heap belongs to a fixed-budget pool, or their hot path must not
take cudaMalloc's implicit synchronisation). It keeps its intermediate data in
a file-scope device array of the library instead of a handle's workspace.

Checked through the C ABI against moe_route on two calls in a row with
different inputs and routing paths (the shared array keeps the first call's
contents when the second one starts), through its status query, and against its
size limit. This file is collected last.
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


# every routing path the entry point can take: the multi-CTA tensor-core router
# with scan and placement (T > 128), the single-CTA router with fused scan and
# placement (16 < T <= 128), the 8-CTA cluster router (T <= 16), and the fp32
# SIMT router whose histogram uses every row of the array (T at the limit)
CASES = [
    (W.Workload("a", 3000, 4096, 64, 8, 768, 1, router_bias="log_zipf"), torch.bfloat16, 1),
    (W.Workload("b", 777, 512, 16, 4, 128, 1), torch.bfloat16, 1),
    (W.Workload("c", 8, 4096, 64, 8, 768, 1), torch.bfloat16, 1),
    (W.Workload("d", 100, 512, 64, 8, 128, 1), torch.bfloat16, 1),
    (W.Workload("e", 16384, 256, 8, 2, 64, 1, dtype="f32"), torch.float32, 0),
]


@pytest.mark.parametrize("first,second", [(0, 1), (2, 3), (4, 2), (3, 4)])
def test_noalloc_routing_matches_moe_route_on_two_calls_in_a_row(first, second):
    """Two different calls back to back (the second starts with the first one's
    data left in the shared array), each equal to moe_route bit for bit, and
    the status query reports a clean run after each."""
    lib = binding.load()
    stream = torch.cuda.current_stream().cuda_stream
    for call, idx in enumerate((first, second)):
        wl, dt, code = CASES[idx]
        inp = W.make_inputs(wl, seed=10 + 7 * idx + call, device="cuda", experts=False)
        layer = binding.MoELayer(wl.H, wl.E, wl.k, 128 if dt == torch.bfloat16 else 64, 1, max_tokens=wl.T,
                                 dtype=dt)
        ref = layer.route(inp["x"], inp["router_w"], inp["router_bias"])
        layer.sync()
        rc, got = _noalloc(lib, inp["x"], inp["router_w"], inp["router_bias"], wl.k, code)
        assert binding.STATUS[rc] == "MOE_OK"
        assert binding.STATUS[lib.moe_route_noalloc_status(stream)] == "MOE_OK"
        assert torch.equal(got["ids"], ref["ids"]), (wl.name, call)
        assert torch.equal(got["perm"], ref["perm"]), (wl.name, call)
        assert torch.equal(got["offsets"], ref["offsets"]), (wl.name, call)
        assert (got["w"] - ref["w"]).abs().max().item() <= 1e-5, (wl.name, call)
        layer.close()


def test_noalloc_rejects_sizes_beyond_its_limit():
    lib = binding.load()
    limit = 16384
    x = torch.zeros((limit + 1, 256), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    rc, _ = _noalloc(lib, x, wr, None, 2, 1)
    assert binding.STATUS[rc] == "MOE_ERR_INVALID_ARG"
    rc, got = _noalloc(lib, x[:limit], wr, None, 2, 1)
    assert binding.STATUS[rc] == "MOE_OK"
    assert binding.STATUS[lib.moe_route_noalloc_status(torch.cuda.current_stream().cuda_stream)] == "MOE_OK"
    # all logits tie (zero inputs): every token takes experts 0 and 1, in order
    assert got["offsets"].tolist() == [0, limit, 2 * limit] + [2 * limit] * 6
    assert torch.equal(got["ids"].cpu(), torch.tensor([[0, 1]], dtype=torch.int32).expand(limit, 2))
