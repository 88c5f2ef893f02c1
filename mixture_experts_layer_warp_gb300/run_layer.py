"""Run one of the seeded workloads through the layer a few times.

    python -m mixture_experts_layer_warp_gb300.run_layer --workload NAME [--tokens T] [--calls N]
                                                        [--weights bf16|mxfp8]

For profiling a call sequence outside the benchmark (an ncu capture of a
kernel picks its launches with -k / -s / -c): it draws the workload's inputs
(``workloads.make_inputs``, seed 0, on the GPU), optionally with a smaller
token count than the workload's own (the weights are unchanged), makes one
layer handle and issues N forward calls back to back, then synchronises and
checks the handle's device error word.
"""
from __future__ import annotations

import argparse

import torch

from . import binding
from . import workloads as W


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS), required=True)
    ap.add_argument("--tokens", type=int, default=0, help="token count (default: the workload's)")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--weights", choices=["bf16", "mxfp8"], default="bf16")
    args = ap.parse_args(argv)
    wl = W.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.with_tokens(args.tokens)
    torch.cuda.set_device(0)
    inp = W.make_inputs(wl, seed=0, device="cuda")
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=wl.T, shared_inter=wl.shared_inter,
                             dtype=wl.torch_dtype)
    w13, w2 = inp["w13"], inp["w2"]
    if args.weights == "mxfp8":
        w13 = [binding.quantize_mxfp8(t) for t in w13]
        w2 = [binding.quantize_mxfp8(t) for t in w2]
    for _ in range(args.calls):
        if args.weights == "mxfp8":
            layer.forward_mxfp8(inp["x"], inp["router_w"], inp["router_bias"], w13, w2, inp["shared_w13"],
                                inp["shared_w2"])
        else:
            layer.forward(inp["x"], inp["router_w"], inp["router_bias"], w13, w2, inp["shared_w13"],
                          inp["shared_w2"])
    layer.sync()
    layer.close()
    print(f"{wl.name}: T={wl.T}, {args.calls} calls, {args.weights} expert weights: ok")


if __name__ == "__main__":
    main()
