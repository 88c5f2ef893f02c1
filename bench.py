#!/usr/bin/env python
"""Throughput of the routed MoE layer on one or more GB300s (one replica per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the whole layer (router, scan, placement, gather,
GEMM1+SwiGLU, GEMM2, shared expert if any, finalize) on one batch of seeded
synthetic tokens whose inputs are already in HBM. The headline workload is the
largest configuration that fits one GPU: the CFG-doubled denoise layer (32768
tokens, H=4096, 64 experts, top-8, two micro-shards of I=1536, and a dense
shared expert of 3072). Between steps the token batch rotates through a pool of
seeded batches; the expert weights (4.9 GB) are far larger than L2.

The same JSON line carries, under "workloads", one record per other
configuration (AR decode, decode with MXFP8 expert weights, the two-micro
denoise, the skewed large denoise, the tiny fp32 layer), each with its own
timing, roofline, end-to-end figure and CPU-oracle baseline.

Prints one JSON line on rank 0. ``--impl reference`` times the fp64 CPU oracle
on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import math
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
import traceback

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_layer_warp_gb300 import binding  # noqa: E402
from mixture_experts_layer_warp_gb300 import workloads as W  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 GB300; % of binding roof (bf16 TC peak or HBM)"
POOL = 8  # distinct token batches rotated through the timed steps
HEADLINE = "cfg_shared"
# the other configurations, measured in the same run ("decode_mxfp8": the
# decode workload with MXFP8 expert weights)
SUB_WORKLOADS = ("decode", "decode_mxfp8", "denoise_multi_micro", "denoise_multi_micro_mxfp8", "skewed",
                 "tiny_fp32")
FP32_LANES_PER_SM = 128  # FP32 FMA units per SM (one FMA = 2 flop per clock)
FP8_PER_BF16 = 2.0  # nominal dense tensor-core rate of fp8 over bf16 (4.5 / 2.25 PFLOP/s)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        out = dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sustained=p["bf16_tflops_sustained"],
                   sm_max_mhz=p.get("sm_max_mhz", 2070.0), source="measured")
    else:
        out = dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, sm_max_mhz=2070.0, source="fallback")
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    # plain fp32 FMA arithmetic (the exact-fp32 GEMMs of fp32 layers): every
    # FP32 lane of every SM retiring one FMA per clock at the maximum SM clock
    out["fp32_alu"] = sms * FP32_LANES_PER_SM * 2 * out["sm_max_mhz"] * 1e6 / 1e12
    out["sms"] = sms
    return out


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def wait_first_sample(self, timeout_s: float = 3.0):
        """Block until nvidia-smi has written its first line (it needs a moment to start)."""
        t0 = time.time()
        while self.proc is not None and self.path is not None and time.time() - t0 < timeout_s:
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        watts = [float(r[3]) for r in rows if r[3] not in ("", "[N/A]")]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(watts) if watts else None,
                "window": f"the timed steps plus {ROLL_S} s of the same steps run back to back before and "
                          f"after them (nvidia-smi samples every 200 ms)"}


# ---------------------------------------------------------------- helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """Largest value over the replicas (the slowest rank's time)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, steps: int, ms_local: float):
    """Whole-job tokens/s of N independent replicas (weak scaling): every rank
    runs `steps` steps of `tokens_per_step` tokens; the job takes as long as the
    slowest rank. Returns (ms_max, tokens_per_s)."""
    ms = max_over_ranks(ms_local, world)
    return ms, world * tokens_per_step * steps / (ms / 1e3)


# The sources each GEMM kernel is compiled from (its translation unit and the
# headers it includes): the small-batch fused kernel, the large-batch tcgen05 GEMM.
KERNEL_SOURCES = {
    "small": ("gemm_small.cu", "gemm_common.cuh", "kernels.h", "ptx.cuh"),
    "large": ("gemm_pair.cu", "gemm_common.cuh", "kernels.h", "ptx.cuh"),
}


def src_sha(kind: str) -> str:
    """Hash of the CUDA sources of one GEMM kernel (KERNEL_SOURCES): recorded
    ncu counters are used only while this matches the hash stored beside them."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "mixture_experts_layer_warp_gb300", "csrc")
    for n in KERNEL_SOURCES[kind]:
        with open(os.path.join(d, n), "rb") as f:
            h.update(n.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str, sha: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    kernel source has not changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == workload and parts[1] == kernel and parts[2] == sha:
                return float(parts[3])
    return None


def oracle_tokens_per_s(wl, host_pool, weights, budget_s: float, min_calls: int = 1):
    """The fp64 oracle on the host cores: whole-layer calls on sample batches."""
    import oracle
    n_tok, calls = 0, 0
    t0 = time.perf_counter()
    while calls < min_calls or time.perf_counter() - t0 < budget_s:
        x = host_pool[calls % len(host_pool)]
        oracle.layer(x, weights["router_w"], weights["router_bias"], weights["w13"], weights["w2"], wl.k,
                     weights["shared_w13"], weights["shared_w2"])
        n_tok += x.shape[0]
        calls += 1
    dt = time.perf_counter() - t0
    return n_tok / dt, calls, dt, oracle.num_threads()


# fp32 logit tolerance for calling a token's top-k decided: the spread of fp32
# sums over H = 4096 products in different orders (the routing tests use it too)
ROUTE_TAU = 4e-6


def routing_check(layer, wl, x, inp, weights) -> dict:
    """The routing contract on one timed batch: the oracle's fp64 logits,
    rounded to fp32, against the CUDA routing of the same batch. A token is
    undecided when its k-th and (k+1)-th logits (set) or two adjacent top-k
    logits (order) lie within 2 * tau, so either choice is correct; every
    decided token must carry the oracle's ids in the oracle's order. fp32
    layers form their logits exactly enough that tau is 0 there."""
    import oracle
    tau = ROUTE_TAU if wl.dtype == "bf16" else 0.0
    lg = oracle.logits(W.to_numpy(x), weights["router_w"], weights["router_bias"])
    ids_o, _ = oracle.route(lg, wl.k)
    ids_g = layer.route(x, inp["router_w"], inp["router_bias"])["ids"].cpu().numpy()
    lf = lg.astype(np.float32).astype(np.float64)
    srt = -np.sort(-lf, axis=1)
    k, E = wl.k, wl.E
    set_ok = (srt[:, k - 1] - srt[:, k]) > 2 * tau if k < E else np.ones(len(lf), bool)
    order_ok = set_ok & np.all((srt[:, :k - 1] - srt[:, 1:k]) > 2 * tau, axis=1)
    if tau == 0:
        set_ok[:] = True
        order_ok[:] = True
    return {"tokens": int(len(lf)), "set_undecided": int((~set_ok).sum()),
            "order_undecided": int((~order_ok).sum()),
            "decided_mismatch": int((order_ok & np.any(ids_g != ids_o, axis=1)).sum()),
            "tau": tau}


def host_weights(inp):
    out = {}
    for k in ("router_w", "shared_w13", "shared_w2"):
        out[k] = W.to_numpy(inp[k]) if inp[k] is not None else None
    out["router_bias"] = None if inp["router_bias"] is None else inp["router_bias"].cpu().numpy()
    out["w13"] = [W.to_numpy(t) for t in inp["w13"]]
    out["w2"] = [W.to_numpy(t) for t in inp["w2"]]
    return out


def sample_tokens(wl) -> int:
    """Tokens per oracle sample call: whole batch when small, else a slice
    sized to a few seconds of fp64 work."""
    per_token = 6 * wl.k * wl.H * wl.I * wl.n_micro + 6 * wl.H * wl.shared_inter
    return int(max(1, min(wl.T, 4e10 // per_token)))


# ---------------------------------------------------------------- arms
def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    torch.cuda.set_device(0) if torch.cuda.is_available() else None
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.make_inputs(wl, seed=0, device=dev)
    weights = host_weights(inp)
    del inp
    Ts = sample_tokens(wl)
    pool = [W.to_numpy(W.make_inputs(wl, seed=100 + i, device=dev, experts=False, T=Ts)["x"])
            for i in range(max(2, min(POOL, args.steps)))]
    import oracle
    for i in range(args.warmup):
        oracle.layer(pool[i % len(pool)], weights["router_w"], weights["router_bias"], weights["w13"],
                     weights["w2"], wl.k, weights["shared_w13"], weights["shared_w2"])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.layer(pool[i % len(pool)], weights["router_w"], weights["router_bias"], weights["w13"],
                     weights["w2"], wl.k, weights["shared_w13"], weights["shared_w2"])
    dt = time.perf_counter() - t0
    value = Ts * args.steps / dt
    sample = f"{Ts} of {wl.T} tokens per step (whole layer: routing, permutation, per-token experts)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl, mx=False):
    cfg = {"workload": wl.name, "T": wl.T, "hidden": wl.H, "experts": wl.E, "top_k": wl.k, "inter": wl.I,
           "n_micro": wl.n_micro, "shared_inter": wl.shared_inter, "dtype": wl.dtype,
           "router": wl.router_init + ("+log_zipf_bias" if wl.router_bias else ""),
           "l2": "inputs larger than L2: expert weights exceed the 129 MB L2; token batches rotate over "
                 f"{POOL} seeded batches"}
    if wl.T * wl.E * wl.H < 2 ** 25:  # the tiny layer: weights fit in L2
        cfg["l2"] = f"inputs smaller than L2 (a correctness-sized layer); token batches rotate over {POOL} " \
                    "seeded batches"
    if mx:
        cfg["weights"] = "mxfp8 (E4M3 codes, E8M0 scale per 32 along K)"
        cfg["activations"] = "mxfp8 token rows and h (block-scaled FP8 MMA, fp32 accumulate)"
    return cfg


def gemm_flops(wl) -> dict:
    """Algorithmic flops per launch of each GEMM slot (padding never counts)."""
    R = wl.T * wl.k
    return {"gemm1_swiglu": 4 * R * wl.H * wl.I * wl.n_micro, "gemm2_down": 2 * R * wl.H * wl.I * wl.n_micro,
            "shared_gemm1": 4 * wl.T * wl.H * wl.shared_inter, "shared_gemm2": 2 * wl.T * wl.H * wl.shared_inter}


def roofline_of(wl, prof, ids_pool, steps, peaks, step_ms, clocks, mxfp8=False):
    """Roofline of the kernel with the largest share of the timed region.

    Decode-sized bf16 layers are bound by HBM (the touched experts' weights),
    the large bf16 layers by the tensor cores (rated against the burst bf16
    peak; the fraction of the sustained peak is reported beside it), fp32
    layers by plain FP32 FMA arithmetic."""
    dom, (ms, n) = max(prof.items(), key=lambda kv: kv[1][0])
    per_launch_s = ms / n / 1e3
    R = wl.T * wl.k
    esz = 4 if wl.dtype == "f32" else 2
    wsz = (1 + 1 / 32) if mxfp8 else esz  # bytes per expert weight (MXFP8: code + a 32nd of a scale)
    asz = wsz  # bytes per element of the gathered rows and h (MXFP8 with MXFP8 weights)
    # touched experts per step, averaged over the batches the timed steps used
    touched = statistics.mean(len(np.unique(ids_pool[i % len(ids_pool)])) for i in range(steps))
    I, H, M = wl.I, wl.H, wl.n_micro
    fused = "gemm2_down" not in prof and wl.dtype == "bf16"  # small batches run both GEMMs in one launch
    flops = gemm_flops(wl)
    extra = {}
    if wl.dtype == "f32":
        bound, unit, peak = "alu", "TFLOP/s", peaks["fp32_alu"]
        algo = flops.get(dom)
        achieved = algo / per_launch_s / 1e12 if algo else None
        peak_kind = (f"fp32 FMA peak: {peaks['sms']} SMs x {FP32_LANES_PER_SM} lanes x 2 flop x "
                     f"{peaks['sm_max_mhz']:g} MHz")
    elif wl.T <= 16:
        bound, unit, peak = "hbm", "GB/s", peaks["hbm"]
        algo = {
            "gemm1_swiglu": (touched * 3 * I * H * wsz * M + R * H * esz + 2 * R * H * asz + 2 * R * M * I * asz
                             + wl.T * H * esz)
            if fused
            else (touched * 2 * I * H * esz * M + R * H * esz + R * M * I * esz),
            "gemm2_down": touched * H * I * esz * M + R * M * I * esz + R * H * esz,
            "gather": 2 * R * H * esz,
            "finalize": R * H * esz + wl.T * H * esz,
            "router": wl.T * H * esz + wl.E * H * esz,
        }.get(dom)
        achieved = algo / per_launch_s / 1e9 if algo else None
        peak_kind = "measured copy bandwidth"
    else:
        # block-scaled FP8 GEMMs: the bf16 peaks times the nominal fp8 : bf16
        # dense tensor ratio (4.5 : 2.25 PFLOP/s)
        ratio = FP8_PER_BF16 if mxfp8 else 1.0
        bound, unit, peak = "tensor", "TFLOP/s", peaks["bf16"] * ratio
        algo = flops.get(dom)
        achieved = algo / per_launch_s / 1e12 if algo else None
        peak_kind = ("fp8: measured cuBLAS bf16 burst x 2 (nominal fp8:bf16 dense ratio)" if mxfp8
                     else "burst (measured cuBLAS bf16 GEMM)")
        if achieved:
            extra["frac_sustained"] = achieved / (peaks["bf16_sustained"] * ratio)
        # every GEMM launch of the step together: their flops over their summed time
        g_ms = sum(prof[s][0] for s in flops if s in prof)
        g_fl = sum(flops[s] * prof[s][1] for s in flops if s in prof)
        if g_ms > 0:
            extra["gemms"] = {"achieved": g_fl / (g_ms / 1e3) / 1e12, "frac": g_fl / (g_ms / 1e3) / 1e12 / peak,
                              "ms_per_step": g_ms / steps,
                              "kernels": [s for s in flops if s in prof]}
        capped = clocks is not None and "sw_power_cap" in clocks.get("reasons", [])
        extra["power_capped"] = capped
    sha = src_sha("small" if fused else "large")
    traffic = recorded_traffic(wl.name + ("_mxfp8" if mxfp8 else ""), dom, sha)
    out = {"kernel": dom + ("+gemm2_down+finalize (one launch)" if fused and dom == "gemm1_swiglu" else ""),
           "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
           "frac": (achieved / peak) if achieved else None, "traffic": traffic,
           "algorithmic_per_launch": algo, "launch_ms": per_launch_s * 1e3,
           "share": ms / sum(v[0] for v in prof.values()), "peak_source": peaks["source"],
           "peak_kind": peak_kind,
           "timing": "per-kernel CUDA events in a profiling pass of the same steps"}
    out.update(extra)
    return out


def time_two_dispatch(args, wl, inp, pool, multi_ms, world):
    """The pages' ablation baseline ("HunyuanImage3 Hybrid Parallelism",
    section 10.3): one full layer call per micro-shard, outputs added (here the
    later calls accumulate into the first one's y), against the multi-micro
    layer that shares one routing, permutation and finalize."""
    layers = [binding.MoELayer(wl.H, wl.E, wl.k, wl.I, 1, max_tokens=wl.T,
                               shared_inter=wl.shared_inter if m == 0 else 0, dtype=wl.torch_dtype)
              for m in range(wl.n_micro)]
    for lay in layers[1:]:
        lay.set_accumulate(True)
    y = torch.empty((wl.T, wl.H), dtype=wl.torch_dtype, device="cuda")

    def step(i):
        x = pool[i % POOL]
        for m, lay in enumerate(layers):
            lay.forward(x, inp["router_w"], inp["router_bias"], [inp["w13"][m]], [inp["w2"][m]],
                        inp["shared_w13"] if m == 0 else None, inp["shared_w2"] if m == 0 else None, out=y)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for i in range(args.steps):
        step(args.warmup + i)
    ev1.record()
    ev1.synchronize()
    for lay in layers:
        lay.sync()
        lay.close()
    two_ms = max_over_ranks(ev0.elapsed_time(ev1), world) / args.steps
    return {"ms_per_step": two_ms, "multi_micro_ms_per_step": multi_ms, "saving_ms": two_ms - multi_ms,
            "saving_pct_of_two_dispatch": 100.0 * (two_ms - multi_ms) / two_ms}


ROLL_S = 0.3  # untimed load before and after the timed steps, so that clock samples see it


def roll_steps(step_ms: float) -> int:
    """Steps of about ROLL_S seconds, run untimed around the timed region."""
    return int(min(20000, max(1, math.ceil(ROLL_S * 1e3 / max(step_ms, 1e-3)))))


def measure(args, wl, world, rank, local, peaks, mx=False, cpu_seconds=12.0, two_dispatch=False) -> dict:
    """Times `args.steps` layer calls of workload `wl` (inputs resident in HBM),
    then the per-kernel split, the end-to-end host-buffer path and the CPU
    oracle; returns the record of the JSON line."""
    inp = W.make_inputs(wl, seed=0, device="cuda")
    pool = [W.make_inputs(wl, seed=100 + i, device="cuda", experts=False)["x"] for i in range(POOL)]
    layer = binding.MoELayer(wl.H, wl.E, wl.k, wl.I, wl.n_micro, max_tokens=wl.T,
                             shared_inter=wl.shared_inter, dtype=wl.torch_dtype)
    if args.shared_stream:
        layer.set_shared_stream(True)
    y = torch.empty((wl.T, wl.H), dtype=wl.torch_dtype, device="cuda")
    args_w = (inp["router_w"], inp["router_bias"], inp["w13"], inp["w2"], inp["shared_w13"], inp["shared_w2"])
    if mx:  # quantised once, outside every timed region (as weights are at load time)
        args_w = (inp["router_w"], inp["router_bias"], [binding.quantize_mxfp8(t) for t in inp["w13"]],
                  [binding.quantize_mxfp8(t) for t in inp["w2"]], inp["shared_w13"], inp["shared_w2"])

    def step(i):
        if mx:
            layer.forward_mxfp8(pool[i % POOL], *args_w, out=y)
        else:
            layer.forward(pool[i % POOL], *args_w, out=y)

    ids_pool = [layer.route(x, inp["router_w"], inp["router_bias"])["ids"].cpu().numpy() for x in pool]
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.warmup):
        step(i)
    ev1.record(stream)
    layer.sync()
    roll = roll_steps(ev0.elapsed_time(ev1) / max(args.warmup, 1))

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.wait_first_sample()
        for i in range(roll):  # untimed: the same load, so the clock samples see it
            step(i)
        l0 = layer.launch_count()
        ev0.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        ev1.record(stream)
        launches = layer.launch_count() - l0
        for i in range(roll):
            step(i)
        ev1.synchronize()
        torch.cuda.synchronize()
    clocks = clk.summary()
    barrier(world)
    layer.sync()
    ms, value = job_throughput(world, wl.T, args.steps, ev0.elapsed_time(ev1))

    # per-kernel durations: the same steps again with an event pair around every
    # launch (kept out of the timed region above, whose launches run back to back)
    layer.profile_begin(args.steps)
    for i in range(args.steps):
        step(args.warmup + i)
    prof = layer.profile_end()
    layer.sync()
    shift = args.warmup % POOL
    ids_timed = ids_pool[shift:] + ids_pool[:shift]
    roof = roofline_of(wl, prof, ids_timed, args.steps, peaks, ms / args.steps, clocks, mxfp8=mx)

    # end to end through the C ABI with host buffers (pinned), copies included
    esz = 4 if wl.dtype == "f32" else 2
    n_host = POOL if wl.T * wl.H * esz <= (64 << 20) else 2  # large batches: two pinned host batches
    host_pool = [pool[i].cpu().pin_memory() for i in range(n_host)]
    y_hosts = [torch.empty((wl.T, wl.H), dtype=wl.torch_dtype).pin_memory() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step(i):
        # the serving loop's form: each call enqueues its own copies and returns;
        # call i+1's copy of x and call i-1's copy of y overlap call i
        if mx:
            layer.forward_mxfp8(host_pool[i % n_host], *args_w, out=y_hosts[i % 2], host_async=True)
        else:
            layer.forward_host(host_pool[i % n_host], *args_w, out_host=y_hosts[i % 2], wait=False)

    for i in range(2):
        e2e_step(i)
    layer.sync()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    layer.sync()  # every step's y is in host memory
    _, e2e_value = job_throughput(world, wl.T, e2e_steps, (time.perf_counter() - t0) * 1e3)
    e2e = {"value": e2e_value, "unit": "tokens/s",
           "h2d_bytes_per_step": wl.T * wl.H * esz, "d2h_bytes_per_step": wl.T * wl.H * esz,
           "entry_point": ("moe_forward_mxfp8_host_async" if mx else "moe_forward_host_async") +
           " from pinned buffers, calls back to back, one moe_sync after the last"}
    del host_pool, y_hosts

    two = None
    if two_dispatch and wl.n_micro > 1 and not mx:
        two = time_two_dispatch(args, wl, inp, pool, ms / args.steps, world)

    cpu = rcheck = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        weights = host_weights(inp)
        Ts = sample_tokens(wl)
        hp = [W.to_numpy(x[:Ts]) for x in pool]
        v, calls, dt, cores = oracle_tokens_per_s(wl, hp, weights, budget_s=cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{calls} whole-layer oracle calls of {Ts} of the {wl.T} tokens ({dt:.1f} s)"}
        if wl.T <= 64:  # the small configurations are also timed on one core
            import oracle
            oracle.set_threads(1)
            v1, calls1, dt1, _ = oracle_tokens_per_s(wl, hp, weights, budget_s=cpu_seconds / 2)
            oracle.set_threads(cores)
            cpu["single_core"] = {"value": v1, "unit": "tokens/s", "cores": 1,
                                  "sample": f"{calls1} whole-layer oracle calls of {Ts} tokens ({dt1:.1f} s)"}
        rcheck = routing_check(layer, wl, pool[0], inp, weights)
        del weights

    layer.close()
    rec = {"value": value, "unit": "tokens/s", "ms_per_step": ms / args.steps, "steps": args.steps,
           "warmup": args.warmup,
           "dtype": "e4m3 (mxfp8 weights and activations)"
           if mx else wl.dtype,
           "config": dict(config_of(wl, mx), **({"shared_stream": True} if args.shared_stream else {})),
           "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
           "kernels_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
           "clocks": clocks}
    if rcheck is not None:
        rec["routing_check"] = rcheck
    if two is not None:
        rec["two_dispatch"] = two
    del inp, pool, y, args_w, layer
    gc.collect()
    torch.cuda.empty_cache()
    return rec


def sub_workload(name):
    """(Workload, mxfp8 weights?) of a name in SUB_WORKLOADS."""
    if name.endswith("_mxfp8"):
        return W.WORKLOADS[name[: -len("_mxfp8")]], True
    return W.WORKLOADS[name], False


def run_ours(args, wl, world, rank, local):
    peaks = load_peaks()
    mx = args.weights == "mxfp8"
    head = measure(args, wl, world, rank, local, peaks, mx=mx, cpu_seconds=args.cpu_seconds,
                   two_dispatch=args.two_dispatch)
    subs = {}
    if not args.no_sub:
        for name in SUB_WORKLOADS:
            swl, smx = sub_workload(name)
            if swl.name == wl.name and smx == mx:
                continue
            try:
                subs[name] = measure(args, swl, world, rank, local, peaks, mx=smx, cpu_seconds=args.sub_cpu_seconds,
                                     two_dispatch=args.two_dispatch)
            except Exception as exc:  # noqa: BLE001 - recorded in the line; the headline stands
                subs[name] = {"error": f"{type(exc).__name__}: {exc}"}
                traceback.print_exc()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic", "config": head["config"],
        "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"], "kernels_ms_per_step": head["kernels_ms_per_step"],
        "clocks": head["clocks"],
    }
    for k in ("routing_check", "two_dispatch"):
        if k in head:
            line[k] = head[k]
    if subs:
        line["workloads"] = subs
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS), default=HEADLINE)
    ap.add_argument("--no-sub", action="store_true",
                    help="measure only --workload (no per-configuration records under 'workloads')")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sub-cpu-seconds", type=float, default=4.0,
                    help="CPU-oracle sample length of each record under 'workloads'")
    ap.add_argument("--weights", choices=["bf16", "mxfp8"], default="bf16",
                    help="routed expert weights: the layer dtype, or MXFP8 (moe_forward_mxfp8)")
    ap.add_argument("--shared-stream", action="store_true",
                    help="run the shared expert's GEMMs on a second stream (moe_set_shared_stream)")
    ap.add_argument("--no-two-dispatch", dest="two_dispatch", action="store_false",
                    help="skip the two-dispatch comparison of the multi-micro workloads")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = W.WORKLOADS[args.workload]
    world, rank, local = (1, 0, 0)
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, wl, int(os.environ.get("WORLD_SIZE", "1")), rank)
        return
    world, rank, local = dist_setup()
    run_ours(args, wl, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
