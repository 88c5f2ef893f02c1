"""Host logic of the benchmark, without a GPU: the roofline's peak choice and
algorithmic work, the traffic records' keying to the kernels' sources, and the
whole-job throughput."""
import os
import re

import numpy as np
import pytest

import bench
from mixture_experts_layer_warp_gb300 import workloads as W

PEAKS = dict(hbm=6783.1, bf16=1891.6, bf16_sustained=1690.3, source="measured", fp32_alu=80.55, sms=152,
             sm_max_mhz=2070.0)


def _large_prof(gemm1_ms, n=10):
    # total ms and launches per slot, as the profiling pass returns them
    return {"router": (0.05 * n, n), "gemm1_swiglu": (gemm1_ms * n, n), "gemm2_down": (gemm1_ms * n / 2, n)}


def test_large_gemms_are_rated_against_the_burst_peak():
    wl = W.WORKLOADS["cfg_shared"]
    ids = [np.zeros((wl.T, wl.k), np.int32)]
    flops = 4 * wl.T * wl.k * wl.H * wl.I * wl.n_micro
    for step_ms, clocks in [(15.0, {"reasons": ["sw_power_cap"]}), (15.0, {"reasons": []}), (15.0, None),
                            (1.5, {"reasons": ["sw_power_cap"]})]:
        r = bench.roofline_of(wl, _large_prof(8.0), ids, 1, PEAKS, step_ms, clocks)
        assert r["bound"] == "tensor" and r["kernel"] == "gemm1_swiglu"
        assert r["peak"] == PEAKS["bf16"] and r["peak_kind"].startswith("burst")
        assert r["achieved"] == pytest.approx(flops / 8.0e-3 / 1e12)
        assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["bf16"])
        assert r["frac_sustained"] == pytest.approx(r["achieved"] / PEAKS["bf16_sustained"])
        assert r["power_capped"] == bool(clocks and clocks["reasons"])


def test_all_gemm_launches_of_a_step_are_rated_together():
    wl = W.WORKLOADS["cfg_shared"]
    ids = [np.zeros((wl.T, wl.k), np.int32)]
    n = 10
    prof = {"router": (0.05 * n, n), "gemm1_swiglu": (8.0 * n, n), "gemm2_down": (4.0 * n, n),
            "shared_gemm1": (1.0 * n, n), "shared_gemm2": (0.5 * n, n), "finalize": (0.4 * n, n)}
    r = bench.roofline_of(wl, prof, ids, n, PEAKS, 15.0, None)
    R = wl.T * wl.k
    fl = 6 * R * wl.H * wl.I * wl.n_micro + 6 * wl.T * wl.H * wl.shared_inter
    g = r["gemms"]
    assert g["ms_per_step"] == pytest.approx(13.5)
    assert g["achieved"] == pytest.approx(fl / 13.5e-3 / 1e12)
    assert g["frac"] == pytest.approx(g["achieved"] / PEAKS["bf16"])
    assert sorted(g["kernels"]) == ["gemm1_swiglu", "gemm2_down", "shared_gemm1", "shared_gemm2"]


def test_fp32_layers_are_rated_against_the_fp32_fma_peak():
    wl = W.WORKLOADS["tiny_fp32"]
    ids = [np.zeros((wl.T, wl.k), np.int32)]
    peaks = dict(PEAKS, fp32_alu=152 * 128 * 2 * 2070e6 / 1e12, sms=152, sm_max_mhz=2070.0)
    prof = {"router": (0.02, 10), "gemm1_swiglu": (0.3, 10), "gemm2_down": (0.2, 10)}
    r = bench.roofline_of(wl, prof, ids, 10, peaks, 0.1, None)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["peak"] == pytest.approx(80.55, rel=1e-3)
    flops = 4 * wl.T * wl.k * wl.H * wl.I
    assert r["achieved"] == pytest.approx(flops / 0.03e-3 / 1e12)


def test_every_sub_workload_names_a_configuration():
    for name in bench.SUB_WORKLOADS:
        wl, mx = bench.sub_workload(name)
        assert wl.name in W.WORKLOADS and mx == name.endswith("_mxfp8")
    assert bench.HEADLINE == "cfg_shared"
    covered = {bench.sub_workload(n)[0].name for n in bench.SUB_WORKLOADS} | {bench.HEADLINE}
    assert covered == set(W.WORKLOADS)


def test_decode_is_rated_against_hbm_over_the_touched_experts():
    wl = W.WORKLOADS["decode"]
    ids = [(np.arange(wl.T * wl.k, dtype=np.int32) % 40).reshape(wl.T, wl.k)]  # 40 experts touched
    prof = {"router": (0.1, 10), "gemm1_swiglu": (1.3, 10)}  # the fused launch: no separate GEMM2
    r = bench.roofline_of(wl, prof, ids, 1, PEAKS, 0.13, None)
    assert r["bound"] == "hbm" and r["peak"] == PEAKS["hbm"]
    assert r["kernel"].startswith("gemm1_swiglu+gemm2_down+finalize")
    weights = 40 * 3 * wl.I * wl.H * 2
    assert weights < r["algorithmic_per_launch"] < weights + 2e6  # plus token rows, h, o, y
    assert r["achieved"] == pytest.approx(r["algorithmic_per_launch"] / 0.13e-3 / 1e9)
    mx = bench.roofline_of(wl, prof, ids, 1, PEAKS, 0.09, None, mxfp8=True)
    assert mx["algorithmic_per_launch"] < 0.6 * r["algorithmic_per_launch"]  # 1 + 1/32 bytes per weight


def test_traffic_records_are_used_only_for_matching_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text("# a comment line\ndecode gemm1_swiglu abc 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("decode", "gemm1_swiglu", "abc") == 123.0
    assert bench.recorded_traffic("decode", "gemm1_swiglu", "abd") is None
    assert bench.recorded_traffic("decode_mxfp8", "gemm1_swiglu", "abc") is None
    assert bench.recorded_traffic("decode", "gemm2_down", "abc") is None


def test_kernel_source_lists_cover_everything_their_kernels_include():
    d = os.path.join(bench.ROOT, "mixture_experts_layer_warp_gb300", "csrc")
    for kind, files in bench.KERNEL_SOURCES.items():
        seen, todo = set(), [files[0]]
        while todo:
            f = todo.pop()
            if f not in seen:
                seen.add(f)
                with open(os.path.join(d, f)) as src:
                    todo += re.findall(r'#include "([^"]+)"', src.read())
        assert seen <= set(files), (kind, sorted(seen - set(files)))
        assert len(bench.src_sha(kind)) == 16
    assert bench.src_sha("small") != bench.src_sha("large")


def test_one_process_throughput_is_tokens_over_time():
    ms, tps = bench.job_throughput(1, 8, 10, 1.5)
    assert ms == 1.5 and tps == pytest.approx(8 * 10 / 1.5e-3)


def test_run_layer_cli_parses_without_a_gpu():
    import subprocess
    import sys
    out = subprocess.run([sys.executable, "-m", "mixture_experts_layer_warp_gb300.run_layer", "--help"],
                         capture_output=True, text=True, cwd=bench.ROOT, timeout=120)
    assert out.returncode == 0 and "--tokens" in out.stdout and "mxfp8" in out.stdout
