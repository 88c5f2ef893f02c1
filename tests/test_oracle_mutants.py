"""Plants one plausible mistake at a time in a copy of the oracle source and
checks that at least one pin fails for each. This shows the pins would catch a
dropped term, a wrong sign or index, or a transposed operand in the oracle."""
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

# (name, text in moe_oracle.c, replacement)
MUTANTS = [
    ("silu_on_up_not_gate", "a[i] = silu(g) * u;", "a[i] = silu(u) * g;"),
    ("no_renormalisation", "w[t * k + j] = p[ids[t * k + j]] / sel;", "w[t * k + j] = p[ids[t * k + j]];"),
    ("ties_to_higher_index", "(best < 0 || l[e] > l[best])", "(best < 0 || l[e] >= l[best])"),
    ("decide_in_fp64", "l[e] = (double)(float)logits[t * E + e];", "l[e] = logits[t * E + e];"),
    ("w2_transposed", "s += elem(w2, dtype, h * I + i) * a[i];", "s += elem(w2, dtype, i * H + h) * a[i];"),
    ("gate_up_interleaved", "u += elem(w13, dtype, (I + i) * H + h) * xv[h];",
     "u += elem(w13, dtype, (2 * i + 1) * H + h) * xv[h];"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("bias_dropped", "            s += (double)bias[e];", "            s += 0.0;"),
    ("unstable_route_sort", "for (int64_t r = 0; r < R; ++r)\n        perm[fill[ids[r]]++] = (int32_t)r;",
     "for (int64_t r = R - 1; r >= 0; --r)\n        perm[fill[ids[r]]++] = (int32_t)r;"),
    ("inverse_not_inverted", "inv[perm[i]] = (int32_t)i;", "inv[i] = perm[i];"),
    ("one_micro_only", "for (int64_t m = 0; m < n_micro; ++m)\n                swiglu_expert_acc(xq,",
     "for (int64_t m = 0; m < 1; ++m)\n                swiglu_expert_acc(xq,"),
    ("gather_wrong_token", "int64_t t = perm[i] / k;", "int64_t t = perm[i] % (k + 1);"),
    ("shared_scaled", "swiglu_expert_acc(xv, H, Is, sw13, sw2, s_dtype, 1.0, acc, a, 0);",
     "swiglu_expert_acc(xv, H, Is, sw13, sw2, s_dtype, 0.5, acc, a, 0);"),
    ("perm_holds_token", "perm[fill[ids[r]]++] = (int32_t)r;", "perm[fill[ids[r]]++] = (int32_t)(r / k);"),
    ("mx_scale_from_ceil", "                shared = (ex - 1) - 8;", "                shared = ex - 8;"),
    ("mx_act_scale_from_ceil", "            shared = (ex - 1) - 8;\n            if (shared < -127)\n                shared = -127;\n            if (shared > 127)\n                shared = 127;\n        }\n        for (int i = 0; i < 32; ++i) {",
     "            shared = ex - 8;\n            if (shared < -127)\n                shared = -127;\n            if (shared > 127)\n                shared = 127;\n        }\n        for (int i = 0; i < 32; ++i) {"),
    ("mx_ties_away_from_zero", "double q = nearbyint(scaled);", "double q = round(scaled);"),
    ("mx_scale_layout_row_major", "scales[(g * nb + b) * rows + r] = (uint8_t)(shared + 127);",
     "scales[(g * rows + r) * nb + b] = (uint8_t)(shared + 127);"),
    ("mx_scale_bias_off_by_one", "ldexp(e4m3_value(codes[gr * cols + c]), S - 127);",
     "ldexp(e4m3_value(codes[gr * cols + c]), S - 126);"),
    ("mx_dequant_scale_of_wrong_block", "int S = scales[(g * nb + c / 32) * rows + r];",
     "int S = scales[(g * nb + c / 64) * rows + r];"),
    ("fp64_weights_read_as_shared_dtype", "w_dtype, w[t * k + j], acc, a, mx_act);",
     "dtype, w[t * k + j], acc, a, mx_act);"),
    ("mx_act_h_not_rounded", "            a[i] = bf16_round(a[i]);\n        mx_round_vec(a, I);",
     "            a[i] = bf16_round(a[i]);\n        (void)0;"),
    ("mx_act_h_not_bf16", "            a[i] = bf16_round(a[i]);", "            a[i] = a[i];"),
    ("bf16_ties_away", "double q = ldexp(nearbyint(ldexp(u, 7 - e)), e - 7);",
     "double q = ldexp(round(ldexp(u, 7 - e)), e - 7);"),
    ("bf16_six_fraction_bits", "ldexp(nearbyint(ldexp(u, 7 - e)), e - 7)", "ldexp(nearbyint(ldexp(u, 6 - e)), e - 6)"),
    ("mx_act_x_not_rounded", "        if (mx_act)\n            mx_round_vec(xq, H);",
     "        if (0)\n            mx_round_vec(xq, H);"),
    ("mx_act_block_of_16", "    for (int64_t b = 0; b < n; b += 32) {\n        double amax = 0.0;\n        for (int i = 0; i < 32; ++i)",
     "    for (int64_t b = 0; b < n; b += 16) {\n        double amax = 0.0;\n        for (int i = 0; i < 16; ++i)"),
]


_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
lib = oracle.load_variant({src!r}, {so!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(lib)
    except Exception as exc:
        failed.append(pin.__name__)
print("FAILED_PINS", ",".join(failed))
"""


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = os.path.join(workdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests), tests=tests, src=path,
                          so=os.path.join(workdir, f"lib{name}.so"))
    # each variant runs in its own process: a planted mistake that crashes the
    # oracle (an out-of-range index) is caught as well
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300)
    if proc.returncode != 0:
        return
    line = [ln for ln in proc.stdout.splitlines() if ln.startswith("FAILED_PINS")][-1]
    failed = [p for p in line.split(" ", 1)[1].split(",") if p]
    assert failed, f"no pin caught the planted mistake {name}"


def test_unmodified_copy_passes_every_pin(workdir):
    """Control for the runner above: the oracle source as it stands fails no pin."""
    path = os.path.join(workdir, "unmodified.c")
    shutil.copy(SRC, path)
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests), tests=tests, src=path,
                          so=os.path.join(workdir, "libunmodified.so"))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300)
    assert proc.returncode == 0, proc.stderr
    line = [ln for ln in proc.stdout.splitlines() if ln.startswith("FAILED_PINS")][-1]
    assert line.split(" ", 1)[1] == "", line
