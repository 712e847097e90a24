"""The JSON line bench.py prints (GPU): every key of the measurement contract,
with consistent values, on a short run of the default workload."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_forward_bench_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "5", "--warmup", "3", "--no-cpu-baseline"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches",
                "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and "workload" in d["config"]
    roof = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    e2e = d["e2e"]
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in e2e, key
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 2 * d["steps"]   # prologue + attention kernel per step
    assert {"sm_mhz", "sm_max_mhz", "reasons", "samples", "samples_under_load", "samples_timed"} <= set(d["clocks"])
    # a 5-step timed region is far shorter than the 50 ms poll: the clock
    # record still has samples (the synchronous queries at both ends of the
    # timed region and the untimed repeats of the same step) and a clock
    assert d["clocks"]["samples"] >= 2 and d["clocks"]["samples_timed"] >= 2
    assert d["clocks"]["samples_under_load"] >= 1 and d["clocks"]["sm_mhz"] is not None
    assert abs(d["pct_bf16_spec_peak"] - 100.0 * d["value"] / 2250.0) < 1e-6


@pytest.mark.parametrize("leg", ["--backward", "--decode"])
def test_backward_and_decode_lines_have_a_clock_record(leg):
    # the backward and decode legs also hold the same step under load after
    # their (here very short) timed region, so that their clock record has
    # samples taken under load
    r = subprocess.run([sys.executable, "bench.py", leg, "--steps", "5", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["value"] > 0 and d["ms_per_step"] > 0
    c = d["clocks"]
    assert c["samples"] >= 2 and c["samples_timed"] >= 2
    assert c["samples_under_load"] >= 1 and c["sm_mhz"] is not None
