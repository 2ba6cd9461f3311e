"""bench.py on one GPU: a short run prints one JSON line with every field of its contract, and
the numbers in it agree with each other."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "20", "--warmup", "3",
           "--no-sweep", "--e2e-steps", "3", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] >= 3
    assert d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["dtype"] == "bf16" and d["data"] == "synthetic" and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("s4k")
    assert d["device_status"] == 0
    # 0.55 TFLOP per step: value and ms_per_step describe the same time
    flops = 4 * 4 * 16 * 4096 * 4096 * 128
    assert abs(flops / (d["ms_per_step"] * 1e-3) / 1e12 - d["value"]) / d["value"] < 0.01
    assert d["value"] > 100.0
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert abs(rf["achieved"] - d["value"]) < 1e-6
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert abs(rf["frac_nominal"] - rf["achieved"] / rf["peak_nominal"]) < 1e-3
    if d["clocks"]["sm_mhz"]:
        assert abs(rf["peak_clock"] - 152 * 8192 * d["clocks"]["sm_mhz"] * 1e-6) < 1.0
        assert abs(rf["frac_clock"] - rf["achieved"] / rf["peak_clock"]) < 1e-3
    assert rf["traffic"] is None or rf["traffic"] > 0
    st = d["step_ms"]
    assert st["min"] <= st["median"] <= st["max"] and st["min"] <= st["mean"] <= st["max"]
    assert abs(st["mean"] - d["ms_per_step"]) < 1e-3
    assert d["value_best"] >= d["value_median"] > 0
    assert abs(d["value_median"] - flops / (st["median"] * 1e-3) / 1e12) / d["value_median"] < 0.01
    e2e = d["e2e"]
    assert e2e["unit"] == "TFLOPS" and 0 < e2e["value"] < d["value"]
    assert e2e["device_status"] == 0 and e2e["outputs_equal_device_call"] is True
    assert e2e["h2d_bytes_per_step"] == 3 * 4 * 16 * 4096 * 128 * 2
    assert e2e["d2h_bytes_per_step"] == 4 * 16 * 4096 * 128 * 2 + 4 * 16 * 4096 * 4
    assert d["gpu_launches"] == 20
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOPS" and cb["cores"] >= 1 and cb["value"] > 0


def test_bench_main_roofline_is_the_main_workload_after_a_sweep():
    # The sweep must not leak into the main line's roofline or median (a causal sweep entry
    # last, as in the default sweep).
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3",
           "--workload", "tiny", "--sweep", "tiny", "--causal-sweep", "tiny", "--sweep-steps", "5",
           "--e2e-steps", "3", "--no-cpu-baseline"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][-1])
    assert abs(d["roofline"]["achieved"] - d["value"]) < 1e-6
    flops = 4 * 1 * 1 * 256 * 256 * 128
    assert abs(d["value_median"] - flops / (d["step_ms"]["median"] * 1e-3) / 1e12) / d["value_median"] < 0.01


def test_bench_sweep_entries_carry_a_roofline():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3",
           "--sweep", "tiny", "--causal-sweep", "tiny", "--sweep-steps", "5", "--e2e-steps", "3",
           "--no-cpu-baseline"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][-1])
    assert set(d["sweep"]) == {"tiny", "tiny_causal"}
    for key, e in d["sweep"].items():
        rf = e["roofline"]
        assert rf["bound"] == "tensor" and abs(rf["achieved"] - e["tflops"]) < 0.1, key
        assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3, key
        assert e["step_ms"]["min"] <= e["step_ms"]["median"], key


def test_reference_arm_config_matches():
    """Both arms describe the workload with the same config keys and values."""
    ref_cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
               "--warmup", "3", "--ref-step-seconds", "0.2", "--workload", "tiny"]
    r = subprocess.run(ref_cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    ref_line = json.loads(r.stdout.strip().splitlines()[-1])
    ours = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
            "--workload", "tiny", "--no-sweep", "--e2e-steps", "3", "--no-cpu-baseline"]
    r = subprocess.run(ours, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    our_line = json.loads(r.stdout.strip().splitlines()[-1])
    assert ref_line["config"] == our_line["config"]
    assert ref_line["metric"] == our_line["metric"] and ref_line["unit"] == our_line["unit"]
