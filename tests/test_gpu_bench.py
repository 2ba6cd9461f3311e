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
    assert rf["traffic"] is None or rf["traffic"] > 0
    e2e = d["e2e"]
    assert e2e["unit"] == "TFLOPS" and 0 < e2e["value"] < d["value"]
    assert e2e["h2d_bytes_per_step"] == 3 * 4 * 16 * 4096 * 128 * 2
    assert e2e["d2h_bytes_per_step"] == 4 * 16 * 4096 * 128 * 2 + 4 * 16 * 4096 * 4
    assert d["gpu_launches"] == 20
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOPS" and cb["cores"] >= 1 and cb["value"] > 0
