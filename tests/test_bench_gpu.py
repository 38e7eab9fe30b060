"""The bench line's contract on a GPU: a short run of bench.py prints one JSON
line with every key the harness reads, with sane values."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    out = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3",
                          "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["gpu_launches"] == 3 and line["config"]["workload"]
    rf = line["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert rf["achieved"] > 0 and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-3)
    l2 = line["l2_modes"]
    assert "error" not in l2, l2
    for mode in ("warm", "cold"):
        t = l2[mode]
        assert 0 < t["min_ms"] <= t["median_ms"] and t["min_ms"] <= t["mean_ms"]
    assert rf["traffic"] is None or rf["traffic"] > 0
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "TFLOP/s"
    assert e2e["h2d_bytes_per_step"] == 2 * 8192 * 8192 * 2
    assert e2e["d2h_bytes_per_step"] == 8192 * 8192 * 2
    # the copies alone bound the end-to-end rate (timing noise aside)
    assert e2e["copies_only_value"] > 0 and e2e["copies_only_gbs"] > 0
    assert e2e["value"] <= 1.05 * e2e["copies_only_value"]
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]


def test_ncu_case_runs():
    """The profiler-capture mode launches the shape it is given and exits 0."""
    out = subprocess.run([sys.executable, "bench.py", "--ncu-case", "bf16:128x1024x512"], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line == {"ncu_case": "bf16:128x1024x512", "launches_each": 3, "cublas": True}
