"""bench.py's own arm on the GPU, on a one-layer cut of the 28-layer workload:
one JSON line with every key of the contract (roofline of the dominant kernel,
CPU oracle baseline, end to end through host buffers, clocks, launch count)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_keeps_the_contract():
    r = subprocess.run(
        [sys.executable, "bench.py", "--layers", "1", "--steps", "2", "--warmup", "3",
         "--e2e-steps", "1", "--cpu-seconds", "1"],
        cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert "workload" in line["config"]
    roof = line["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["unit"] in ("GB/s", "TFLOP/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-6
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["value"] != line["value"]  # measured through host buffers, not a copy
    clocks = line["clocks"]
    assert "sm_mhz" in clocks and "sm_max_mhz" in clocks and "reasons" in clocks
    # two attention passes, the fused mass/segment/select kernel and the gather
    # per event (units of 1536 slots), two timed events
    assert line["gpu_launches"] == 4 * 2
    assert sum(k["launches"] for k in line["kernels"]) == line["gpu_launches"]
