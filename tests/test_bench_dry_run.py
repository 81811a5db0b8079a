"""bench.py's contract without a GPU: every leg of the benchmark runs through the real binding
(its argument checks on every call) with the kernels stubbed, and the JSON line carries the
keys the benchmark contract names."""
import json
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))

pytestmark = pytest.mark.slow


def test_bench_line_without_a_gpu():
    r = subprocess.run([sys.executable, os.path.join(HERE, "bench_dry_run.py"), "--steps", "2", "--warmup", "1",
                        "--no-cpu-baseline", "--no-per-workload"], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] >= 3   # at least three warm-up steps
    assert set(line["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert set(line["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["gpu_launches"] > 0
    assert "workload" in line["config"]
    assert line["roofline_attention"]["key_tile"] == 64          # d_head 256 runs 64-key tiles
    assert {"decode_step"} <= set(line["searched_slots"])
