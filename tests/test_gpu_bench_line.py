"""The GPU arm of bench.py prints one JSON line with the keys its consumers read."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    cmd = [sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--no-e2e", "--no-cpu-baseline",
           "--no-next-rows", "--no-configs", "--no-ceilings"]
    out = subprocess.run(cmd, cwd=REPO, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is False and d["unit"] == "us"
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1000 - d["value"]) < 1e-6 * d["value"] + 1e-9
    assert d["gpu_launches"] == 3 * d["steps"]  # Markov draft, probe batch, grouped WS matvec
    assert isinstance(d["config"], dict) and "workload" in d["config"] and d["config"]["num_reqs"] == 8
    r = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    parts = d["parts"]
    assert parts["markov_draft_us"] > 0 and parts["conf_probe_batch_us"] > 0 and parts["ws_matvec_4_shapes_grouped_us"] > 0
