"""The bench's JSON line on the small profiling workload (profile-16k,
L = 16384), end to end: every key the line promises is there and consistent
(device throughput, the roofline of the dominant kernel, the fp64 oracle's
rate on the host, the end-to-end rate through the public calls with host
buffers, clocks, launch count)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keys_on_profile_16k():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "bench.py", "--workload", "profile-16k", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
              "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "profile-16k"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    rl = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rl, k
    assert rl["bound"] == "tensor" and 0 < rl["frac"] < 1.5
    assert abs(rl["frac"] - rl["achieved"] / rl["peak"]) < 1e-3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # the loop's own computation per step cannot take longer than the whole pipelined step
    assert 0 < e["compute_ms_per_step"] <= e["ms_per_step"] * 1.05
    assert "clocks" in e
    # forward (1) + preprocess (2) + dK/dV (1) + dQ (1) per step, at least
    assert d["gpu_launches"] >= 5 * d["steps"]
