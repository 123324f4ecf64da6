"""bench.py's JSON line on a GPU: one line, last on stdout, with the keys the
benchmark contract names, on a small parameter set (GPT-2 124M, a short run)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_has_the_contract_keys():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "gpt2_124m", "--steps", "10",
                          "--warmup", "3", "--cpu-seconds", "2"], capture_output=True, text=True, cwd=ROOT,
                         timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    line = json.loads(lines[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    r = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["kernel_ms_samples"] >= 16
    # frac recomputes from the line: 28 B x params / mean step-kernel time / peak
    achieved = 28 * line["config"]["params"] / (r["kernel_ms_per_step"] / 1e3) / 1e9
    assert abs(achieved - r["achieved"]) <= 1e-3 * achieved and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert 0.5 < r["frac"] < 1.2
    e = line["e2e"]
    assert e["h2d_bytes_per_step"] == 2 * line["config"]["params"] and e["d2h_bytes_per_step"] > 0 and e["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["gpu_launches"] == line["steps"] * (2 + r["launches_per_step"])
    assert line["variants"]["sr_stress"]["drift"]["steps"] == 1000
