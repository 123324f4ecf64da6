"""Host-side pieces of bench.py (no GPU): the DRAM-traffic lookup that fills
roofline.traffic, and the JSON line's contract on the reference arm."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_lookup_uses_only_captures_of_the_current_kernel_source(tmp_path, monkeypatch):
    cur = bench.kernel_source_hash()
    prof = {"captures": [
        {"kernel_source_sha256_16": "0" * 16, "launch_elems": 100, "dram_bytes_read": 1, "dram_bytes_write": 1},
        {"kernel_source_sha256_16": cur, "launch_elems": 1000, "dram_bytes_read": 14000, "dram_bytes_write": 13000},
        {"kernel_source_sha256_16": cur, "launch_elems": 10_000, "dram_bytes_read": 140_000,
         "dram_bytes_write": 139_000},
    ]}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(prof))
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(p))
    # the capture closest in size, scaled by elements
    assert bench.profiled_traffic_bytes(2000) == (54_000, 1000)
    assert bench.profiled_traffic_bytes(20_000) == (558_000, 10_000)
    # no capture of the current source: no traffic figure
    prof["captures"] = prof["captures"][:1]
    p.write_text(json.dumps(prof))
    assert bench.profiled_traffic_bytes(2000) == (None, None)


def test_committed_traffic_summary_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "adamw_step_traffic.json")) as f:
        prof = json.load(f)
    for c in prof["captures"]:
        assert len(c["kernel_source_sha256_16"]) == 16 and c["launch_elems"] > 0
        # reads never fall below the algorithmic 14 B per parameter
        assert c["dram_bytes_read"] >= 14 * c["launch_elems"]
        assert "ncu" in c["command"] and "--clock-control none" in c["command"]


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "3", "--cpu-seconds", "3"], capture_output=True, text=True, cwd=ROOT,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    line = json.loads(lines[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert "Llama-3-8B" in line["config"]["workload"]
