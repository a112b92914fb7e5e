"""bench.py's JSON line on a GPU: one line with every field the measurement
contract names (the throughput and its step time, the dominant kernel's
roofline, the CPU oracle's timed sample, the end-to-end figure with its host
copies, the launch count and the clocks seen during the timed steps)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_json_line_contract():
    cmd = [sys.executable, "bench.py", "--config", "v2lite", "--steps", "3", "--warmup", "3", "--cpu-sample", "64"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])

    assert isinstance(d["metric"], str) and d["unit"] == "tokens/s"
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    T = 8192                                   # the V2-Lite workload's tokens, L = 4 blocks
    assert abs(d["value"] - T / (d["ms_per_step"] / 1e3)) <= 1e-3 * d["value"]
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert "vs_baseline" in d and d["dtype"] == "bf16" and d["data"].startswith("synthetic")
    assert d["config"]["workload"].startswith("v2lite")

    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor") and rf["unit"] in ("GB/s", "TFLOP/s")
    assert rf["achieved"] > 0 and rf["peak"] > 0 and "traffic" in rf
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3

    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]

    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "tokens/s"
    assert e2e["h2d_bytes_per_step"] == T * 2048 * 2       # x, bf16 [T, d]
    assert e2e["d2h_bytes_per_step"] == T * 2048 * 2       # o_L, bf16 [T, d]

    assert d["gpu_launches"] > 0
    ck = d["clocks"]
    assert ck["sm_max_mhz"] > 0 and isinstance(ck["reasons"], list)
