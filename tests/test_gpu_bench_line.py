"""The bench's JSON line on a GB300: a short decode-batch run (the default
workload) prints one line with every key the bench contract names, and the
figures inside it agree with one another."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_decode_line_keeps_the_contract():
    cmd = [sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--cpu-budget", "2", "--no-prefill",
           "--no-hybrid70", "--no-transfer", "--no-tree", "--no-fp8", "--no-multi"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["n_gpus"] == 1
    assert d["steps"] == 3 and d["warmup"] == 3 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == "bf16" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "decode_batch" and "l2" in d["config"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["achieved"] > 0 and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert rf["traffic"] is None or rf["traffic"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "GB/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    ck = d["clocks"]
    assert "sm_mhz" in ck and "sm_max_mhz" in ck and isinstance(ck["reasons"], list)
