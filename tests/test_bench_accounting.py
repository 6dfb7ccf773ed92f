"""The benchmark's accounting: the algorithmic FLOPs and bytes every reported
rate divides by, checked by brute force on small cases against the method's
definitions ("MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 1.1:
a Full-attention query sees every earlier token, an SWA query the last W),
and the window filter of the clock record that goes beside each rate."""
import datetime
import os
import time

import numpy as np
import pytest

import bench
import hswa_workloads as wl


def work(window, page=64, hq=4, hkv=2, d=16, dtype=wl.DTYPE_BF16):
    return wl.Workload("accounting", 0, hq, hkv, d, page, window, dtype, (0,), 1, (wl.KIND_FULL, wl.KIND_SWA))


CASES = [  # (window, prefix per sequence, chunk per sequence)
    (128, [0, 100, 300, 64], [130, 64, 257, 1]),
    (40, [5, 1000, 127], [300, 0, 129]),
    (1, [0, 63], [1, 200]),
    (128, [8192 + 17, 12000], [4096, 700]),
]


def brute_pairs(prefix, chunk, window):
    """Valid (query, key) pairs of the chunk rows: keys [0, t] and, for the
    window, [max(0, t - W + 1), t]."""
    full = swa = 0
    for p, c in zip(prefix, chunk):
        t = p + np.arange(c)
        full += int(np.sum(t + 1))
        swa += int(np.sum(np.minimum(t + 1, window)))
    return full, swa


@pytest.mark.parametrize("window,prefix,chunk", CASES)
def test_prefill_valid_pairs(window, prefix, chunk):
    w = work(window)
    f = bench.prefill_flops(w, prefix, chunk)
    k = 4 * w.head_dim * w.n_q_heads
    full, swa = brute_pairs(prefix, chunk, window)
    assert f["full"] == k * full and f["swa"] == k * swa
    assert f["step"] == f["full"] + f["swa"]


@pytest.mark.parametrize("window,prefix,chunk", CASES)
def test_prefill_executed_pairs(window, prefix, chunk):
    """Executed pairs: a Full block of 128 chunk rows runs every 128-key tile
    up to its last row; an SWA block (on 128-position boundaries) runs every
    64-key page some row of it sees, for all 128 tile rows."""
    w = work(window)
    f = bench.prefill_flops(w, prefix, chunk)
    k = 4 * w.head_dim * w.n_q_heads
    full = swa = 0
    for p, c in zip(prefix, chunk):
        for start in range(0, c, 128):  # Full blocks: chunk rows [start, start + 128)
            last = p + min(c, start + 128) - 1
            full += len(set(j // 128 for j in range(last + 1))) * 128 * 128
        rows = p + np.arange(c)
        for m in sorted(set(rows // 128)):  # SWA blocks: positions [128 m, 128 m + 128)
            ts = rows[rows // 128 == m]
            pages = set()
            for t in ts:
                pages.update(range(max(0, t - window + 1) // 64, t // 64 + 1))
            assert pages == set(range(min(pages), max(pages) + 1))  # contiguous
            swa += len(pages) * 64 * 128
    assert f["full_exec"] == k * full and f["swa_exec"] == k * swa


@pytest.mark.parametrize("window,prefix,chunk", CASES)
def test_swa_prefill_bytes(window, prefix, chunk):
    """q read and o written once, and every K / V page some chunk row's window
    touches read once."""
    w = work(window)
    es = 2
    pages = 0
    for p, c in zip(prefix, chunk):
        touched = set()
        for t in range(p, p + c):
            touched.update(range(max(0, t - window + 1) // 64, t // 64 + 1))
        pages += len(touched)
    expect = 2 * sum(chunk) * w.n_q_heads * w.head_dim * es + pages * w.n_kv_heads * 2 * 64 * w.head_dim * es
    assert bench.swa_prefill_bytes(w, prefix, chunk) == expect


def test_decode_bytes():
    """One decode step: every valid K / V row once (all of a Full sequence,
    the last W of an SWA one), q and o, and the new token's K / V read and
    written, per layer; FP8 rows carry one byte an element plus a scale."""
    w = work(128, hq=8, hkv=2, d=32)
    lens = [1, 64, 129, 5000]
    row = w.n_kv_heads * w.head_dim * 2
    b = bench.decode_bytes(w, lens)
    qo = 2 * len(lens) * w.n_q_heads * w.head_dim * 2
    new = 2 * 2 * len(lens) * row
    assert b["full_layer"] == 2 * row * sum(lens) + qo + new
    assert b["swa_layer"] == 2 * row * sum(min(L, 128) for L in lens) + qo + new
    assert b["step"] == b["full_layer"] + b["swa_layer"]
    b8 = bench.decode_bytes_fp8(w, lens)
    row8 = w.n_kv_heads * (w.head_dim + 4)
    assert b8["full_kv"] == 2 * row8 * sum(lens)
    assert b8["full_layer"] == b8["full_kv"] + qo + 2 * len(lens) * row + 2 * len(lens) * row8


def test_hybrid70_bytes():
    """70 layers, Full at every 7th: ten Full layers read every row, sixty SWA
    layers the last W, each layer q, o and the new token's K / V."""
    w = wl.hybrid70(n_seqs=3, context=300)
    lens = [300, 301, 17]
    b = bench.hybrid70_bytes(w, lens)
    assert (b["n_full"], b["n_swa"]) == (10, 60)
    row = w.n_kv_heads * w.head_dim * 2
    per_layer = 2 * 3 * w.n_q_heads * w.head_dim * 2 + 2 * 2 * 3 * row
    assert b["step"] == 10 * 2 * row * sum(lens) + 60 * 2 * row * sum(min(L, w.window) for L in lens) \
        + 70 * per_layer


def test_clock_record_keeps_only_the_marked_window(tmp_path, monkeypatch):
    """Samples outside [first mark, last mark] are left out of the summary,
    and a throttle reason inside the window is reported."""
    monkeypatch.setenv("HSWA_CLOCKS_DIR", str(tmp_path))
    c = bench.ClockSampler(0, "_test")
    now = time.time()

    def ts(t):
        return datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]

    with open(c.path, "w") as f:
        for dt, mhz, cap in ((-5, 900, "Not Active"), (0.5, 2070, "Not Active"), (1.0, 1980, "Active"),
                             (1.5, 2070, "Not Active"), (5, 700, "Active")):
            f.write("%s, 0, %d, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, %s\n" % (ts(now + dt), mhz, cap))

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    c.proc, c.fh = Done(), open(os.devnull, "w")
    c.marks = [now, now + 2]
    info = c.stop()
    assert info["samples"] == 3 and info["sm_mhz"] == 2070.0 and info["reasons"] == ["sw_power_cap"]


def _reference_line(env):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=root, env={**os.environ, **env}, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_line_keeps_the_contract():
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the keys, types and units of the library's own line, and an e2e
    object of its own value with no host-device bytes."""
    lines = _reference_line({"RANK": "0", "WORLD_SIZE": "1"})
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["config"]["workload"] == "decode_batch"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    assert _reference_line({"RANK": "1", "WORLD_SIZE": "2"}) == []
