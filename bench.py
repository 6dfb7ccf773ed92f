"""Benchmark of the Hybrid-SWA dual-pool hot path on one GB300 (or N replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hswa|reference]
                [--workload decode_batch|chunked_prefill]

decode_batch (default): 64 sequences, cached lengths uniform in [1024, 32768],
64 Q / 8 KV heads, d 128, page 64, bf16, one Full and one SWA (W = 128) layer.
One step = reserve one token per sequence (both pools) -> sync the device
tables -> append + decode the Full layer -> append + decode the SWA layer
(hswa_decode_append: the append is fused into the decode); the SWA release
runs every 64 steps.
Metric: algorithmic HBM bytes of the step (valid KV rows read, q read, o
written, new K/V read and written) per second.

chunked_prefill: 8 sequences, cached prefix uniform in [8192, 65536], a
4096-token chunk each; one step = reserve the chunk -> sync -> append ->
prefill the Full layer -> prefill the SWA layer -> release. Metric: TFLOP/s
over the valid (query, key) pairs, 4 * d * Hq per pair.

With --impl reference the CPU oracle runs the same workload on a bounded
sample of sequences per step and reports the same metric.
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import hswa_workloads as wl  # noqa: E402

KV_ROW = {wl.DTYPE_BF16: 2, wl.DTYPE_F32: 4}


# DRAM traffic of the decode kernel per launch over its algorithmic bytes, from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) at full size,
# valid only for the kernel sources it was taken on.
DECODE_TRAFFIC = {"ratio": 1.0030, "sources": ("decode.cu", "common.cuh"),
                  "sha256": "b59ebe1612be30dc6f35023ce6596d1698fb1a1e736a576d2d1b7662166a9d03"}


def source_digest(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "hybrid_sliding_window_dual_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic(alg_bytes):
    """Captured traffic scaled to this launch, or None if the kernel changed."""
    if DECODE_TRAFFIC["sha256"] != source_digest(DECODE_TRAFFIC["sources"]):
        return None
    return int(DECODE_TRAFFIC["ratio"] * alg_bytes)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 100 ms in the background; with mark() the
    summary keeps only the samples taken between the first and the last
    mark (host clock)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, tag=""):
        self.gpu = gpu_index
        self.proc = None
        # raw samples (the JSON line carries their summary); HSWA_CLOCKS_DIR picks the folder
        out = os.environ.get("HSWA_CLOCKS_DIR") or os.path.join(ROOT, "bench_out")
        self.path = os.path.join(out, "clocks%s_rank%d.csv" % (tag, gpu_index))
        self.marks = []

    def mark(self):
        self.marks.append(time.time())

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = (min(self.marks), max(self.marks)) if len(self.marks) >= 2 else (None, None)
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                if lo is not None:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    if not lo <= ts <= hi:
                        continue
                sm.append(float(parts[2]))
                mx = float(parts[3])
            except ValueError:
                continue
            for name, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ dist helpers
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(x, world, op):
    """All-reduce one float over the ranks (host timing data, not the data
    path): on the GPU under nccl, on the CPU under gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x, world):
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.MAX if world > 1 else None)


def sum_over_ranks(x, world):
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.SUM if world > 1 else None)


# ------------------------------------------------------------- workloads
def decode_bytes(w, lens_after):
    """Algorithmic bytes of one decode step over the Full and the SWA layer."""
    es = KV_ROW[w.dtype]
    row = w.n_kv_heads * w.head_dim * es          # one K (or V) row of all kv heads
    B = len(lens_after)
    full_kv = 2 * row * int(np.sum(lens_after))
    swa_kv = 2 * row * int(np.sum(np.minimum(lens_after, w.window)))
    qo = 2 * B * w.n_q_heads * w.head_dim * es   # q read + o written, per layer
    new = 2 * 2 * B * row                          # new K/V read + written, per layer
    return {"full_kv": full_kv, "swa_kv": swa_kv, "full_layer": full_kv + qo + new,
            "swa_layer": swa_kv + qo + new, "step": full_kv + swa_kv + 2 * (qo + new)}


def decode_bytes_fp8(w, lens_after):
    """Algorithmic bytes of one decode step over FP8 pools: per key and kv
    head one E4M3 byte per element of K and of V plus their two fp32 scales."""
    row = w.n_kv_heads * (w.head_dim + 4)  # one K (or V) row of all kv heads, with its scale
    B = len(lens_after)
    es = KV_ROW[w.dtype]
    full_kv = 2 * row * int(np.sum(lens_after))
    swa_kv = 2 * row * int(np.sum(np.minimum(lens_after, w.window)))
    qo = 2 * B * w.n_q_heads * w.head_dim * es
    new = 2 * B * w.n_kv_heads * w.head_dim * es + 2 * B * row  # bf16 new K/V read, FP8 rows written
    return {"full_kv": full_kv, "swa_kv": swa_kv, "full_layer": full_kv + qo + new,
            "swa_layer": swa_kv + qo + new, "step": full_kv + swa_kv + 2 * (qo + new)}


def measure_decode_fp8(steps, warmup):
    """The decode-batch step over FP8 pools: GB/s of FP8 bytes and tokens/s."""
    import torch
    w = wl.decode_batch()
    bench = DecodeBatch(w, warmup + steps + 8, fp8=True)
    for _ in range(warmup):
        bench.step()
    bench.stream.synchronize()
    before = decode_bytes_fp8(w, bench.lens() + 1)
    secs = time_steps(lambda: bench.step(time_full_decode=True), steps, bench.stream, 1)
    after = decode_bytes_fp8(w, bench.lens())
    dec_ms = float(np.mean([a.elapsed_time(b) for a, b in bench.decode_events]))
    bench.finish()
    step_bytes = 0.5 * (before["step"] + after["step"])
    full_bytes = 0.5 * (before["full_layer"] + after["full_layer"])
    out = {"gbs": step_bytes * steps / secs / 1e9, "ms_per_step": secs / steps * 1e3,
           "tokens_per_s": len(w.cached) * steps / secs, "full_layer_gbs": full_bytes / (dec_ms / 1e3) / 1e9,
           "full_layer_ms": dec_ms}
    del bench
    torch.cuda.empty_cache()
    return out


def measure_decode_multi(reps, w, token_counts=(1, 2, 3, 4, 8, 16), fp8=False):
    """Multi-token decode (n_tok query tokens per sequence at positions
    L - n_tok .. L - 1) over the decode-batch pools (FP8 E4M3 pools when fp8):
    one step is the Full and the SWA layer of hswa_decode_multi, events
    around each layer. Returns per n_tok the step time, query tokens/s and
    the Full layer's GB/s (KV bytes read once, q and o of every token)."""
    import torch
    from hybrid_sliding_window_dual_gb300 import hswa_last_kernel
    bench = DecodeBatch(w, 8, hold=max(token_counts), fp8=fp8)
    sess, B, es = bench.sess, bench.B, KV_ROW[w.dtype]
    lens = bench.lens()
    kv = decode_bytes_fp8(w, lens) if fp8 else decode_bytes(w, lens)
    out = {}
    for T in token_counts:
        q = [wl.normal((B * T, w.n_q_heads, w.head_dim), 700 + 10 * T + i, w.dtype, "cuda") for i in range(2)]
        o = [torch.empty_like(x) for x in q]
        sess.workspace(B, T)
        ev = []
        with torch.cuda.stream(bench.stream):
            for r in range(reps + 3):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record(bench.stream)
                sess.decode_multi(0, q[0], o[0], B, T, bench.scale)
                e[1].record(bench.stream)
                sess.decode_multi(1, q[1], o[1], B, T, bench.scale)
                e[2].record(bench.stream)
                if r >= 3:
                    ev.append(e)
        bench.stream.synchronize()
        assert sess.check() == 0
        kernel = hswa_last_kernel()
        full_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in ev]))
        step_ms = float(np.mean([a.elapsed_time(c) for a, _, c in ev]))
        full_bytes = kv["full_kv"] + 2 * B * T * w.n_q_heads * w.head_dim * es
        out[T] = {"step_ms": step_ms, "full_layer_ms": full_ms, "tokens_per_s": B * T / (step_ms / 1e3),
                  "full_layer_gbs": full_bytes / (full_ms / 1e3) / 1e9, "kernel": kernel}
    bench.finish()
    del bench
    torch.cuda.empty_cache()
    return out


def prefill_flops(w, prefix, chunk):
    """Valid (query, key) pairs x 4 d Hq for a Full and an SWA layer, and the
    pairs the tensor-core kernels execute. Full-layer blocks are 128 chunk
    rows from the prefix and read 128-key tiles [0, last row]; SWA blocks
    (W <= 128) sit on 128-position boundaries and read the 64-key pages from
    their first row's window start to their last row."""
    full = sum(c * p + c * (c + 1) // 2 for p, c in zip(prefix, chunk))
    swa = sum(sum(min(p + r + 1, w.window) for r in range(c)) for p, c in zip(prefix, chunk))
    full_exec = swa_exec = 0
    for p, c in zip(prefix, chunk):
        for qb in range((c + 127) // 128):
            last = p + min(c, 128 * (qb + 1)) - 1
            full_exec += (last // 128 + 1) * 128 * 128
        if c > 0:
            for m in range(p // 128, (p + c - 1) // 128 + 1):
                p0, p_end = max(p, 128 * m), min(p + c, 128 * (m + 1))
                P = w.page_size
                swa_exec += ((p_end - 1) // P - max(0, p0 - w.window + 1) // P + 1) * P * 128
    k = 4 * w.head_dim * w.n_q_heads
    return {"full": k * full, "swa": k * swa, "step": k * (full + swa), "full_exec": k * full_exec,
            "swa_exec": k * swa_exec}


def swa_prefill_bytes(w, prefix, chunk):
    """Algorithmic bytes of an SWA layer's chunk: q read and o written
    (rows x Hq x d) and every K / V page the chunk's windows touch, once."""
    es, P = KV_ROW[w.dtype], w.page_size
    qo = 2 * sum(chunk) * w.n_q_heads * w.head_dim * es
    pages = sum((p + c - 1) // P - max(0, p - w.window + 1) // P + 1 for p, c in zip(prefix, chunk) if c > 0)
    return qo + pages * w.n_kv_heads * 2 * P * w.head_dim * es


class DecodeBatch:
    """The decode-batch workload on the GPU through the C ABI (bf16 pools, or
    FP8 E4M3 pools with per-token-head scales when fp8=True)."""

    def __init__(self, w, extra_steps, fp8=False, hold=0):
        import torch
        import hybrid_sliding_window_dual_gb300 as H
        from hybrid_sliding_window_dual_gb300.session import DualPoolSession
        self.H, self.torch, self.w = H, torch, w
        B, P, W = len(w.cached), w.page_size, w.window
        self.B = B
        full_pages = sum(math.ceil((L + extra_steps + 1) / P) for L in w.cached) + 16
        swa_pages = B * (math.ceil((W + 4096) / P) + 2) + 16
        max_pages = max(math.ceil((L + extra_steps + 1) / P) for L in w.cached) + 1
        self.fp8 = fp8
        cfg = H.Config(window=W, page_size=P, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, dtype=H.HSWA_DTYPE_FP8_E4M3 if fp8 else w.dtype,
                       full_pages=full_pages, swa_pages=swa_pages, max_seqs=B, max_pages_per_seq=max_pages)
        self.stream = torch.cuda.Stream()
        self.sess = DualPoolSession(cfg, [wl.KIND_FULL, wl.KIND_SWA], wl.permutation(full_pages, w.seed),
                                    wl.permutation(swa_pages, w.seed + 1), stream=self.stream, init="empty")
        # the last `hold` tokens are reserved after the last release (the
        # draft tokens of a multi-token step keep the window of the first)
        for s, L in enumerate(w.cached):
            for start in range(0, L - hold, 4096):
                self.sess.reserve([s], [min(4096, L - hold - start)])
                self.sess.release([s])
            if hold:
                self.sess.reserve([s], [hold])
        with torch.cuda.stream(self.stream):
            for i in range(2):
                for t, seed in ((self.sess.k[i], 10 + i), (self.sess.v[i], 20 + i)):
                    if fp8:  # seeded E4M3 codes without the NaN patterns
                        g = torch.Generator(device="cuda")
                        g.manual_seed(seed)
                        flat = t.view(-1)
                        for j in range(0, flat.numel(), 1 << 28):
                            n = min(1 << 28, flat.numel() - j)
                            mag = torch.randint(0, 0x7F, (n,), generator=g, device="cuda", dtype=torch.int32)
                            sgn = torch.randint(0, 2, (n,), generator=g, device="cuda", dtype=torch.int32)
                            flat[j:j + n] = (mag | (sgn << 7)).to(torch.uint8)
                    else:
                        fill_normal(t, seed)
                if fp8:
                    self.sess.ks[i].uniform_(0.001, 0.011)
                    self.sess.vs[i].uniform_(0.001, 0.011)
            self.sess.sync()
        dt = wl.TORCH_DTYPE[w.dtype]
        # a step's inputs (q, new K, new V of both layers) and outputs each
        # live in one contiguous block, so the host-buffer path moves them
        # with one copy per direction
        nq, nkv = B * w.n_q_heads * w.head_dim, B * w.n_kv_heads * w.head_dim
        # two input blocks: the end-to-end step copies step k + 1's inputs into
        # one while step k reads the other
        self.io_ins = [torch.empty(2 * (nq + 2 * nkv), dtype=dt, device="cuda") for _ in range(2)]
        self.io_in = self.io_ins[0]
        # two output blocks: the end-to-end step reads block k % 2 back on a
        # copy stream while the next step writes the other one
        self.io_outs = [torch.empty(2 * nq, dtype=dt, device="cuda") for _ in range(2)]
        self.io_out = self.io_outs[0]
        views = lambda buf, off, n, shape: buf[off:off + n].view(shape)
        qs, kvs = (B, w.n_q_heads, w.head_dim), (B, w.n_kv_heads, w.head_dim)
        per = nq + 2 * nkv
        # per input block: (q, new K, new V) of both layers
        self.in_views = [([views(blk, i * per, nq, qs) for i in range(2)],
                          [views(blk, i * per + nq, nkv, kvs) for i in range(2)],
                          [views(blk, i * per + nq + nkv, nkv, kvs) for i in range(2)]) for blk in self.io_ins]
        self.q, self.kn, self.vn = self.in_views[0]
        for i in range(2):
            self.q[i].copy_(wl.normal(qs, 100 + i, w.dtype, "cuda"))
            self.kn[i].copy_(wl.normal(kvs, 200 + i, w.dtype, "cuda"))
            self.vn[i].copy_(wl.normal(kvs, 300 + i, w.dtype, "cuda"))
        self.o_bufs = [[views(blk, i * nq, nq, qs) for i in range(2)] for blk in self.io_outs]
        self.o = self.o_bufs[0]
        # double-buffered pinned staging for the slots of a step, each buffer
        # reused only after its previous copy has run
        self.slot_host = [torch.empty(2, B, dtype=torch.int32, pin_memory=True) for _ in range(2)]
        self.slot_ready = [None, None]
        self.slot_dev = torch.empty(2, B, dtype=torch.int32, device="cuda")
        self.sess.workspace(B)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        self.steps_done = 0
        self.launches = 0
        self.decode_events = []
        # host-buffer (end-to-end) variants: the pinned input block, and the
        # outputs double-buffered: step k's result goes back to the host on a
        # copy stream while step k + 1 runs (the host waits for step k's copy
        # before it returns from step k + 1, and step k + 2 writes the block
        # only after that copy)
        self.h_in = self.io_in.cpu().pin_memory()
        self.h_o = [torch.empty_like(self.io_out, device="cpu").pin_memory() for _ in range(2)]
        self.out_ready = [None, None]
        self.in_ready = [None, None]  # input block b's copy from the host (on the copy stream)
        self.in_free = [None, None]   # the last step that read input block b has run
        self.copy_stream = torch.cuda.Stream()  # results to the host
        self.in_stream = torch.cuda.Stream()    # inputs from the host: never queued behind a result copy
        self.out_sum = 0.0
        torch.cuda.synchronize()

    def lens(self):
        return self.sess.tables()[2][:self.B].astype(np.int64)

    def step(self, time_full_decode=False, host_io=False):
        torch, sess, B = self.torch, self.sess, self.B
        fs, ss = sess.reserve(range(B), [1] * B)
        buf = self.steps_done & 1
        if self.slot_ready[buf] is not None:
            self.slot_ready[buf].synchronize()
        if host_io:
            # the result of the step two back, which used output block buf,
            # is read on the host before this step's copy overwrites it:
            # two steps stay in flight
            self.read_output(buf)
        with torch.cuda.stream(self.stream):
            q, kn, vn = self.q, self.kn, self.vn
            if host_io:
                # the step's inputs, both layers, one copy (issued ahead by
                # the previous step); waited for before the step's small
                # copies, so that no cross-stream wait sits between the
                # table update and the decode kernels
                if self.in_ready[buf] is None:
                    self.copy_in(buf)
                self.stream.wait_event(self.in_ready[buf])
                self.in_ready[buf] = None
                q, kn, vn = self.in_views[buf]
                if self.out_ready[buf] is not None:  # block buf's previous copy to the host
                    self.stream.wait_event(self.out_ready[buf])
            self.slot_host[buf][0].numpy()[:] = fs
            self.slot_host[buf][1].numpy()[:] = ss
            self.slot_dev.copy_(self.slot_host[buf], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.stream)
            self.slot_ready[buf] = ev
            sess.sync()
            self.launches += 1
            out = self.o_bufs[buf] if host_io else self.o
            for i in range(2):
                if time_full_decode and i == 0:
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(self.stream)
                # append the new token's K/V and attend, one call (plan, main, combine)
                sess.decode_append(i, q[i], kn[i], vn[i], self.slot_dev[i], out[i], B, self.scale)
                if time_full_decode and i == 0:
                    e1.record(self.stream)
                    self.decode_events.append((e0, e1))
                self.launches += 3
            if host_io:  # the step's outputs, both layers, one copy, on the copy stream
                done = torch.cuda.Event()
                done.record(self.stream)
                self.copy_stream.wait_event(done)
                with torch.cuda.stream(self.copy_stream):
                    self.h_o[buf].copy_(self.io_outs[buf], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(self.copy_stream)
                self.out_ready[buf] = ev
                self.in_free[buf] = done
                self.copy_in(1 - buf)  # the next step's inputs, while this one runs
        self.steps_done += 1
        if self.steps_done % 64 == 0:
            sess.release(range(B))

    def copy_in(self, b):
        """Copy a step's inputs from pinned host memory into input block b on
        the input stream, once the last step that read the block has run."""
        torch = self.torch
        with torch.cuda.stream(self.in_stream):
            if self.in_free[b] is not None:
                self.in_stream.wait_event(self.in_free[b])
            self.io_ins[b].copy_(self.h_in, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.in_stream)
        self.in_ready[b] = ev

    def join_copies(self):
        """The compute stream waits for the copies still in flight."""
        for ev in self.out_ready + self.in_ready:
            if ev is not None:
                self.stream.wait_event(ev)

    def read_output(self, buf):
        if self.out_ready[buf] is not None:
            self.out_ready[buf].synchronize()
            self.out_ready[buf] = None
            self.out_sum += float(self.h_o[buf][0]) + float(self.h_o[buf][-1])

    def breakdown(self, steps):
        """Average device time of each call of the decode step (events around
        every call; a diagnostic, not the timed bench)."""
        torch, sess, B = self.torch, self.sess, self.B
        names = ["sync", "append_full", "decode_full", "append_swa", "decode_swa"]
        acc = {n: 0.0 for n in names}
        for _ in range(steps):
            fs, ss = sess.reserve(range(B), [1] * B)
            self.stream.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            with torch.cuda.stream(self.stream):
                self.slot_host[0][0].numpy()[:] = fs
                self.slot_host[0][1].numpy()[:] = ss
                self.slot_dev.copy_(self.slot_host[0], non_blocking=True)
                ev[0].record(self.stream)
                sess.sync()
                ev[1].record(self.stream)
                for i in range(2):
                    sess.append(i, self.kn[i], self.vn[i], self.slot_dev[i])
                    ev[2 + 2 * i].record(self.stream)
                    sess.decode(i, self.q[i], self.o[i], B, self.scale)
                    ev[3 + 2 * i].record(self.stream)
            self.stream.synchronize()
            for k, n in enumerate(names):
                acc[n] += ev[k].elapsed_time(ev[k + 1]) * 1e3
            self.steps_done += 1
            if self.steps_done % 64 == 0:
                sess.release(range(B))
        out = {n: round(v / steps, 2) for n, v in acc.items()}
        # the same calls queued back to back (launch latency hidden)
        def queued(fn, reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                e0.record(self.stream)
                for _ in range(reps):
                    fn()
                e1.record(self.stream)
            self.stream.synchronize()
            return round(e0.elapsed_time(e1) * 1e3 / reps, 2)
        out["queued_append"] = queued(lambda: sess.append(1, self.kn[1], self.vn[1], self.slot_dev[1]), 200)
        out["queued_decode_swa"] = queued(lambda: sess.decode(1, self.q[1], self.o[1], B, self.scale), 200)
        out["queued_decode_full"] = queued(lambda: sess.decode(0, self.q[0], self.o[0], B, self.scale), 20)
        out["queued_decode_append_swa"] = queued(
            lambda: sess.decode_append(1, self.q[1], self.kn[1], self.vn[1], self.slot_dev[1], self.o[1], B,
                                       self.scale), 200)
        return out

    def finish(self):
        self.stream.synchronize()
        st = self.sess.check()
        if st != 0:
            raise RuntimeError("device status %d after benchmark" % st)


class ChunkedPrefill:
    """The chunked-prefill workload on the GPU through the C ABI.

    Setup reserves the cached prefixes (chunk by chunk, releasing the SWA
    window after each) and then the 4096-token chunk of every sequence. A
    timed step appends the chunk's K/V to the Full and the SWA pool and runs
    the Full and the SWA prefill; repeating it recomputes the same chunk, so
    every step has the same prefixes. The SWA release of the chunk runs once,
    after the last step."""

    def __init__(self, w, fp8=False):
        import torch
        import hybrid_sliding_window_dual_gb300 as H
        from hybrid_sliding_window_dual_gb300.session import DualPoolSession
        self.torch, self.w = torch, w
        B, P, W, C = len(w.cached), w.page_size, w.window, w.n_new
        self.B = B
        full_pages = sum(math.ceil((L + C) / P) for L in w.cached) + 16
        swa_pages = B * (math.ceil((W + C) / P) + 2) + 16
        max_pages = max(math.ceil((L + C) / P) for L in w.cached) + 1
        cfg = H.Config(window=W, page_size=P, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, dtype=H.HSWA_DTYPE_FP8_E4M3 if fp8 else w.dtype,
                       full_pages=full_pages, swa_pages=swa_pages, max_seqs=B, max_pages_per_seq=max_pages)
        self.stream = torch.cuda.Stream()
        self.sess = DualPoolSession(cfg, [wl.KIND_FULL, wl.KIND_SWA], wl.permutation(full_pages, w.seed),
                                    wl.permutation(swa_pages, w.seed + 1), stream=self.stream, init="empty")
        for s, L in enumerate(w.cached):
            for start in range(0, L, C):
                self.sess.reserve([s], [min(C, L - start)])
                self.sess.release([s])
        self.prefix = np.array(w.cached, np.int64)
        fs, ss = self.sess.reserve(range(B), [C] * B)
        with torch.cuda.stream(self.stream):
            for i in range(2):
                for t, seed in ((self.sess.k[i], 10 + i), (self.sess.v[i], 20 + i)):
                    g = torch.Generator(device="cuda")
                    g.manual_seed(seed)
                    flat = t.view(-1)
                    for j in range(0, flat.numel(), 1 << 28):
                        n = min(1 << 28, flat.numel() - j)
                        if fp8:  # seeded E4M3 codes without the NaN patterns
                            mag = torch.randint(0, 0x7F, (n,), generator=g, device="cuda", dtype=torch.int32)
                            sgn = torch.randint(0, 2, (n,), generator=g, device="cuda", dtype=torch.int32)
                            flat[j:j + n] = (mag | (sgn << 7)).to(torch.uint8)
                        else:
                            flat[j:j + n] = torch.randn(n, generator=g, device="cuda").to(t.dtype)
                if fp8:
                    self.sess.ks[i].uniform_(0.001, 0.011)
                    self.sess.vs[i].uniform_(0.001, 0.011)
            self.sess.sync()
        T = B * C
        self.T, self.C = T, C
        dt = wl.TORCH_DTYPE[w.dtype]
        self.slots = [torch.as_tensor(fs, device="cuda"), torch.as_tensor(ss, device="cuda")]
        self.q = [wl.normal((T, w.n_q_heads, w.head_dim), 400 + i, w.dtype, "cuda") for i in range(2)]
        self.kn = [wl.normal((T, w.n_kv_heads, w.head_dim), 500 + i, w.dtype, "cuda") for i in range(2)]
        self.vn = [wl.normal((T, w.n_kv_heads, w.head_dim), 600 + i, w.dtype, "cuda") for i in range(2)]
        self.o = [torch.empty(T, w.n_q_heads, w.head_dim, dtype=dt, device="cuda") for _ in range(2)]
        self.d_prefix = torch.as_tensor(self.prefix.astype(np.int32), device="cuda")
        self.d_qs = torch.arange(0, T + 1, C, dtype=torch.int32, device="cuda")
        self.q_start_host = np.arange(0, T + 1, C)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        self.events = [[], []]
        self.kernels = ["", ""]
        self.launches = 0
        torch.cuda.synchronize()

    def flops(self):
        return prefill_flops(self.w, self.prefix.tolist(), [self.C] * self.B)

    def step(self, timed=False):
        torch = self.torch
        from hybrid_sliding_window_dual_gb300 import hswa_last_kernel
        with torch.cuda.stream(self.stream):
            for i in range(2):
                self.sess.append(i, self.kn[i], self.vn[i], self.slots[i])
                if timed:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(self.stream)
                self.sess.prefill(i, self.q[i], self.o[i], self.d_prefix, self.d_qs, self.B, self.C, self.scale,
                                  prefix_host=self.prefix, q_start_host=self.q_start_host)
                self.kernels[i] = hswa_last_kernel()
                if timed:
                    e1.record(self.stream)
                    self.events[i].append((e0, e1))
                self.launches += 2

    def finish(self):
        self.sess.release(range(self.B))
        self.stream.synchronize()
        st = self.sess.check()
        if st != 0:
            raise RuntimeError("device status %d after benchmark" % st)


def measure_prefill(steps, warmup, w, fp8=False, clocks=None):
    """Whole-chunk TFLOP/s of the chunked-prefill workload (valid pairs only);
    over FP8 pools when fp8 (the staging pass is inside each layer's time).
    clocks: a ClockSampler, summarised over the warm-up and timed steps."""
    if clocks is not None:
        clocks.start()  # before the set-up, so that sampling runs by the first step
    pb = ChunkedPrefill(w, fp8=fp8)
    if clocks is not None:
        pb.stream.synchronize()
        clocks.mark()
    for _ in range(warmup):
        pb.step()
    pb.stream.synchronize()
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pb.stream)
    for _ in range(steps):
        pb.step(timed=True)
    e1.record(pb.stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark()
    clock_info = clocks.stop() if clocks is not None else None
    secs = e0.elapsed_time(e1) / 1e3
    f = pb.flops()
    full_ms = float(np.mean([a.elapsed_time(b) for a, b in pb.events[0]]))
    swa_ms = float(np.mean([a.elapsed_time(b) for a, b in pb.events[1]]))
    pb.finish()
    return {"kernel": pb.kernels[0], "swa_kernel": pb.kernels[1],
            "step_tflops": f["step"] * steps / secs / 1e12, "ms_per_step": secs / steps * 1e3,
            "full_tflops": f["full"] / (full_ms / 1e3) / 1e12, "full_ms": full_ms,
            "full_exec_tflops": f["full_exec"] / (full_ms / 1e3) / 1e12,
            "swa_tflops": f["swa"] / (swa_ms / 1e3) / 1e12, "swa_ms": swa_ms,
            "swa_exec_tflops": f["swa_exec"] / (swa_ms / 1e3) / 1e12,
            "swa_gbs": swa_prefill_bytes(w, pb.prefix.tolist(), [pb.C] * pb.B) / (swa_ms / 1e3) / 1e9,
            "valid_tflop_per_step": f["step"] / 1e12, "tokens_per_s": pb.T * steps / secs,
            "launches": pb.launches, "clocks": clock_info}


def fill_normal(t, seed):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    flat = t.view(-1)
    for j in range(0, flat.numel(), 1 << 28):
        n = min(1 << 28, flat.numel() - j)
        flat[j:j + n] = torch.randn(n, generator=g, device="cuda").to(t.dtype)


def hybrid70_bytes(w, lens):
    """Algorithmic bytes of one 70-layer decode step and the pool sizing."""
    es = KV_ROW[w.dtype]
    row = w.n_kv_heads * w.head_dim * es
    B = len(lens)
    n_full = sum(1 for k in w.layer_kinds if k == wl.KIND_FULL)
    n_swa = len(w.layer_kinds) - n_full
    full_kv = 2 * row * int(np.sum(lens))
    swa_kv = 2 * row * int(np.sum(np.minimum(lens, w.window)))
    per_layer = 2 * B * w.n_q_heads * w.head_dim * es + 2 * 2 * B * row
    return {"step": n_full * full_kv + n_swa * swa_kv + len(w.layer_kinds) * per_layer,
            "full_layer": full_kv + per_layer, "n_full": n_full, "n_swa": n_swa}


class Hybrid70:
    """The 70-layer attention-only decode step (10 Full + 60 SWA, Full at
    every 7th layer), batch 128 at 128K cached tokens each. The ten Full
    layers read one physical Full pool (640 GiB of per-layer Full pools do
    not fit in HBM; each layer still reads its 64 GiB from HBM)."""

    def __init__(self, w, extra_steps, n_seqs=None):
        import torch
        import hybrid_sliding_window_dual_gb300 as H
        from hybrid_sliding_window_dual_gb300.session import DualPoolSession
        self.torch, self.w = torch, w
        B, P, W = len(w.cached), w.page_size, w.window
        self.B = B
        pages_per_seq = math.ceil((max(w.cached) + extra_steps + 1) / P)
        full_pages = B * pages_per_seq + 16
        swa_pages = B * (math.ceil((W + 64) / P) + 2) + math.ceil((W + 4096) / P) + 16
        cfg = H.Config(window=W, page_size=P, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, dtype=w.dtype, full_pages=full_pages, swa_pages=swa_pages,
                       max_seqs=B, max_pages_per_seq=pages_per_seq + 1)
        self.stream = torch.cuda.Stream()
        self.sess = DualPoolSession(cfg, list(w.layer_kinds), None, None, stream=self.stream, init="empty",
                                    share_full_pool=True)
        for s, L in enumerate(w.cached):
            for start in range(0, L, 4096):
                self.sess.reserve([s], [min(4096, L - start)])
                self.sess.release([s])
        self.full_pool_layer = list(w.layer_kinds).index(wl.KIND_FULL)
        with torch.cuda.stream(self.stream):
            for i, kind in enumerate(w.layer_kinds):
                if kind == wl.KIND_FULL and i != self.full_pool_layer:
                    continue
                fill_normal(self.sess.k[i], 1000 + 2 * i)
                fill_normal(self.sess.v[i], 1001 + 2 * i)
            self.sess.sync()
        dt = wl.TORCH_DTYPE[w.dtype]
        nl = len(w.layer_kinds)
        self.q = [wl.normal((B, w.n_q_heads, w.head_dim), 2000 + i, w.dtype, "cuda") for i in range(nl)]
        self.kn = [wl.normal((B, w.n_kv_heads, w.head_dim), 3000 + i, w.dtype, "cuda") for i in range(nl)]
        self.vn = [wl.normal((B, w.n_kv_heads, w.head_dim), 4000 + i, w.dtype, "cuda") for i in range(nl)]
        self.o = [torch.empty(B, w.n_q_heads, w.head_dim, dtype=dt, device="cuda") for _ in range(nl)]
        self.slot_host = torch.empty(2, B, dtype=torch.int32, pin_memory=True)
        self.slot_dev = torch.empty(2, B, dtype=torch.int32, device="cuda")
        self.sess.workspace(B)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        self.steps_done = 0
        self.launches = 0
        self.full_events = []
        torch.cuda.synchronize()

    def lens(self):
        return self.sess.tables()[2][:self.B].astype(np.int64)

    def step(self, timed=False):
        torch, sess, B = self.torch, self.sess, self.B
        fs, ss = sess.reserve(range(B), [1] * B)
        self.stream.synchronize()  # the slot staging of the previous step has been copied
        with torch.cuda.stream(self.stream):
            self.slot_host[0].numpy()[:] = fs
            self.slot_host[1].numpy()[:] = ss
            self.slot_dev.copy_(self.slot_host, non_blocking=True)
            sess.sync()
            self.launches += 1
            for i, kind in enumerate(self.w.layer_kinds):
                if timed and kind == wl.KIND_FULL:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(self.stream)
                sess.decode_append(i, self.q[i], self.kn[i], self.vn[i],
                                   self.slot_dev[0 if kind == wl.KIND_FULL else 1], self.o[i], B, self.scale)
                if timed and kind == wl.KIND_FULL:
                    e1.record(self.stream)
                    self.full_events.append((e0, e1))
                self.launches += 3
        self.steps_done += 1
        if self.steps_done % 64 == 0:
            sess.release(range(B))

    def offload(self):
        """Untimed: gather every SWA window to pinned host memory, evict the
        SWA segments and give the windows new pages (their bytes are stale
        until reloaded)."""
        torch, sess, B = self.torch, self.sess, self.B
        swa = [i for i, k in enumerate(self.w.layer_kinds) if k == wl.KIND_SWA]
        off, nbytes = sess.window_offsets(swa[0], B)
        self.d_off = torch.as_tensor(off, device="cuda")
        n = nbytes // KV_ROW[self.w.dtype]
        if not hasattr(self, "host") or self.host[0].numel() != n:
            self.host = [torch.empty(n, dtype=wl.TORCH_DTYPE[self.w.dtype], pin_memory=True) for _ in swa]
        with torch.cuda.stream(self.stream):
            for buf, ly in zip(self.host, swa):
                sess.gather(ly, self.d_off, B, buf)
        self.stream.synchronize()
        sess.swa_drop(range(B))
        sess.swa_restore(range(B))
        with torch.cuda.stream(self.stream):
            sess.sync()
            self.d_len_snap = sess.d_seq_len.clone()
        self.stream.synchronize()
        self.reload_bytes = len(swa) * n * KV_ROW[self.w.dtype]
        return swa

    def reload_step(self, mode):
        """One 70-layer step whose SWA windows all come back from the host
        tier: "serial" (every window before layer 0), "direct" (scatter
        kernels reading pinned host memory on a side stream, layer by layer)
        or "staged" (copy engines into a staging ring, device scatter right
        before each layer). Returns the device time in ms."""
        torch, sess, B = self.torch, self.sess, self.B
        swa = self.offload()
        if not hasattr(self, "side"):
            self.side = torch.cuda.Stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fs, ss = sess.reserve(range(B), [1] * B)
        self.stream.synchronize()
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            self.slot_host[0].numpy()[:] = fs
            self.slot_host[1].numpy()[:] = ss
            self.slot_dev.copy_(self.slot_host, non_blocking=True)
            sess.sync()
            self.side.wait_stream(self.stream)
            events, staged = {}, None
            if mode == "staged":
                from hybrid_sliding_window_dual_gb300.session import LayerwiseReload
                n = self.host[0].numel()
                if not hasattr(self, "staging"):
                    self.staging = [torch.empty(n, dtype=self.host[0].dtype, device="cuda") for _ in range(8)]
                staged = LayerwiseReload(sess, swa, self.d_len_snap, self.d_off, B, self.host, self.side,
                                         self.staging)
                staged.start(self.stream)
            else:
                events = sess.reload_async(swa, self.d_len_snap, self.d_off, B, self.host, self.side)
                if mode == "serial":
                    self.stream.wait_stream(self.side)
            for i, kind in enumerate(self.w.layer_kinds):
                if mode == "direct" and i in events:
                    self.stream.wait_event(events[i])
                if staged is not None:
                    staged.before_layer(i, self.stream)
                sess.decode_append(i, self.q[i], self.kn[i], self.vn[i],
                                   self.slot_dev[0 if kind == wl.KIND_FULL else 1], self.o[i], B, self.scale)
            e1.record(self.stream)
        self.stream.synchronize()
        self.steps_done += 1
        return e0.elapsed_time(e1)

    def sizing(self):
        """Dual pool (per-layer Full pools + live SWA pages) against one O(N)
        pool for all 70 layers, in bytes, at the current lengths."""
        w = self.w
        page_bytes = 2 * w.n_kv_heads * w.page_size * w.head_dim * KV_ROW[w.dtype]
        f, s, lens = self.sess.tables()
        full_live = int((f >= 0).sum())
        swa_live = int((s >= 0).sum())
        n_full = sum(1 for k in w.layer_kinds if k == wl.KIND_FULL)
        n_swa = len(w.layer_kinds) - n_full
        dual = (n_full * full_live + n_swa * swa_live) * page_bytes
        single = len(w.layer_kinds) * full_live * page_bytes
        return {"dual_pool_bytes": dual, "single_pool_bytes": single, "ratio": round(dual / single, 5),
                "capacity_gain": round(single / dual, 3), "live_swa_pages_per_seq": round(swa_live / self.B, 2)}


class SwaTransfer:
    """Transfer by SWA mask: 256 sequences (lognormal lengths, median 16K, cap
    256K), 60 SWA layers. A step gathers the in-window tokens of every layer
    into a pinned host buffer (the kernel writes host memory directly), evicts
    the SWA segments, gives the windows fresh pages and scatters the host
    copies back. fp8=True: FP8 E4M3 pools with per-token-head scales (the
    packed window carries codes and scales)."""

    def __init__(self, w, fp8=False):
        import torch
        import hybrid_sliding_window_dual_gb300 as H
        from hybrid_sliding_window_dual_gb300.session import DualPoolSession
        self.torch, self.w, self.H = torch, w, H
        B, P, W = len(w.cached), w.page_size, w.window
        self.B = B
        extra = 4 * 64 + 8
        full_pages = sum(math.ceil((L + extra) / P) for L in w.cached) + 16
        swa_pages = 2 * B * (math.ceil((W + 64) / P) + 2) + math.ceil((W + 4096) / P) + 16
        max_pages = max(math.ceil((L + extra) / P) for L in w.cached) + 1
        self.fp8 = fp8
        cfg = H.Config(window=W, page_size=P, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, dtype=H.HSWA_DTYPE_FP8_E4M3 if fp8 else w.dtype,
                       full_pages=full_pages, swa_pages=swa_pages, max_seqs=B, max_pages_per_seq=max_pages)
        self.stream = torch.cuda.Stream()
        self.sess = DualPoolSession(cfg, list(w.layer_kinds), None, wl.permutation(swa_pages, w.seed),
                                    stream=self.stream, init="empty")
        for s, L in enumerate(w.cached):
            for start in range(0, L, 4096):
                self.sess.reserve([s], [min(4096, L - start)])
                self.sess.release([s])
        with torch.cuda.stream(self.stream):
            for i in range(len(w.layer_kinds)):
                if fp8:  # seeded E4M3 codes without the NaN patterns, seeded scales
                    for t, seed in ((self.sess.k[i], 5000 + 2 * i), (self.sess.v[i], 5001 + 2 * i)):
                        g = torch.Generator(device="cuda")
                        g.manual_seed(seed)
                        mag = torch.randint(0, 0x7F, t.shape, generator=g, device="cuda", dtype=torch.uint8)
                        sgn = torch.randint(0, 2, t.shape, generator=g, device="cuda", dtype=torch.uint8)
                        t.copy_(mag | (sgn << 7))
                    self.sess.ks[i].uniform_(0.001, 0.011)
                    self.sess.vs[i].uniform_(0.001, 0.011)
                else:
                    fill_normal(self.sess.k[i], 5000 + 2 * i)
                    fill_normal(self.sess.v[i], 5001 + 2 * i)
            self.sess.sync()
        self.refresh_offsets()
        if fp8:
            self.host = [torch.empty(self.moved_bytes(), dtype=torch.uint8, pin_memory=True)
                         for _ in range(len(w.layer_kinds))]
        else:
            n = self.moved_bytes() // KV_ROW[w.dtype]
            self.host = [torch.empty(n, dtype=wl.TORCH_DTYPE[w.dtype], pin_memory=True)
                         for _ in range(len(w.layer_kinds))]
        self.launches = 0
        torch.cuda.synchronize()

    def refresh_offsets(self):
        self.off, self.nbytes = self.sess.window_offsets(0, self.B)
        self.d_off = self.torch.as_tensor(self.off, device="cuda")

    def moved_bytes(self):
        """Bytes of one layer's packed windows (FP8: a code byte per element
        plus an fp32 scale per token, head and tensor), from the library."""
        return self.nbytes

    def gather_all(self):
        with self.torch.cuda.stream(self.stream):
            for i in range(len(self.w.layer_kinds)):
                self.sess.gather(i, self.d_off, self.B, self.host[i])
                self.launches += 1

    def scatter_all(self):
        with self.torch.cuda.stream(self.stream):
            for i in range(len(self.w.layer_kinds)):
                self.sess.scatter(i, self.d_off, self.B, self.host[i])
                self.launches += 1

    def evict_and_restore(self):
        self.stream.synchronize()
        self.sess.swa_drop(range(self.B))
        self.sess.swa_restore(range(self.B))
        with self.torch.cuda.stream(self.stream):
            self.sess.sync()
            self.launches += 1

    def release_rounds(self, rounds=4, tokens=64):
        """Ring release: `tokens` decode tokens per sequence, then one release."""
        times, live = [], []
        for _ in range(rounds):
            for _ in range(tokens):
                self.sess.reserve(range(self.B), [1] * self.B)
            t0 = time.perf_counter()
            self.sess.release(range(self.B))
            times.append(time.perf_counter() - t0)
            live.append(int((self.sess.tables()[1] >= 0).sum(axis=1).max()))
        with self.torch.cuda.stream(self.stream):
            self.sess.sync()
        self.refresh_offsets()
        return times, live


def time_steps(run, steps, stream, world, finish=None):
    """Seconds for `steps` calls of run(), events on `stream`; finish() (if
    given) makes `stream` wait for work the steps left on other streams."""
    import torch
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    if finish is not None:
        finish()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / 1e3


def workload(args, name):
    if name == "decode_batch":
        w = wl.decode_batch()
    elif name == "swa_transfer":
        w = wl.swa_transfer()
    else:
        w = wl.chunked_prefill()
    if args.seqs:
        import dataclasses
        w = dataclasses.replace(w, cached=w.cached[:args.seqs])
    return w


def decode_config(w, world):
    """The decode-batch workload as both arms report it."""
    kv = decode_bytes(w, np.asarray(w.cached, np.int64) + 1)
    return {"workload": "decode_batch", "seqs": len(w.cached), "cached_len": "uniform[1024,32768] seed 2",
            "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
            "page": w.page_size, "window": w.window, "layers": "1 Full + 1 SWA",
            "l2": "inputs larger than L2 (%.1f GB KV per step)" % (kv["step"] / 1e9),
            "parallelism": "replicas" if world > 1 else "single"}


def run_decode(args, world, rank, local):
    import torch
    w = workload(args, "decode_batch")
    total_steps = args.warmup + 2 * args.steps + 64
    bench = DecodeBatch(w, total_steps)
    hbm, _, _, peak_kind = peaks()
    # clocks are sampled from before the warm-up to the end of the timed region
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    for _ in range(args.warmup):
        bench.step()
    bench.stream.synchronize()
    bytes_before = decode_bytes(w, bench.lens() + 1)  # lengths the first timed step decodes
    launches0 = bench.launches
    secs = time_steps(lambda: bench.step(time_full_decode=True), args.steps, bench.stream, world)
    clock_info = clocks.stop()
    launches = bench.launches - launches0
    bytes_after = decode_bytes(w, bench.lens())
    step_bytes = 0.5 * (bytes_before["step"] + bytes_after["step"])  # lengths grow by one per step
    full_layer_bytes = 0.5 * (bytes_before["full_layer"] + bytes_after["full_layer"])
    dec_ms = [a.elapsed_time(b) for a, b in bench.decode_events]
    bench.decode_events.clear()
    if args.breakdown:
        bd = bench.breakdown(50)
    # end to end: host buffers in, host buffers out, copies inside the timed
    # region; these steps come after the device-timed ones, so their bytes
    # are counted from their own lengths (every step appends a token)
    e2e_before = decode_bytes(w, bench.lens() + 1)
    e2e_secs = time_steps(lambda: bench.step(host_io=True), args.steps, bench.stream, world,
                          finish=bench.join_copies)
    for b in range(2):  # the last two steps' results
        bench.read_output(b)
    e2e_after = decode_bytes(w, bench.lens())
    e2e_step_bytes = 0.5 * (e2e_before["step"] + e2e_after["step"])
    bench.finish()
    secs = max_over_ranks(secs, world)
    e2e_secs = max_over_ranks(e2e_secs, world)
    total_bytes = sum_over_ranks(step_bytes * args.steps, world)
    e2e_bytes = sum_over_ranks(e2e_step_bytes * args.steps, world)
    value = total_bytes / secs / 1e9
    es = KV_ROW[w.dtype]
    B = len(w.cached)
    h2d = 2 * (B * w.n_q_heads * w.head_dim * es + 2 * B * w.n_kv_heads * w.head_dim * es)
    d2h = 2 * B * w.n_q_heads * w.head_dim * es
    dec_s = float(np.mean(dec_ms)) / 1e3
    achieved = full_layer_bytes / dec_s / 1e9
    line = {
        "metric": "Hybrid-SWA attn: decode HBM GB/s and prefill TFLOP/s (% of GB300 peak)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": decode_config(w, world),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": decode_traffic(full_layer_bytes),
                     "kernel": "decode_mma_bf16_d128 with fused append (Full layer; plan + main + combine)",
                     "peak_source": peak_kind, "frac_of_8tbs": round(achieved / 8000.0, 4)},
        "e2e": {"value": round(e2e_bytes / e2e_secs / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clock_info,
        "tokens_per_s": round(world * B * args.steps / secs, 1),
    }
    if args.breakdown:
        line["breakdown_us"] = bd
    if not args.no_fp8:
        del bench
        torch.cuda.empty_cache()
        f8 = measure_decode_fp8(200, 5)
        line["fp8_decode"] = {
            "workload": "decode_batch over FP8 E4M3 pools (scale per token, kv head, 128-element tile)",
            "gbs": round(f8["gbs"], 1), "unit": "GB/s", "frac": round(f8["gbs"] / hbm, 4),
            "ms_per_step": round(f8["ms_per_step"], 4), "tokens_per_s": round(f8["tokens_per_s"], 1),
            "full_layer_gbs": round(f8["full_layer_gbs"], 1), "full_layer_ms": round(f8["full_layer_ms"], 4),
            "kernel": "decode_mma_fp8_d128"}
        bench = None
    if not args.no_multi:
        del bench
        torch.cuda.empty_cache()
        mt = measure_decode_multi(50, workload(args, "decode_batch"))
        base = mt[1]["step_ms"]
        line["multi_token_decode"] = {
            "workload": "decode_batch, n_tok query tokens per sequence (MTP / speculative verification), "
                        "Full + SWA layer per step, no append",
            "by_n_tok": {str(T): {"kernel": v["kernel"], "step_ms": round(v["step_ms"], 4),
                                  "tokens_per_s": round(v["tokens_per_s"], 1),
                                  "full_layer_gbs": round(v["full_layer_gbs"], 1),
                                  "frac": round(v["full_layer_gbs"] / hbm, 4),
                                  "time_vs_1": round(v["step_ms"] / base, 3)} for T, v in mt.items()}}
        if not args.no_fp8:
            torch.cuda.empty_cache()
            mt8 = measure_decode_multi(50, workload(args, "decode_batch"), token_counts=(1, 2, 3, 4, 8, 16), fp8=True)
            base8 = mt8[1]["step_ms"]
            line["multi_token_decode_fp8"] = {
                "workload": "decode_batch over FP8 E4M3 pools, n_tok query tokens per sequence, Full + SWA "
                            "layer per step (2 tokens: one mma.sync pass; 3 and more: the tensor-core kernel)",
                "by_n_tok": {str(T): {"kernel": v["kernel"], "step_ms": round(v["step_ms"], 4),
                                      "tokens_per_s": round(v["tokens_per_s"], 1),
                                      "full_layer_gbs": round(v["full_layer_gbs"], 1),
                                      "time_vs_1": round(v["step_ms"] / base8, 3)} for T, v in mt8.items()}}
        bench = None
    if not args.no_prefill:
        del bench
        torch.cuda.empty_cache()
        hbm, bf16, bf16_sus, _ = peaks()
        pf = measure_prefill(args.prefill_steps, 1, workload(args, "chunked_prefill"),
                             clocks=ClockSampler(local, "_prefill"))
        line["prefill"] = {
            "workload": "chunked_prefill (8 seqs, prefix U[8192,65536] seed 3, chunk 4096, Full + SWA layer)",
            "tflops": round(pf["step_tflops"], 1), "unit": "TFLOP/s", "frac": round(pf["step_tflops"] / bf16, 4),
            "peak": bf16, "peak_kind": "bf16 burst (measured; the timed region is a few steps of ~30 ms)",
            "frac_of_sustained": round(pf["step_tflops"] / bf16_sus, 4), "peak_sustained": bf16_sus,
            "full_layer_frac": round(pf["full_tflops"] / bf16, 4),
            "full_layer_tflops": round(pf["full_tflops"], 1), "full_layer_ms": round(pf["full_ms"], 3),
            "full_layer_exec_tflops": round(pf["full_exec_tflops"], 1),
            "swa_layer_tflops": round(pf["swa_tflops"], 2), "swa_layer_ms": round(pf["swa_ms"], 3),
            "swa_layer_exec_tflops": round(pf["swa_exec_tflops"], 2),
            "swa_layer_frac": round(pf["swa_tflops"] / bf16, 4),
            "swa_layer_gbs": round(pf["swa_gbs"], 1), "swa_layer_hbm_frac": round(pf["swa_gbs"] / hbm, 4),
            "valid_tflop_per_step": round(pf["valid_tflop_per_step"], 3),
            "ms_per_step": round(pf["ms_per_step"], 3), "tokens_per_s": round(pf["tokens_per_s"], 1),
            "kernel": pf["kernel"], "swa_kernel": pf["swa_kernel"], "clocks": pf["clocks"]}
        if not args.no_fp8:
            del pf
            torch.cuda.empty_cache()
            p8 = measure_prefill(max(2, args.prefill_steps // 2), 1, workload(args, "chunked_prefill"), fp8=True)
            line["prefill"]["fp8"] = {
                "workload": "the same chunk over FP8 E4M3 pools (scale per token, kv head, 128-element tile)",
                "tflops": round(p8["step_tflops"], 1), "frac": round(p8["step_tflops"] / bf16, 4),
                "full_layer_tflops": round(p8["full_tflops"], 1), "full_layer_ms": round(p8["full_ms"], 3),
                "swa_layer_ms": round(p8["swa_ms"], 3), "ms_per_step": round(p8["ms_per_step"], 3),
                "kernel": p8["kernel"].replace("+", " + prefill_q_to_f16 + ") + " (staging inside the layer time)"}
    if not args.no_hybrid70:
        h = measure_hybrid70(args.hybrid_steps, 2)
        line["hybrid70"] = {
            "workload": "hybrid70 (10 Full + 60 SWA layers, batch 128 x 131072 cached, 64/8 heads, d 128)",
            "gbs": round(h["gbs"], 1), "unit": "GB/s", "frac": round(h["gbs"] / hbm, 4),
            "ms_per_step": round(h["ms_per_step"], 3), "tokens_per_s": round(h["tokens_per_s"], 1),
            "full_layer_gbs": round(h["full_layer_gbs"], 1), "full_layer_ms": round(h["full_layer_ms"], 3),
            "step_gb": round(h["step_bytes"] / 1e9, 2), "sizing": h["sizing"],
            "swa_reload": {"gb_from_host": round(h["reload"]["bytes"] / 1e9, 3),
                           "step_ms_resident": round(h["reload"]["step_ms_resident"], 3),
                           "step_ms_serial_reload": round(h["reload"]["step_ms_serial"], 3),
                           "step_ms_layerwise_direct": round(h["reload"]["step_ms_direct"], 3),
                           "step_ms_layerwise_staged": round(h["reload"]["step_ms_staged"], 3)},
            "note": "the 10 Full layers read one physical 64 GiB Full pool"}
    if not args.no_tree:
        pt = measure_prefix_tree()
        line["prefix_tree"] = {
            "workload": "1000 requests sharing a 16384-token system prompt + 4096 own tokens each, W 128, P 64; "
                        "chunked prefill storing each chunk's prefix after its release, then a follow-up turn "
                        "each (host bookkeeping)", "tree_nodes": pt["nodes"],
            "unit": "us per call (median)", "match_us": round(pt["match"], 1), "share_us": round(pt["share"], 1),
            "insert_us": round(pt["insert"], 1), "evict_64_pages_us": round(pt["evict"], 1),
            "follow_up_full_hits": "%d/%d" % (pt["follow_up_hits"], pt["requests"])}
    if not args.no_transfer:
        t = measure_transfer(3)
        line["swa_transfer"] = {
            "workload": "swa_transfer (256 seqs, lognormal median 16K cap 256K, 60 SWA layers, pinned host)",
            "gather_gbs": round(t["gather_gbs"], 1), "scatter_gbs": round(t["scatter_gbs"], 1), "unit": "GB/s",
            "memcpy_d2h_gbs": round(t["memcpy_d2h_gbs"], 1), "memcpy_h2d_gbs": round(t["memcpy_h2d_gbs"], 1),
            "gather_frac_of_memcpy": round(t["gather_gbs"] / t["memcpy_d2h_gbs"], 3),
            "scatter_frac_of_memcpy": round(t["scatter_gbs"] / t["memcpy_h2d_gbs"], 3),
            "gb_each_way": round(t["bytes_each_way"] / 1e9, 3),
            "gb_if_whole_sequences": round(t["bytes_if_full_sequences"] / 1e9, 1),
            "release_us_per_call": round(t["release_us_per_call"], 1),
            "max_live_swa_pages_per_seq_after_release": t["max_live_swa_pages_per_seq_after_release"]}
        if not args.no_fp8:
            t8 = measure_transfer(2, fp8=True)
            line["swa_transfer"]["fp8"] = {
                "workload": "the same windows over FP8 E4M3 pools (codes + per-token-head scales)",
                "gather_gbs": round(t8["gather_gbs"], 1), "scatter_gbs": round(t8["scatter_gbs"], 1),
                "gb_each_way": round(t8["bytes_each_way"] / 1e9, 3),
                "gather_frac_of_memcpy": round(t8["gather_gbs"] / t8["memcpy_d2h_gbs"], 3),
                "scatter_frac_of_memcpy": round(t8["scatter_gbs"] / t8["memcpy_h2d_gbs"], 3),
                "kernel": "swa_xfer_fp8_kernel"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(w, budget_s=args.cpu_budget)
    return line


# ------------------------------------------------------------ CPU oracle
def oracle_decode_state(w, samples):
    """Oracle-side state of the decode-batch workload: bookkeeping for every
    sequence, KV values only on the pages of the sampled sequences."""
    import oracle
    P, W = w.page_size, w.window
    B = len(w.cached)
    full_pages = sum(math.ceil((L + 256) / P) for L in w.cached) + 16
    swa_pages = B * (math.ceil((W + 4096) / P) + 2) + 16
    max_pages = max(math.ceil((L + 256) / P) for L in w.cached) + 1
    pool = oracle.DualPool(W, P, full_pages, swa_pages, B, max_pages, wl.permutation(full_pages, w.seed),
                           wl.permutation(swa_pages, w.seed + 1))
    for s, L in enumerate(w.cached):
        for start in range(0, L, 4096):
            pool.reserve([s], [min(4096, L - start)])
            pool.swa_release([s])
    rng = np.random.default_rng(7)
    kv = []
    for kind, bt, n in ((0, pool.full_bt, full_pages), (1, pool.swa_bt, swa_pages)):
        shape = (n, w.n_kv_heads, P, w.head_dim)
        k = np.zeros(shape, np.uint16)
        v = np.zeros(shape, np.uint16)
        for s in samples:
            for p in bt[s][bt[s] >= 0]:
                k[p] = (rng.standard_normal(shape[1:]).astype(np.float32).view(np.uint32) >> 16)
                v[p] = (rng.standard_normal(shape[1:]).astype(np.float32).view(np.uint32) >> 16)
        kv.append((k, v))
    return pool, kv


def oracle_decode_step(w, pool, kv, samples, seed):
    """One decode step of the oracle on the sampled sequences: reserve,
    append, Full and SWA attention. Returns the algorithmic bytes covered."""
    import oracle
    B = len(w.cached)
    fs, ss = pool.reserve(range(B), [1] * B)
    rng = np.random.default_rng(seed)
    lens = pool.seq_len[samples]
    nbytes = 0
    for layer, (slots, bt) in enumerate(((fs, pool.full_bt), (ss, pool.swa_bt))):
        k, v = kv[layer]
        newk = (rng.standard_normal((len(samples), w.n_kv_heads, w.head_dim)).astype(np.float32)
                .view(np.uint32) >> 16).astype(np.uint16)
        newv = newk[::-1].copy()
        oracle.append_kv(k, newk, slots[samples])
        oracle.append_kv(v, newv, slots[samples])
        q = (rng.standard_normal((len(samples), w.n_q_heads, w.head_dim)).astype(np.float32)
             .view(np.uint32) >> 16).astype(np.uint16)
        oracle.attention(q, k, v, bt, np.array(samples), lens - 1, 0 if layer == 0 else w.window,
                         1.0 / math.sqrt(w.head_dim))
    b = decode_bytes(w, lens)
    return b["step"]


def cpu_baseline_decode(w, budget_s=20.0):
    import oracle
    B = len(w.cached)
    samples = list(range(8))
    pool, kv = oracle_decode_state(w, samples)
    t0 = time.perf_counter()
    done_bytes, steps = 0, 0
    while time.perf_counter() - t0 < budget_s and steps < 200:
        done_bytes += oracle_decode_step(w, pool, kv, samples, steps)
        steps += 1
    el = time.perf_counter() - t0
    return {"value": round(done_bytes / el / 1e9, 4), "unit": "GB/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": "%d decode steps over sequences %s of %d (Full + SWA layer, bookkeeping for all), %.1f s"
                      % (steps, samples, B, el)}


def run_reference(args, world, rank):
    """The oracle as the reference arm: same workload, metric and unit."""
    if rank != 0:
        return None
    import oracle
    w = wl.decode_batch()
    B = len(w.cached)
    per_step = 2
    samples_all = list(range(B))
    pool, kv = oracle_decode_state(w, samples_all[:per_step * 2])
    for i in range(args.warmup):
        oracle_decode_step(w, pool, kv, samples_all[:per_step], i)
    t0 = time.perf_counter()
    total = 0
    for i in range(args.steps):
        total += oracle_decode_step(w, pool, kv, samples_all[per_step:2 * per_step], 1000 + i)
    el = time.perf_counter() - t0
    value = total / el / 1e9
    return {
        "impl": "reference", "metric": "Hybrid-SWA attn: decode HBM GB/s and prefill TFLOP/s (% of GB300 peak)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(w, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": "%d of %d sequences per step, Full + SWA layer" % (per_step, B)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def measure_hybrid70(steps, warmup, n_seqs=None):
    import torch
    w = wl.hybrid70()
    if n_seqs:
        import dataclasses
        w = dataclasses.replace(w, cached=w.cached[:n_seqs])
    hb = Hybrid70(w, warmup + steps + 2)
    for _ in range(warmup):
        hb.step()
    hb.stream.synchronize()
    before = hybrid70_bytes(w, hb.lens() + 1)
    l0 = hb.launches
    secs = time_steps(lambda: hb.step(timed=True), steps, hb.stream, 1)
    after = hybrid70_bytes(w, hb.lens())
    step_bytes = 0.5 * (before["step"] + after["step"])
    full_ms = float(np.mean([a.elapsed_time(b) for a, b in hb.full_events]))
    sizing = hb.sizing()
    # reload of every SWA window from the host tier inside one step
    reload = {"bytes": 0, "step_ms_resident": secs / steps * 1e3}
    for mode in ("serial", "direct", "staged"):
        # one untimed step per mode first: on a host that has run other jobs,
        # the copy engines' first pass over newly pinned buffers ran at ~47
        # GB/s against ~209 GB/s for every later pass
        hb.reload_step(mode)
        reload["step_ms_" + mode] = float(np.mean([hb.reload_step(mode) for _ in range(2)]))
    reload["bytes"] = hb.reload_bytes
    st = hb.sess.check()
    if st != 0:
        raise RuntimeError("device status %d after hybrid70" % st)
    out = {"gbs": step_bytes * steps / secs / 1e9, "ms_per_step": secs / steps * 1e3,
           "full_layer_gbs": 0.5 * (before["full_layer"] + after["full_layer"]) / (full_ms / 1e3) / 1e9,
           "full_layer_ms": full_ms, "step_bytes": step_bytes, "tokens_per_s": len(w.cached) * steps / secs,
           "launches": hb.launches - l0, "sizing": sizing, "reload": reload}
    del hb
    torch.cuda.empty_cache()
    return out


def measure_prefix_tree(n_req=1000, prompt=16384, turn=4096, reps=1):
    """Host cost of the SWA-aware prefix cache tree (bookkeeping only, no
    device memory): n_req requests share a prompt-token system prompt, each
    adds turn tokens of its own, runs as a chunked prefill (4096-token chunks,
    release after each) and is stored at its end; then every request comes
    back for a follow-up turn (match, share the hit). Each chunk's prefix is
    stored right after the chunk's release, so the tree keeps the SWA window
    of every chunk end (the system prompt's end among them). Returns
    microseconds per call of match, share, insert, and of an eviction that
    frees 64 pages of each kind."""
    import hybrid_sliding_window_dual_gb300 as H
    W, P = 128, 64
    pages_per = (prompt + 2 * turn) // P + 2
    full = n_req * ((turn * 2) // P + 2) + prompt // P + 64
    swa = n_req * 16 + 64  # the tree keeps the window of every chunk end
    cfg = H.Config(window=W, page_size=P, n_q_heads=64, n_kv_heads=8, head_dim=128, dtype=H.HSWA_DTYPE_BF16,
                   full_pages=full, swa_pages=swa, max_seqs=n_req, max_pages_per_seq=pages_per)
    rng = np.random.default_rng(6)
    system = rng.integers(0, 32000, prompt).tolist()
    reqs = [np.array(system + rng.integers(0, 32000, turn).tolist(), np.int32) for _ in range(n_req)]
    t = {"match": [], "share": [], "insert": [], "evict": []}
    for _ in range(reps):
        pool = H.hswa_pool_create(cfg)
        tree = H.hswa_tree_create(pool)
        for s, toks in enumerate(reqs):
            t0 = time.perf_counter()
            m, fp, sp, raw = H.hswa_tree_match(tree, toks, pages_per)
            t1 = time.perf_counter()
            if m:
                H.hswa_seq_share_prefix(pool, s, fp, sp)
            t2 = time.perf_counter()
            t["match"].append(t1 - t0)
            if m:
                t["share"].append(t2 - t1)
            L = m * P
            while L < len(toks):  # prefill chunks: release, then store the prefix
                n = min(4096, len(toks) - L)
                H.hswa_reserve(pool, [s], [n])
                L += n
                H.hswa_swa_release(pool, [s])
                t0 = time.perf_counter()
                H.hswa_tree_insert(tree, s, toks[:L])
                t["insert"].append(time.perf_counter() - t0)
            H.hswa_seq_free(pool, [s])
        nodes = H.hswa_tree_stats(tree)[0]
        hits = 0
        for s, toks in enumerate(reqs):  # follow-up turns
            follow = np.concatenate([toks, np.ones(100, np.int32)])
            t0 = time.perf_counter()
            m, fp, sp, raw = H.hswa_tree_match(tree, follow, pages_per)
            t["match"].append(time.perf_counter() - t0)
            hits += m == len(toks) // P
        t0 = time.perf_counter()
        H.hswa_tree_evict(tree, 64, 64)
        t["evict"].append(time.perf_counter() - t0)
        H.hswa_tree_destroy(tree)
        H.hswa_pool_destroy(pool)
    out = {k: float(np.median(v)) * 1e6 for k, v in t.items()}
    out["follow_up_hits"] = hits
    out["requests"] = n_req
    out["nodes"] = nodes
    return out


def measure_transfer(steps, fp8=False, w=None):
    import torch
    w = w or wl.swa_transfer()
    tb = SwaTransfer(w, fp8=fp8)
    moved = tb.moved_bytes() * len(w.layer_kinds)
    # warm-up round trip
    tb.gather_all()
    tb.evict_and_restore()
    tb.scatter_all()
    tb.stream.synchronize()
    g_s = s_s = 0.0
    for _ in range(steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(tb.stream)
        tb.gather_all()
        e[1].record(tb.stream)
        tb.stream.synchronize()
        tb.evict_and_restore()
        e[2].record(tb.stream)
        tb.scatter_all()
        e[3].record(tb.stream)
        tb.stream.synchronize()
        g_s += e[0].elapsed_time(e[1]) / 1e3
        s_s += e[2].elapsed_time(e[3]) / 1e3
    # the host-link ceiling: a copy-engine memcpy of one layer's packed bytes,
    # two warm-up copies each way, then the median of seven timed copies
    one = tb.host[0].numel()
    dev = torch.empty(one, dtype=tb.host[0].dtype, device="cuda")
    nbytes = one * dev.element_size()
    link = {}
    with torch.cuda.stream(tb.stream):
        for name, dst, src in (("d2h", tb.host[1], dev), ("h2d", dev, tb.host[1])):
            for _ in range(2):
                dst.copy_(src, non_blocking=True)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
            ev[0].record(tb.stream)
            for k in range(7):
                dst.copy_(src, non_blocking=True)
                ev[k + 1].record(tb.stream)
            tb.stream.synchronize()
            link[name] = float(np.median([nbytes / (ev[k].elapsed_time(ev[k + 1]) / 1e3) / 1e9 for k in range(7)]))
    d2h, h2d = link["d2h"], link["h2d"]
    del dev
    rel_times, live = tb.release_rounds()
    st = tb.sess.check()
    if st != 0:
        raise RuntimeError("device status %d after transfer" % st)
    full_len = sum(w.cached) * 2 * w.n_kv_heads * w.head_dim * KV_ROW[w.dtype] * len(w.layer_kinds)
    out = {"gather_gbs": moved * steps / g_s / 1e9, "scatter_gbs": moved * steps / s_s / 1e9,
           "bytes_each_way": moved, "bytes_if_full_sequences": full_len,
           "release_us_per_call": 1e6 * float(np.median(rel_times)),
           "max_live_swa_pages_per_seq_after_release": max(live), "launches": tb.launches,
           "memcpy_d2h_gbs": d2h, "memcpy_h2d_gbs": h2d}
    del tb
    torch.cuda.empty_cache()
    return out


def run_transfer_line(args, world, rank, local):
    """--workload swa_transfer: one line whose value is the gather's GB/s into
    pinned host memory (the 60-layer in-window transfer; --seqs cuts it to a
    small profiling case)."""
    w = workload(args, "swa_transfer")
    t = measure_transfer(max(1, args.steps), fp8=args.fp8_pools, w=w)
    return {
        "metric": "Hybrid-SWA attn: SWA-mask transfer GB/s into pinned host memory",
        "value": round(t["gather_gbs"], 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": 1, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8" if args.fp8_pools else "bf16", "data": "synthetic",
        "config": {"workload": "swa_transfer", "seqs": len(w.cached), "layers": len(w.layer_kinds),
                   "window": w.window, "gb_each_way": round(t["bytes_each_way"] / 1e9, 3)},
        "scatter_gbs": round(t["scatter_gbs"], 2), "memcpy_d2h_gbs": round(t["memcpy_d2h_gbs"], 2),
        "memcpy_h2d_gbs": round(t["memcpy_h2d_gbs"], 2), "gpu_launches": t["launches"],
    }


def run_prefill_line(args, world, rank, local):
    """--workload chunked_prefill: one line whose value is the chunk's TFLOP/s."""
    w = workload(args, "chunked_prefill")
    _, bf16, bf16_sus, kind = peaks()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    barrier(world)
    pf = measure_prefill(args.steps, args.warmup, w)
    clock_info = clocks.stop()
    secs = max_over_ranks(pf["ms_per_step"] * args.steps / 1e3, world)
    total = sum_over_ranks(pf["valid_tflop_per_step"] * args.steps, world)
    value = total / secs
    return {
        "metric": "Hybrid-SWA attn: decode HBM GB/s and prefill TFLOP/s (% of GB300 peak)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "chunked_prefill", "seqs": len(w.cached), "prefix": "uniform[8192,65536] seed 3",
                   "chunk": w.n_new, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
                   "page": w.page_size, "window": w.window, "layers": "1 Full + 1 SWA",
                   "l2": "inputs larger than L2", "flops": "4 d Hq per valid (query, key) pair"},
        "roofline": {"bound": "tensor", "achieved": round(pf["full_tflops"], 1), "peak": bf16,
                     "unit": "TFLOP/s", "frac": round(pf["full_tflops"] / bf16, 4), "traffic": None,
                     "kernel": pf["kernel"] + " (Full layer)", "peak_source": kind + " burst",
                     "frac_of_sustained": round(pf["full_tflops"] / bf16_sus, 4)},
        "swa_layer_tflops": round(pf["swa_tflops"], 2), "swa_layer_exec_tflops": round(pf["swa_exec_tflops"], 2),
        "swa_kernel": pf["swa_kernel"],
        "gpu_launches": 4 * args.steps,
        "clocks": clock_info,
        "tokens_per_s": round(world * pf["tokens_per_s"], 1),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="hswa", choices=["hswa", "reference"])
    ap.add_argument("--workload", default="decode_batch", choices=["decode_batch", "chunked_prefill", "swa_transfer"])
    ap.add_argument("--fp8-pools", action="store_true", help="swa_transfer over FP8 pools")
    ap.add_argument("--seqs", type=int, default=0, help="use only the first N sequences (small profiling case)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-multi", action="store_true")
    ap.add_argument("--no-hybrid70", action="store_true")
    ap.add_argument("--no-transfer", action="store_true")
    ap.add_argument("--no-tree", action="store_true")
    ap.add_argument("--hybrid-steps", type=int, default=5)
    ap.add_argument("--breakdown", action="store_true", help="per-call device times of the decode step")
    ap.add_argument("--prefill-steps", type=int, default=5)
    args = ap.parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    world, rank, local = dist_setup(args)
    if args.workload == "chunked_prefill":
        line = run_prefill_line(args, world, rank, local)
    elif args.workload == "swa_transfer":
        line = run_transfer_line(args, world, rank, local)
    else:
        line = run_decode(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
