"""CPU oracle for Hybrid-SWA attention over a dual KV pool.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and
bench.py's cpu_baseline / reference leg import this package. It shares no
code with the CUDA library (``hybrid_sliding_window_dual_gb300``) and never
imports it.

* ``attention``  -- float64 paged Full / SWA GQA attention (hswa_oracle.c)
* ``append_kv``  -- slot-mapped write of new K/V rows into a pool
* ``swa_pack`` / ``swa_unpack`` -- transfer of in-window SWA tokens only
* ``pool.DualPool`` -- dual-pool bookkeeping (reserve, release, ...)

Source: "MiMo-V2.5 Series Inference Full-Link Optimization" Sec. 1.1 and
Sec. 2.1; "Tiered KV Cache Offloading in vLLM", hybrid-model support
(sliding-window layers move only the tokens inside their window).

Parity status: every function here is pinned by tests/test_oracle.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .pool import DualPool, NoSpace  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hswa_oracle.c")
_OUT = os.path.join(_HERE, "_build", "libhswa_oracle.so")
_lib = None


def build(force=False):
    """Compile the C oracle with gcc (plain -O2, OpenMP, no fast-math)."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _OUT)
    return _OUT


def load_library(path):
    """ctypes handle on a compiled oracle library (the default one, or a
    test-built variant of the same source)."""
    lib = ctypes.CDLL(path)
    lib.hswa_oracle_attention.restype = ctypes.c_int
    lib.hswa_oracle_attention.argtypes = [
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    lib.hswa_oracle_threads.restype = ctypes.c_int
    lib.hswa_oracle_attention_fp8.restype = ctypes.c_int
    lib.hswa_oracle_attention_fp8.argtypes = [
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def threads():
    return _load().hswa_oracle_threads()


def _raw(x):
    """numpy view of a CPU array/tensor: (contiguous array, dtype code)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), 1
            if x.dtype == torch.float32:
                return x.numpy(), 0
            raise TypeError("oracle inputs are fp32 or bf16, got %s" % x.dtype)
    except ImportError:
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, 0
    if x.dtype == np.uint16:
        return x, 1
    raise TypeError("oracle inputs are float32 or raw bf16 (uint16), got %s" % x.dtype)


def attention(q, k_pool, v_pool, block_table, q_seq, q_pos, window, scale, lib=None):
    """float64 attention for each query row.

    q: [nq, Hq, d]; k_pool, v_pool: [pages, Hkv, P, d] (same dtype as q);
    block_table: int32 [rows, max_pages]; q_seq[i]: table row of query i;
    q_pos[i]: its position t; window: W (SWA layer) or 0 (Full layer).
    Returns float64 [nq, Hq, d].
    """
    qa, dt = _raw(q)
    ka, dk = _raw(k_pool)
    va, dv = _raw(v_pool)
    assert dt == dk == dv, "q, k and v must share a dtype"
    nq, hq, d = qa.shape
    pages, hkv, P, d2 = ka.shape
    assert d2 == d and va.shape == ka.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    qs = np.ascontiguousarray(q_seq, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    assert qs.shape == (nq,) and qp.shape == (nq,)
    out = np.zeros((nq, hq, d), np.float64)
    rc = (lib or _load()).hswa_oracle_attention(
        nq, qs.ctypes.data, qp.ctypes.data, hq, hkv, d, P, int(window), float(scale), dt,
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, pages, bt.ctypes.data,
        bt.shape[1], out.ctypes.data)
    if rc == -1:
        raise IndexError("a key's block-table entry is not a live page")
    if rc != 0:
        raise ValueError("bad attention sizes")
    return out


def attention_fp8(q, k_codes, k_scale, v_codes, v_scale, block_table, q_seq, q_pos, window, scale,
                  lib=None):
    """float64 attention over an FP8 pool (exact dequantization).

    k_codes: uint8 [pages, Hkv, P, d]; v_codes: uint8 [pages, Hkv, d, P]
    (pages stored transposed); k_scale, v_scale: float32 [pages, Hkv, P, d/128].
    q: [nq, Hq, d] fp32 or bf16. Returns float64 [nq, Hq, d]."""
    qa, dt = _raw(q)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    nq, hq, d = qa.shape
    pages, hkv, P, d2 = kc.shape
    assert d2 == d and vc.shape == (pages, hkv, d, P) and ks.shape == (pages, hkv, P, d // 128)
    assert vs.shape == ks.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    qs = np.ascontiguousarray(q_seq, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    out = np.zeros((nq, hq, d), np.float64)
    rc = (lib or _load()).hswa_oracle_attention_fp8(
        nq, qs.ctypes.data, qp.ctypes.data, hq, hkv, d, P, int(window), float(scale), dt, qa.ctypes.data,
        kc.ctypes.data, ks.ctypes.data, vc.ctypes.data, vs.ctypes.data, pages, bt.ctypes.data, bt.shape[1],
        out.ctypes.data)
    if rc == -1:
        raise IndexError("a key's block-table entry is not a live page")
    if rc != 0:
        raise ValueError("bad attention sizes")
    return out


def append_kv_fp8(k_codes, k_scale, v_codes, v_scale, k_new, v_new, slots):
    """Quantize new K/V rows ([T, Hkv, d] fp32 values) per 128-element tile
    and write them at their slots: K row-major, V into the transposed page."""
    from .fp8 import quantize_tiles
    P = k_codes.shape[2]
    kq, ks = quantize_tiles(k_new)
    vq, vs = quantize_tiles(v_new)
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        page, row = slot // P, slot % P
        k_codes[page, :, row, :] = kq[t]
        k_scale[page, :, row, :] = ks[t]
        v_codes[page, :, :, row] = vq[t]
        v_scale[page, :, row, :] = vs[t]


def append_kv(pool, new, slots):
    """pool[slot // P, :, slot % P, :] = new[t] for every token t (slot -1 skipped).

    pool: numpy [pages, Hkv, P, d]; new: [T, Hkv, d]; returns nothing."""
    P = pool.shape[2]
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        pool[slot // P, :, slot % P, :] = new[t]


def swa_window_counts(seq_len, window):
    """n_s = min(L_s, W) in-window tokens per sequence, and their prefix sum."""
    n = np.minimum(np.asarray(seq_len, np.int64), window)
    off = np.zeros(len(n) + 1, np.int64)
    off[1:] = np.cumsum(n)
    return n, off


def swa_pack(k_pool, v_pool, swa_bt, seq_len, window):
    """Pack the in-window tokens of sequences 0..n-1 of one SWA layer.

    For each sequence s in order, n_s = min(L_s, W) tokens at positions
    [L_s - n_s, L_s): a K block [Hkv][n_s][d] followed by a V block
    [Hkv][n_s][d]. Returns a flat array of the pool's element type.
    """
    P = k_pool.shape[2]
    hkv, d = k_pool.shape[1], k_pool.shape[3]
    n, off = swa_window_counts(seq_len, window)
    out = np.zeros(int(off[-1]) * 2 * hkv * d, k_pool.dtype)
    for s in range(len(n)):
        L = int(seq_len[s])
        base = int(off[s]) * 2 * hkv * d
        ns = int(n[s])
        for which, pool in ((0, k_pool), (1, v_pool)):
            block = np.zeros((hkv, ns, d), pool.dtype)
            for i, t in enumerate(range(L - ns, L)):
                page = int(swa_bt[s, t // P])
                if page < 0:
                    raise IndexError("in-window token without an SWA page")
                block[:, i, :] = pool[page, :, t % P, :]
            start = base + which * hkv * ns * d
            out[start:start + hkv * ns * d] = block.reshape(-1)
    return out


def swa_unpack(packed, k_pool, v_pool, swa_bt, seq_len, window):
    """Inverse of swa_pack: write the packed tokens back into the pools."""
    P = k_pool.shape[2]
    hkv, d = k_pool.shape[1], k_pool.shape[3]
    n, off = swa_window_counts(seq_len, window)
    for s in range(len(n)):
        L = int(seq_len[s])
        base = int(off[s]) * 2 * hkv * d
        ns = int(n[s])
        for which, pool in ((0, k_pool), (1, v_pool)):
            start = base + which * hkv * ns * d
            block = packed[start:start + hkv * ns * d].reshape(hkv, ns, d)
            for i, t in enumerate(range(L - ns, L)):
                page = int(swa_bt[s, t // P])
                if page < 0:
                    raise IndexError("in-window token without an SWA page")
                pool[page, :, t % P, :] = block[:, i, :]


def swa_pack_fp8(k_codes, k_scale, v_codes, v_scale, swa_bt, seq_len, window):
    """Pack the in-window tokens of sequences 0..n-1 of one SWA layer over
    FP8 pools ("Baidu AI Cloud: Day-0 support for hybrid-architecture LLMs",
    Optimization 2 item 2: codes with one scale per token, head and
    128-element tile; MiMo Sec. 2.1: only in-window data moves).

    Pools: k_codes [pages][Hkv][P][d] uint8, v_codes [pages][Hkv][d][P]
    (pages stored transposed), scales [pages][Hkv][P][d/128] float32 with
    d = 128. For each sequence s in order, n_s = min(L_s, W) tokens at
    positions [L_s - n_s, L_s), starting at byte 2 * Hkv * (d + 4) * (sum of
    the earlier n): K codes [Hkv][n_s][d], V codes [Hkv][n_s][d] (token rows,
    not transposed), K scales [Hkv][n_s] float32, V scales [Hkv][n_s]
    float32. Returns a flat uint8 array."""
    P, hkv, d = k_codes.shape[2], k_codes.shape[1], k_codes.shape[3]
    assert d == 128 and k_scale.shape[-1] == 1
    n, off = swa_window_counts(seq_len, window)
    out = np.zeros(int(off[-1]) * 2 * hkv * (d + 4), np.uint8)
    for s in range(len(n)):
        L, ns = int(seq_len[s]), int(n[s])
        kb = np.zeros((hkv, ns, d), np.uint8)
        vb = np.zeros((hkv, ns, d), np.uint8)
        kss = np.zeros((hkv, ns), np.float32)
        vss = np.zeros((hkv, ns), np.float32)
        for i, t in enumerate(range(L - ns, L)):
            page = int(swa_bt[s, t // P])
            if page < 0:
                raise IndexError("in-window token without an SWA page")
            row = t % P
            kb[:, i, :] = k_codes[page, :, row, :]
            vb[:, i, :] = v_codes[page, :, :, row]
            kss[:, i] = k_scale[page, :, row, 0]
            vss[:, i] = v_scale[page, :, row, 0]
        blob = np.concatenate([kb.reshape(-1), vb.reshape(-1), kss.reshape(-1).view(np.uint8),
                               vss.reshape(-1).view(np.uint8)])
        start = int(off[s]) * 2 * hkv * (d + 4)
        out[start:start + blob.size] = blob
    return out


def swa_unpack_fp8(packed, k_codes, k_scale, v_codes, v_scale, swa_bt, seq_len, window):
    """Inverse of swa_pack_fp8: write the packed tokens back into the pools."""
    P, hkv, d = k_codes.shape[2], k_codes.shape[1], k_codes.shape[3]
    n, off = swa_window_counts(seq_len, window)
    for s in range(len(n)):
        L, ns = int(seq_len[s]), int(n[s])
        start = int(off[s]) * 2 * hkv * (d + 4)
        c = hkv * ns * d
        kb = packed[start:start + c].reshape(hkv, ns, d)
        vb = packed[start + c:start + 2 * c].reshape(hkv, ns, d)
        kss = packed[start + 2 * c:start + 2 * c + 4 * hkv * ns].view(np.float32).reshape(hkv, ns)
        vss = packed[start + 2 * c + 4 * hkv * ns:start + 2 * c + 8 * hkv * ns].view(np.float32).reshape(hkv, ns)
        for i, t in enumerate(range(L - ns, L)):
            page = int(swa_bt[s, t // P])
            if page < 0:
                raise IndexError("in-window token without an SWA page")
            row = t % P
            k_codes[page, :, row, :] = kb[:, i, :]
            v_codes[page, :, :, row] = vb[:, i, :]
            k_scale[page, :, row, 0] = kss[:, i]
            v_scale[page, :, row, 0] = vss[:, i]


def kv_bytes(pool: DualPool, layer_kinds, seq_ids, kv_bytes_per_token):
    """KV bytes held by the dual pool for the given sequences (live pages),
    summed over layers: Full layers count Full pages, SWA layers SWA pages."""
    n_full = sum(1 for k in layer_kinds if k == 0)
    n_swa = len(layer_kinds) - n_full
    full = sum(pool.live_full_pages(s) for s in seq_ids)
    swa = sum(pool.live_swa_pages(s) for s in seq_ids)
    page_bytes = pool.P * kv_bytes_per_token
    return (n_full * full + n_swa * swa) * page_bytes
