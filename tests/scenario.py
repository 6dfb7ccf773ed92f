"""Test harness: one dual-pool scenario driven through both the CUDA library
(via the torch session) and the CPU oracle with the same call sequence.

Inputs come only from hswa_workloads (seeded). Expected values come only
from the oracle. Device results are compared against them.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import hswa_workloads as wl
import oracle
import hybrid_sliding_window_dual_gb300 as H
from hybrid_sliding_window_dual_gb300.session import DualPoolSession

TOL = {wl.DTYPE_BF16: 2e-2, wl.DTYPE_F32: 1e-5}


def raw_host(t):
    """CPU copy of a device tensor as numpy (bf16 -> raw uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def fill_normal_(t, seed, chunk=1 << 26):
    """Fill a device tensor with seeded N(0,1) values (chunked draws)."""
    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed))
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=g, device=t.device, dtype=torch.float32).to(t.dtype)


class Scenario:
    def __init__(self, hq, hkv, d, P, W, dtype, cached, layer_kinds=(0, 1), seed=0, full_pages=None,
                 swa_pages=None, max_pages=None, permute=True, chunk=4096, extra_tokens=64,
                 share_full_pool=False):
        self.hq, self.hkv, self.d, self.P, self.W, self.dtype = hq, hkv, d, P, W, dtype
        self.cached = list(cached)
        S = len(self.cached)
        need_full = sum(math.ceil((L + extra_tokens) / P) for L in self.cached) + 4
        if max_pages is None:
            max_pages = max(math.ceil((L + extra_tokens) / P) for L in self.cached) + 1
        if full_pages is None:
            full_pages = need_full
        if swa_pages is None:
            swa_pages = S * (math.ceil((W + max(chunk, extra_tokens)) / P) + 2) + 4
        self.cfg = H.Config(window=W, page_size=P, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, dtype=dtype,
                            full_pages=full_pages, swa_pages=swa_pages, max_seqs=S, max_pages_per_seq=max_pages)
        fo = wl.permutation(full_pages, seed) if permute else None
        so = wl.permutation(swa_pages, seed + 1) if permute else None
        self.sess = DualPoolSession(self.cfg, layer_kinds, fo, so, share_full_pool=share_full_pool)
        self.ora = oracle.DualPool(W, P, full_pages, swa_pages, S, max_pages, fo, so)
        self.kinds = list(layer_kinds)
        self.seed = seed
        # cached state: chunked prefill of every sequence with a release per chunk
        for s, L in enumerate(self.cached):
            for start in range(0, L, chunk):
                n = min(chunk, L - start)
                self.reserve([s], [n])
                self.release([s])
        self.assert_tables_equal()
        self.sess.sync()
        for i in range(len(self.kinds)):
            if share_full_pool and self.kinds[i] == 0 and i != self.kinds.index(0):
                continue
            fill_normal_(self.sess.k[i], seed * 1000 + 2 * i)
            fill_normal_(self.sess.v[i], seed * 1000 + 2 * i + 1)
        torch.cuda.synchronize()
        self.scale = 1.0 / math.sqrt(d)

    # --------------------------------------------------------- bookkeeping
    def reserve(self, seq_ids, n_new):
        got = self.sess.reserve(seq_ids, n_new)
        exp = self.ora.reserve(seq_ids, n_new)
        assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1]), "slot mapping differs"
        return got

    def release(self, seq_ids):
        a = self.sess.release(seq_ids)
        b = self.ora.swa_release(seq_ids)
        assert a == b
        return a

    def assert_tables_equal(self, device=False):
        f, s, lens = self.sess.tables()
        assert np.array_equal(f, self.ora.full_bt) and np.array_equal(s, self.ora.swa_bt)
        assert np.array_equal(lens.astype(np.int64), self.ora.seq_len)
        if device:
            assert np.array_equal(self.sess.d_full_bt.cpu().numpy(), self.ora.full_bt)
            assert np.array_equal(self.sess.d_swa_bt.cpu().numpy(), self.ora.swa_bt)
            assert np.array_equal(self.sess.d_seq_len.cpu().numpy().astype(np.int64), self.ora.seq_len)

    def table(self, layer):
        return self.ora.full_bt if self.kinds[layer] == 0 else self.ora.swa_bt

    def window(self, layer):
        return 0 if self.kinds[layer] == 0 else self.W

    # ---------------------------------------------------------- snapshots
    def snapshot(self, layer, seqs):
        """Host copy of the pages the given sequences reference in the layer's
        pool, with the table rows remapped onto the compact copy."""
        bt = self.table(layer)[seqs]
        pages = np.unique(bt[bt >= 0])
        remap = np.full(max(int(pages.max()) + 1 if pages.size else 1, 1), -1, np.int64)
        remap[pages] = np.arange(pages.size)
        new_bt = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
        idx = torch.as_tensor(pages, device=self.sess.device, dtype=torch.long)
        k = raw_host(self.sess.k[layer].index_select(0, idx))
        v = raw_host(self.sess.v[layer].index_select(0, idx))
        return k, v, new_bt, pages

    @staticmethod
    def oracle_append(snap, slots, new, P):
        """Write new rows into a snapshot through the oracle's append."""
        k, v, new_bt, pages = snap
        pos = {int(p): i for i, p in enumerate(pages)}
        local = np.array([pos.get(int(s) // P, -1) * P + int(s) % P if int(s) // P in pos else -1
                          for s in slots], np.int64)
        oracle.append_kv(k, new[0], local)
        oracle.append_kv(v, new[1], local)

    def gen(self, shape, seed):
        return wl.normal(shape, seed, self.dtype)

    def to_dev(self, x):
        return x.to(self.sess.device)


def window_offsets(sess, layer, lens, W):
    """The library's packed-buffer token offsets and byte count for these
    lengths (hswa_swa_window_offsets), with the offsets checked against the
    oracle's in-window counts."""
    lens = np.asarray(lens, np.int64)
    off, nbytes = sess.window_offsets(layer, len(lens), lens.astype(np.int32))
    assert np.array_equal(off, oracle.swa_window_counts(lens, W)[1])
    return off, nbytes


def prefill_kernel(kind, window, fp8=False):
    """Name hswa_last_kernel reports after a tensor-core prefill of this
    layer kind: SWA layers with W <= 128 run the persistent window kernel."""
    name = "prefill_swa_tc_d128" if kind == wl.KIND_SWA and 0 < window <= 128 else "prefill_tc_bf16_d128"
    return "prefill_stage_fp8+%s<f16>" % name if fp8 else name


def max_err(got, exp):
    return float(np.abs(got.astype(np.float64) - exp).max()) if exp.size else 0.0


def device_out(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
