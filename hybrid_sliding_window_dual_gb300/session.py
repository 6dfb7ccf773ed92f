"""PyTorch-side plumbing around the C ABI: device memory for the layer pools,
the block tables and the decode workspace, and the stream to enqueue on.

No attention arithmetic happens here; every step calls a libhswa entry point.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as B

_TORCH_DTYPE = {B.HSWA_DTYPE_F32: torch.float32, B.HSWA_DTYPE_BF16: torch.bfloat16,
                B.HSWA_DTYPE_FP8_E4M3: torch.uint8}


class DualPoolSession:
    """A dual pool on one GPU: host bookkeeping (libhswa) + device buffers.

    ``layer_kinds`` lists HSWA_KIND_FULL / HSWA_KIND_SWA per layer; each
    layer gets its own K and V pool tensors unless ``share_full_pool`` is set,
    in which case all Full layers read one physical Full pool (used where the
    per-layer Full pools would not fit in HBM; the bytes each layer reads are
    the same).
    """

    def __init__(self, config: B.Config, layer_kinds, full_free_order=None, swa_free_order=None,
                 device="cuda", share_full_pool=False, stream=None, init="zeros"):
        self.cfg = config
        self.device = torch.device(device)
        self.stream = stream
        self.pool = B.hswa_pool_create(config, full_free_order, swa_free_order)
        self.dtype = _TORCH_DTYPE[config.dtype]
        rows = (config.max_seqs, config.max_pages_per_seq)
        self.d_full_bt = torch.full(rows, -1, dtype=torch.int32, device=self.device)
        self.d_swa_bt = torch.full(rows, -1, dtype=torch.int32, device=self.device)
        self.d_seq_len = torch.zeros(config.max_seqs, dtype=torch.int32, device=self.device)
        self.kinds = list(layer_kinds)
        self.k, self.v, self.ks, self.vs, self.layers = [], [], [], [], []
        self.fp8 = config.dtype == B.HSWA_DTYPE_FP8_E4M3
        shared = None
        for kind in self.kinds:
            pages = config.full_pages if kind == B.HSWA_KIND_FULL else config.swa_pages
            P, d, hkv = config.page_size, config.head_dim, config.n_kv_heads
            shape = (pages, hkv, P, d)
            if kind == B.HSWA_KIND_FULL and share_full_pool and shared is not None:
                k, v, ks, vs = shared
            else:
                alloc = torch.zeros if init == "zeros" else torch.empty
                k = alloc(shape, dtype=self.dtype, device=self.device)
                # FP8 pools keep each page of V transposed, [d][P], plus fp32
                # scales per (token, kv head, 128-element tile)
                v = alloc((pages, hkv, d, P) if self.fp8 else shape, dtype=self.dtype, device=self.device)
                ks = vs = None
                if self.fp8:
                    ks = torch.ones((pages, hkv, P, d // 128), dtype=torch.float32, device=self.device)
                    vs = torch.ones_like(ks)
                if kind == B.HSWA_KIND_FULL and share_full_pool:
                    shared = (k, v, ks, vs)
            self.k.append(k)
            self.v.append(v)
            self.ks.append(ks)
            self.vs.append(vs)
            self.layers.append(B.Layer(kind=kind, window=config.window, k_pool=k.data_ptr(), v_pool=v.data_ptr(),
                                       k_scale=ks.data_ptr() if ks is not None else None,
                                       v_scale=vs.data_ptr() if vs is not None else None))
        self.ws = None
        self.prefill_ws = None
        self.tree = None

    def close(self):
        if self.pool:
            if self.tree:
                B.hswa_tree_destroy(self.tree)
                self.tree = None
            B.hswa_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -------------------------------------------------------- bookkeeping
    def reserve(self, seq_ids, n_new):
        return B.hswa_reserve(self.pool, seq_ids, n_new)

    def release(self, seq_ids):
        return B.hswa_swa_release(self.pool, seq_ids)

    def seq_free(self, seq_ids):
        B.hswa_seq_free(self.pool, seq_ids)

    def swa_drop(self, seq_ids):
        return B.hswa_swa_drop(self.pool, seq_ids)

    def swa_restore(self, seq_ids):
        return B.hswa_swa_restore(self.pool, seq_ids)

    # ------------------------------------------------ prefix cache (host)
    def prefix_tree(self):
        """The pool's SWA-aware prefix cache tree (created on first use)."""
        if self.tree is None:
            self.tree = B.hswa_tree_create(self.pool)
        return self.tree

    def match_prefix(self, tokens):
        """Window-safe hit: (pages m, Full pages, SWA pages, raw pages)."""
        return B.hswa_tree_match(self.prefix_tree(), tokens, self.cfg.max_pages_per_seq)

    def share_prefix(self, seq_id, full_pages, swa_pages):
        B.hswa_seq_share_prefix(self.pool, seq_id, full_pages, swa_pages)

    def store_prefix(self, seq_id, tokens):
        return B.hswa_tree_insert(self.prefix_tree(), seq_id, tokens)

    def evict(self, want_full, want_swa):
        return B.hswa_tree_evict(self.prefix_tree(), want_full, want_swa)

    def tables(self):
        return B.hswa_get_tables(self.pool, self.cfg)

    def sync(self):
        B.hswa_sync_tables(self.pool, self.d_full_bt, self.d_swa_bt, self.d_seq_len, self.stream)

    def bt(self, layer):
        return self.d_full_bt if self.kinds[layer] == B.HSWA_KIND_FULL else self.d_swa_bt

    # ------------------------------------------------------------ device
    def workspace(self, n_seqs, n_tok=1):
        need = B.hswa_decode_multi_workspace_size(self.pool, n_seqs, n_tok)
        if self.ws is None or self.ws.numel() < need:
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self.ws

    def append(self, layer, k, v, d_slots):
        B.hswa_append_kv(self.pool, self.layers[layer], k, v, d_slots, k.shape[0], self.stream)

    def decode(self, layer, q, o, n_seqs, scale):
        ws = self.workspace(n_seqs)
        B.hswa_decode(self.pool, self.layers[layer], q, o, self.bt(layer), self.d_seq_len, n_seqs, scale, ws,
                      ws.numel(), self.stream)

    def decode_append(self, layer, q, k_new, v_new, d_slots, o, n_seqs, scale):
        ws = self.workspace(n_seqs)
        B.hswa_decode_append(self.pool, self.layers[layer], q, k_new, v_new, d_slots, o, self.bt(layer),
                             self.d_seq_len, n_seqs, scale, ws, ws.numel(), self.stream)

    def decode_multi(self, layer, q, o, n_seqs, n_tok, scale):
        """n_tok query tokens per sequence (q, o: [n_seqs * n_tok, Hq, d])."""
        ws = self.workspace(n_seqs, n_tok)
        B.hswa_decode_multi(self.pool, self.layers[layer], q, o, self.bt(layer), self.d_seq_len, n_seqs, n_tok,
                            scale, ws, ws.numel(), self.stream)

    def prefill(self, layer, q, o, d_prefix_len, d_q_start, n_seqs, max_q_len, scale, prefix_host=None,
                q_start_host=None):
        """prefix_host / q_start_host: host copies of the device arrays; with
        them an FP8 pool's staging workspace is sized for this chunk exactly,
        without them for any chunk of n_seqs sequences of max_q_len rows."""
        if prefix_host is not None and q_start_host is not None:
            need = B.hswa_prefill_workspace_size_exact(self.pool, self.layers[layer], prefix_host, q_start_host)
        else:
            need = B.hswa_prefill_workspace_size(self.pool, self.layers[layer], n_seqs, max_q_len)
        ws = None
        if need:  # FP8 pools stage f16 copies of the pages the chunk reads (and of q)
            if self.prefill_ws is None or self.prefill_ws.numel() < need:
                self.prefill_ws = torch.empty(need, dtype=torch.uint8, device=self.device)
            ws = self.prefill_ws
        B.hswa_prefill_chunk_ws(self.pool, self.layers[layer], q, o, self.bt(layer), d_prefix_len, d_q_start,
                                n_seqs, q.shape[0], max_q_len, scale, ws, need, self.stream)

    def window_offsets(self, layer, n_seqs, seq_len=None):
        """Packed-buffer token offsets [n_seqs + 1] (host int64) and the
        buffer's bytes, from the library (seq_len None: current lengths)."""
        return B.hswa_swa_window_offsets(self.pool, self.layers[layer], n_seqs, seq_len)

    def gather(self, layer, d_tok_offset, n_seqs, dst):
        B.hswa_swa_gather(self.pool, self.layers[layer], self.d_swa_bt, self.d_seq_len, d_tok_offset, n_seqs,
                          dst, self.stream)

    def scatter(self, layer, d_tok_offset, n_seqs, src):
        B.hswa_swa_scatter(self.pool, self.layers[layer], self.d_swa_bt, self.d_seq_len, d_tok_offset, n_seqs,
                           src, self.stream)

    def reload_async(self, layer_ids, d_seq_len, d_tok_offset, n_seqs, host_bufs, stream):
        """Reload offloaded SWA windows layer by layer with the scatter kernel
        reading pinned host memory directly, on a side stream; one event per
        layer ({layer: event}) for the compute stream to wait on."""
        events = {}
        with torch.cuda.stream(stream):
            for ly, buf in zip(layer_ids, host_bufs):
                B.hswa_swa_scatter(self.pool, self.layers[ly], self.d_swa_bt, d_seq_len, d_tok_offset, n_seqs,
                                   buf, stream)
                ev = torch.cuda.Event()
                ev.record(stream)
                events[ly] = ev
        return events

    def check(self):
        return B.hswa_check(self.stream)


class LayerwiseReload:
    """Layer-by-layer reload of offloaded SWA windows, overlapped with the
    attention of earlier layers ("MiMo-V2.5 Series Inference Full-Link
    Optimization", Sec. 2.1, asynchronous layer-by-layer pulling).

    The copy engines move each layer's packed window from pinned host memory
    into one of ``n_staging`` device staging buffers on ``copy_stream``; right
    before an SWA layer's attention, ``before_layer`` makes the compute stream
    wait for that copy and scatters the window from staging into the layer's
    pool pages (hswa_swa_scatter, device to device). The copy stream runs
    ``n_staging`` layers ahead; a staging buffer is refilled only after its
    scatter has run. ``d_seq_len`` is the lengths the windows were gathered at
    (a snapshot), so the step's own reserve may change the live lengths.
    """

    def __init__(self, sess, layer_ids, d_seq_len, d_tok_offset, n_seqs, host_bufs, copy_stream, staging):
        self.sess, self.layers = sess, list(layer_ids)
        self.d_seq_len, self.d_off, self.n = d_seq_len, d_tok_offset, n_seqs
        self.host, self.copy, self.staging = list(host_bufs), copy_stream, list(staging)
        self.copied = {}
        self.free = [None] * len(self.staging)
        self.next = 0

    def _enqueue_copy(self):
        k = self.next
        if k >= len(self.layers):
            return
        slot = k % len(self.staging)
        with torch.cuda.stream(self.copy):
            if self.free[slot] is not None:
                self.copy.wait_event(self.free[slot])
            n = self.host[k].numel()
            self.staging[slot][:n].copy_(self.host[k], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(self.copy)
            self.copied[self.layers[k]] = (ev, slot, n)
        self.next += 1

    def start(self, compute_stream):
        """Enqueue the first copies (after the work already on compute_stream)."""
        self.copy.wait_stream(compute_stream)
        for _ in range(len(self.staging)):
            self._enqueue_copy()

    def before_layer(self, layer, compute_stream):
        """Call before enqueueing `layer`'s attention on compute_stream."""
        if layer not in self.copied:
            return
        ev, slot, n = self.copied.pop(layer)
        with torch.cuda.stream(compute_stream):
            compute_stream.wait_event(ev)
            B.hswa_swa_scatter(self.sess.pool, self.sess.layers[layer], self.sess.d_swa_bt, self.d_seq_len,
                               self.d_off, self.n, self.staging[slot][:n], compute_stream)
            free = torch.cuda.Event()
            free.record(compute_stream)
            self.free[slot] = free
        self._enqueue_copy()
