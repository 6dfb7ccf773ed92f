"""ctypes binding of libhswa.so: one Python function per C entry point,
same names, argument marshalling only.

Device buffers are torch CUDA tensors (any object with ``data_ptr()``) or raw
integer addresses; host arrays are numpy arrays. Every non-zero status raises
``HswaError``. The library must have been built (``build.build()``); there is
no fallback: importing without it raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

HSWA_OK = 0
HSWA_ERR_INVALID_ARG = 1
HSWA_ERR_NO_SPACE = 2
HSWA_ERR_UNSUPPORTED = 3
HSWA_ERR_CUDA = 4
HSWA_ERR_TIMEOUT = 5
HSWA_ERR_BOUNDS = 6

HSWA_KIND_FULL = 0
HSWA_KIND_SWA = 1
HSWA_DTYPE_F32 = 0
HSWA_DTYPE_BF16 = 1
HSWA_DTYPE_FP8_E4M3 = 2
HSWA_DECODE_MAX_TOKENS = 16


class HswaError(RuntimeError):
    def __init__(self, status, call):
        self.status = status
        detail = ""
        if status == HSWA_ERR_CUDA:
            detail = " [%s]" % lib.hswa_last_cuda_error().decode()
        super().__init__("%s: %s (status %d)%s" % (call, status_string(status), status, detail))


class NoSpace(HswaError):
    pass


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "window", "page_size", "n_q_heads", "n_kv_heads", "head_dim", "dtype",
        "full_pages", "swa_pages", "max_seqs", "max_pages_per_seq")]


class Layer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SIG = {
    "hswa_pool_create": (_I, [ctypes.POINTER(Config), _P, _P, ctypes.POINTER(_P)]),
    "hswa_pool_destroy": (_I, [_P]),
    "hswa_reserve": (_I, [_P, _I, _P, _P, _P, _P]),
    "hswa_swa_release": (_I, [_P, _I, _P, _P]),
    "hswa_seq_free": (_I, [_P, _I, _P]),
    "hswa_swa_drop": (_I, [_P, _I, _P, _P]),
    "hswa_swa_restore": (_I, [_P, _I, _P, _P]),
    "hswa_get_tables": (_I, [_P, _P, _P, _P]),
    "hswa_get_free_list": (_I, [_P, _I, _P, ctypes.c_int32, _P]),
    "hswa_seq_share_prefix": (_I, [_P, ctypes.c_int32, ctypes.c_int32, _P, _P]),
    "hswa_get_page_refs": (_I, [_P, _I, _P, ctypes.c_int32]),
    "hswa_tree_create": (_I, [_P, ctypes.POINTER(_P)]),
    "hswa_tree_destroy": (_I, [_P]),
    "hswa_tree_match": (_I, [_P, _P, ctypes.c_int64, _P, _P, ctypes.c_int32, _P, _P]),
    "hswa_tree_insert": (_I, [_P, ctypes.c_int32, _P, ctypes.c_int64, _P]),
    "hswa_tree_evict": (_I, [_P, ctypes.c_int32, ctypes.c_int32, _P, _P]),
    "hswa_tree_stats": (_I, [_P, _P, _P, _P]),
    "hswa_tree_nodes": (_I, [_P, _P, ctypes.c_int32, _P]),
    "hswa_sync_tables": (_I, [_P, _P, _P, _P, _P]),
    "hswa_append_kv": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _I, _P]),
    "hswa_decode_workspace_size": (ctypes.c_size_t, [_P, _I]),
    "hswa_decode": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _P, _I, ctypes.c_float, _P,
                         ctypes.c_size_t, _P]),
    "hswa_decode_append": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _P, _P, _P, _P, _I, ctypes.c_float, _P,
                                ctypes.c_size_t, _P]),
    "hswa_decode_noalloc": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _P, _I, ctypes.c_float, _P]),
    "hswa_decode_multi_workspace_size": (ctypes.c_size_t, [_P, _I, _I]),
    "hswa_decode_multi": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _P, _I, _I, ctypes.c_float, _P,
                               ctypes.c_size_t, _P]),
    "hswa_prefill_chunk": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _P, _P, _I, _I, _I,
                                ctypes.c_float, _P]),
    "hswa_prefill_workspace_size": (ctypes.c_size_t, [_P, ctypes.POINTER(Layer), _I, _I]),
    "hswa_prefill_workspace_size_exact": (ctypes.c_size_t, [_P, ctypes.POINTER(Layer), _I, _P, _P]),
    "hswa_prefill_chunk_ws": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _P, _P, _I, _I, _I,
                                   ctypes.c_float, _P, ctypes.c_size_t, _P]),
    "hswa_swa_window_offsets": (_I, [_P, ctypes.POINTER(Layer), _I, _P, _P, _P]),
    "hswa_swa_gather": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _I, _P, _P]),
    "hswa_swa_scatter": (_I, [_P, ctypes.POINTER(Layer), _P, _P, _P, _I, _P, _P]),
    "hswa_check": (_I, [_P]),
    "hswa_selftest_bounded_wait": (_I, [_P]),
    "hswa_last_kernel": (ctypes.c_char_p, []),
    "hswa_last_cuda_error": (ctypes.c_char_p, []),
    "hswa_status_string": (ctypes.c_char_p, [_I]),
}


def library_path():
    return _build.LIB


def _load():
    path = library_path()
    if not os.path.exists(path):
        raise ImportError("libhswa.so is not built (%s); run hybrid_sliding_window_dual_gb300.build.build()"
                          % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIG.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status):
    return lib.hswa_status_string(int(status)).decode()


def _check(status, call):
    if status == HSWA_ERR_NO_SPACE:
        raise NoSpace(status, call)
    if status != HSWA_OK:
        raise HswaError(status, call)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ------------------------------------------------------------- pool (host)
def hswa_pool_create(config: Config, full_free_order=None, swa_free_order=None):
    out = ctypes.c_void_p()
    f = None if full_free_order is None else _i32(full_free_order)
    s = None if swa_free_order is None else _i32(swa_free_order)
    _check(lib.hswa_pool_create(ctypes.byref(config), _ptr(f), _ptr(s), ctypes.byref(out)),
           "hswa_pool_create")
    return out.value


def hswa_pool_destroy(pool):
    _check(lib.hswa_pool_destroy(pool), "hswa_pool_destroy")


def hswa_reserve(pool, seq_ids, n_new):
    ids, n = _i32(seq_ids), _i32(n_new)
    total = max(int(n.sum()), 0) if n.size else 0
    full = np.empty(total, np.int32)
    swa = np.empty(total, np.int32)
    _check(lib.hswa_reserve(pool, len(ids), _ptr(ids), _ptr(n), _ptr(full), _ptr(swa)), "hswa_reserve")
    return full, swa


def _count_call(name, pool, seq_ids):
    ids = _i32(seq_ids)
    out = ctypes.c_int32()
    _check(getattr(lib, name)(pool, len(ids), _ptr(ids), ctypes.addressof(out)), name)
    return out.value


def hswa_swa_release(pool, seq_ids):
    return _count_call("hswa_swa_release", pool, seq_ids)


def hswa_swa_drop(pool, seq_ids):
    return _count_call("hswa_swa_drop", pool, seq_ids)


def hswa_swa_restore(pool, seq_ids):
    return _count_call("hswa_swa_restore", pool, seq_ids)


def hswa_seq_free(pool, seq_ids):
    ids = _i32(seq_ids)
    _check(lib.hswa_seq_free(pool, len(ids), _ptr(ids)), "hswa_seq_free")


def hswa_get_tables(pool, config: Config):
    full = np.empty((config.max_seqs, config.max_pages_per_seq), np.int32)
    swa = np.empty_like(full)
    lens = np.empty(config.max_seqs, np.int32)
    _check(lib.hswa_get_tables(pool, _ptr(full), _ptr(swa), _ptr(lens)), "hswa_get_tables")
    return full, swa, lens


def hswa_get_free_list(pool, kind):
    count = ctypes.c_int32()
    _check(lib.hswa_get_free_list(pool, kind, None, 0, ctypes.addressof(count)), "hswa_get_free_list")
    out = np.empty(count.value, np.int32)
    _check(lib.hswa_get_free_list(pool, kind, _ptr(out), count.value, ctypes.addressof(count)),
           "hswa_get_free_list")
    return out


# ------------------------------------------------------ prefix tree
def hswa_seq_share_prefix(pool, seq_id, full_pages, swa_pages):
    f, w = _i32(full_pages), _i32(swa_pages)
    _check(lib.hswa_seq_share_prefix(pool, int(seq_id), len(f), _ptr(f), _ptr(w)), "hswa_seq_share_prefix")


def hswa_get_page_refs(pool, kind, n_pages):
    out = np.empty(int(n_pages), np.int32)
    _check(lib.hswa_get_page_refs(pool, kind, _ptr(out), len(out)), "hswa_get_page_refs")
    return out


def hswa_tree_create(pool):
    out = ctypes.c_void_p()
    _check(lib.hswa_tree_create(pool, ctypes.byref(out)), "hswa_tree_create")
    return out.value


def hswa_tree_destroy(tree):
    _check(lib.hswa_tree_destroy(tree), "hswa_tree_destroy")


def hswa_tree_match(tree, tokens, cap_pages):
    """(m, full_pages[:m], swa_pages[:m], raw_pages)."""
    t = _i32(tokens)
    full = np.empty(max(int(cap_pages), 0), np.int32)
    swa = np.empty_like(full)
    m, raw = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.hswa_tree_match(tree, _ptr(t), len(t), _ptr(full), _ptr(swa), len(full), ctypes.addressof(m),
                               ctypes.addressof(raw)), "hswa_tree_match")
    return m.value, full[:m.value].copy(), swa[:m.value].copy(), raw.value


def hswa_tree_insert(tree, seq_id, tokens):
    t = _i32(tokens)
    n = ctypes.c_int32()
    _check(lib.hswa_tree_insert(tree, int(seq_id), _ptr(t), len(t), ctypes.addressof(n)), "hswa_tree_insert")
    return n.value


def hswa_tree_evict(tree, want_full, want_swa):
    ff, fs = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.hswa_tree_evict(tree, int(want_full), int(want_swa), ctypes.addressof(ff), ctypes.addressof(fs)),
           "hswa_tree_evict")
    return ff.value, fs.value


def hswa_tree_stats(tree):
    a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib.hswa_tree_stats(tree, ctypes.addressof(a), ctypes.addressof(b), ctypes.addressof(c)),
           "hswa_tree_stats")
    return a.value, b.value, c.value


def hswa_tree_nodes(tree):
    """[n_nodes, 5] int32: id, parent id (-1 = root), logical page, Full page, SWA page."""
    count = ctypes.c_int32()
    _check(lib.hswa_tree_nodes(tree, None, 0, ctypes.addressof(count)), "hswa_tree_nodes")
    out = np.empty((count.value, 5), np.int32)
    _check(lib.hswa_tree_nodes(tree, _ptr(out), out.size, ctypes.addressof(count)), "hswa_tree_nodes")
    return out


# --------------------------------------------------------------- device
def hswa_sync_tables(pool, d_full_bt, d_swa_bt, d_seq_len, stream=None):
    _check(lib.hswa_sync_tables(pool, _ptr(d_full_bt), _ptr(d_swa_bt), _ptr(d_seq_len), _stream(stream)),
           "hswa_sync_tables")


def hswa_append_kv(pool, layer: Layer, k, v, d_slots, n_tokens, stream=None):
    _check(lib.hswa_append_kv(pool, ctypes.byref(layer), _ptr(k), _ptr(v), _ptr(d_slots), int(n_tokens),
                              _stream(stream)), "hswa_append_kv")


def hswa_decode_workspace_size(pool, n_seqs):
    return int(lib.hswa_decode_workspace_size(pool, int(n_seqs)))


def hswa_decode(pool, layer: Layer, q, o, d_bt, d_seq_len, n_seqs, scale, ws, ws_bytes, stream=None):
    _check(lib.hswa_decode(pool, ctypes.byref(layer), _ptr(q), _ptr(o), _ptr(d_bt), _ptr(d_seq_len),
                           int(n_seqs), float(scale), _ptr(ws), int(ws_bytes), _stream(stream)), "hswa_decode")


def hswa_decode_append(pool, layer: Layer, q, k_new, v_new, d_slots, o, d_bt, d_seq_len, n_seqs, scale, ws,
                       ws_bytes, stream=None):
    _check(lib.hswa_decode_append(pool, ctypes.byref(layer), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(d_slots),
                                  _ptr(o), _ptr(d_bt), _ptr(d_seq_len), int(n_seqs), float(scale), _ptr(ws),
                                  int(ws_bytes), _stream(stream)), "hswa_decode_append")


def hswa_decode_multi_workspace_size(pool, n_seqs, n_tok):
    return int(lib.hswa_decode_multi_workspace_size(pool, int(n_seqs), int(n_tok)))


def hswa_decode_multi(pool, layer: Layer, q, o, d_bt, d_seq_len, n_seqs, n_tok, scale, ws, ws_bytes, stream=None):
    _check(lib.hswa_decode_multi(pool, ctypes.byref(layer), _ptr(q), _ptr(o), _ptr(d_bt), _ptr(d_seq_len),
                                 int(n_seqs), int(n_tok), float(scale), _ptr(ws), int(ws_bytes), _stream(stream)),
           "hswa_decode_multi")


def hswa_decode_noalloc(pool, layer: Layer, q, o, d_bt, d_seq_len, n_seqs, scale, stream=None):
    _check(lib.hswa_decode_noalloc(pool, ctypes.byref(layer), _ptr(q), _ptr(o), _ptr(d_bt), _ptr(d_seq_len),
                                   int(n_seqs), float(scale), _stream(stream)), "hswa_decode_noalloc")


def hswa_prefill_chunk(pool, layer: Layer, q, o, d_bt, d_prefix_len, d_q_start, n_seqs, total_q, max_q_len,
                       scale, stream=None):
    _check(lib.hswa_prefill_chunk(pool, ctypes.byref(layer), _ptr(q), _ptr(o), _ptr(d_bt), _ptr(d_prefix_len),
                                  _ptr(d_q_start), int(n_seqs), int(total_q), int(max_q_len), float(scale),
                                  _stream(stream)), "hswa_prefill_chunk")


def hswa_prefill_workspace_size(pool, layer: Layer, n_seqs, max_q_len):
    return int(lib.hswa_prefill_workspace_size(pool, ctypes.byref(layer), int(n_seqs), int(max_q_len)))


def hswa_prefill_workspace_size_exact(pool, layer: Layer, prefix_len, q_start):
    pre = np.ascontiguousarray(prefix_len, np.int32)
    qs = np.ascontiguousarray(q_start, np.int32)
    if qs.shape != (pre.size + 1,):
        raise ValueError("q_start must hold len(prefix_len) + 1 offsets")
    return int(lib.hswa_prefill_workspace_size_exact(pool, ctypes.byref(layer), int(pre.size), _ptr(pre), _ptr(qs)))


def hswa_prefill_chunk_ws(pool, layer: Layer, q, o, d_bt, d_prefix_len, d_q_start, n_seqs, total_q, max_q_len,
                          scale, ws, ws_bytes, stream=None):
    _check(lib.hswa_prefill_chunk_ws(pool, ctypes.byref(layer), _ptr(q), _ptr(o), _ptr(d_bt), _ptr(d_prefix_len),
                                     _ptr(d_q_start), int(n_seqs), int(total_q), int(max_q_len), float(scale),
                                     _ptr(ws), int(ws_bytes), _stream(stream)), "hswa_prefill_chunk_ws")


def hswa_swa_window_offsets(pool, layer: Layer, n_seqs, seq_len=None):
    """(tok_offset int64 [n_seqs + 1], packed bytes); seq_len None = the
    pool's current lengths."""
    out = np.empty(int(n_seqs) + 1, np.int64)
    nbytes = ctypes.c_size_t()
    lens = None if seq_len is None else np.ascontiguousarray(seq_len, np.int32)
    if lens is not None and lens.shape != (int(n_seqs),):
        raise ValueError("seq_len must hold n_seqs lengths")
    _check(lib.hswa_swa_window_offsets(pool, ctypes.byref(layer), int(n_seqs), _ptr(lens), _ptr(out),
                                       ctypes.addressof(nbytes)), "hswa_swa_window_offsets")
    return out, int(nbytes.value)


def hswa_swa_gather(pool, layer: Layer, d_swa_bt, d_seq_len, d_tok_offset, n_seqs, dst, stream=None):
    _check(lib.hswa_swa_gather(pool, ctypes.byref(layer), _ptr(d_swa_bt), _ptr(d_seq_len), _ptr(d_tok_offset),
                               int(n_seqs), _ptr(dst), _stream(stream)), "hswa_swa_gather")


def hswa_swa_scatter(pool, layer: Layer, d_swa_bt, d_seq_len, d_tok_offset, n_seqs, src, stream=None):
    _check(lib.hswa_swa_scatter(pool, ctypes.byref(layer), _ptr(d_swa_bt), _ptr(d_seq_len), _ptr(d_tok_offset),
                                int(n_seqs), _ptr(src), _stream(stream)), "hswa_swa_scatter")


def hswa_check(stream=None):
    """Wait for the stream and return the device status word (0 = clean)."""
    return int(lib.hswa_check(_stream(stream)))


def hswa_selftest_bounded_wait(stream=None):
    _check(lib.hswa_selftest_bounded_wait(_stream(stream)), "hswa_selftest_bounded_wait")


def hswa_last_kernel():
    return lib.hswa_last_kernel().decode()


def hswa_last_cuda_error():
    return lib.hswa_last_cuda_error().decode()
