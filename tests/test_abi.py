"""The C ABI without a GPU: the library loads, exports every function that
include/hswa.h declares, and its host-side pool bookkeeping matches the
oracle's bit for bit (tables, slots, free lists) on random call traces."""
import ctypes
import os
import re

import numpy as np
import pytest

import hswa_workloads as wl
import oracle
import hybrid_sliding_window_dual_gb300 as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"^[A-Za-z_][\w \*]*?\b(hswa_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("hswa_append_kv", "hswa_decode", "hswa_prefill_chunk", "hswa_swa_release",
                     "hswa_swa_gather", "hswa_swa_scatter", "hswa_reserve", "hswa_pool_create"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(H.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def make_pair(W=128, P=16, full=600, swa=120, S=6, MP=64, seed=0, permute=True):
    fo = wl.permutation(full, seed) if permute else None
    so = wl.permutation(swa, seed + 100) if permute else None
    cfg = H.Config(window=W, page_size=P, n_q_heads=8, n_kv_heads=2, head_dim=64,
                   dtype=H.HSWA_DTYPE_BF16, full_pages=full, swa_pages=swa, max_seqs=S,
                   max_pages_per_seq=MP)
    lib_pool = H.hswa_pool_create(cfg, fo, so)
    ora = oracle.DualPool(W, P, full, swa, S, MP, full_free_order=fo, swa_free_order=so)
    return cfg, lib_pool, ora


def assert_same_state(cfg, lib_pool, ora):
    f, s, lens = H.hswa_get_tables(lib_pool, cfg)
    assert np.array_equal(f, ora.full_bt)
    assert np.array_equal(s, ora.swa_bt)
    assert np.array_equal(lens.astype(np.int64), ora.seq_len)
    assert np.array_equal(H.hswa_get_free_list(lib_pool, H.HSWA_KIND_FULL), np.array(ora.full_free, np.int32))
    assert np.array_equal(H.hswa_get_free_list(lib_pool, H.HSWA_KIND_SWA), np.array(ora.swa_free, np.int32))


@pytest.mark.parametrize("seed", range(4))
def test_bookkeeping_matches_oracle_on_random_trace(seed):
    rng = np.random.default_rng(seed)
    cfg, lp, ora = make_pair(seed=seed)
    S = cfg.max_seqs
    for step in range(400):
        op = rng.choice(["reserve", "reserve", "reserve", "release", "free", "drop_restore"])
        ids = np.sort(rng.choice(S, size=int(rng.integers(1, S + 1)), replace=False))
        if op == "reserve":
            n_new = rng.choice([0, 1, 1, 5, 17, 40], size=len(ids))
            try:
                exp = ora.reserve(ids, n_new)
            except oracle.NoSpace:
                with pytest.raises(H.NoSpace):
                    H.hswa_reserve(lp, ids, n_new)
            except ValueError:
                with pytest.raises(H.HswaError):
                    H.hswa_reserve(lp, ids, n_new)
            else:
                got = H.hswa_reserve(lp, ids, n_new)
                assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])
        elif op == "release":
            assert H.hswa_swa_release(lp, ids[::-1]) == ora.swa_release(ids)
        elif op == "free":
            H.hswa_seq_free(lp, ids[:1])
            ora.seq_free(ids[:1])
        else:
            assert H.hswa_swa_drop(lp, ids) == ora.swa_drop(ids)
            try:
                n = ora.swa_restore(ids)
            except oracle.NoSpace:
                with pytest.raises(H.NoSpace):
                    H.hswa_swa_restore(lp, ids)
            else:
                assert H.hswa_swa_restore(lp, ids) == n
        assert_same_state(cfg, lp, ora)
    H.hswa_pool_destroy(lp)


def test_invalid_arguments_are_rejected():
    cfg, lp, _ = make_pair()
    with pytest.raises(H.HswaError) as e:
        H.hswa_reserve(lp, [3, 1], [1, 1])  # not ascending
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    with pytest.raises(H.HswaError):
        H.hswa_reserve(lp, [cfg.max_seqs], [1])  # id out of range
    with pytest.raises(H.HswaError):
        H.hswa_reserve(lp, [0], [-1])
    with pytest.raises(H.HswaError):
        H.hswa_reserve(lp, [0], [cfg.max_pages_per_seq * cfg.page_size + 1])
    with pytest.raises(H.HswaError):
        H.hswa_swa_release(lp, [2, 2])
    bad = H.Config(window=0, page_size=16, n_q_heads=8, n_kv_heads=2, head_dim=64, dtype=1,
                   full_pages=8, swa_pages=8, max_seqs=2, max_pages_per_seq=4)
    with pytest.raises(H.HswaError):
        H.hswa_pool_create(bad)
    bad.window, bad.n_kv_heads = 128, 3  # 8 % 3 != 0
    with pytest.raises(H.HswaError):
        H.hswa_pool_create(bad)
    bad.n_kv_heads = 2
    with pytest.raises(H.HswaError):
        H.hswa_pool_create(bad, full_free_order=[0, 1, 2, 3, 4, 5, 6, 6])  # not a permutation
    H.hswa_pool_destroy(lp)


def test_no_space_leaves_state_unchanged():
    cfg, lp, ora = make_pair(full=20, swa=6, permute=False)
    H.hswa_reserve(lp, [0], [60])
    ora.reserve([0], [60])
    with pytest.raises(H.NoSpace):
        H.hswa_reserve(lp, [1, 2], [16, 40])  # SWA needs 4 more, has 2
    assert_same_state(cfg, lp, ora)
    H.hswa_pool_destroy(lp)


def test_device_calls_validate_before_launching():
    """Argument errors come back as status codes without touching a GPU."""
    cfg, lp, _ = make_pair()
    layer = H.Layer(kind=7, window=128, k_pool=16, v_pool=16)
    with pytest.raises(H.HswaError) as e:
        H.hswa_decode(lp, layer, 16, 16, 16, 16, 1, 1.0, 256, 1 << 20)
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    layer = H.Layer(kind=H.HSWA_KIND_SWA, window=0, k_pool=16, v_pool=16)
    with pytest.raises(H.HswaError):
        H.hswa_prefill_chunk(lp, layer, 16, 16, 16, 16, 16, 1, 4, 4, 1.0)
    with pytest.raises(H.HswaError):
        H.hswa_swa_gather(lp, H.Layer(kind=H.HSWA_KIND_FULL, window=128, k_pool=16, v_pool=16),
                          16, 16, 16, 1, 16)
    assert H.hswa_decode_workspace_size(lp, 64) > 0
    # multi-token decode: the token count is checked first
    ok_layer = H.Layer(kind=H.HSWA_KIND_FULL, window=0, k_pool=16, v_pool=16)
    for n_tok in (0, -1, H.HSWA_DECODE_MAX_TOKENS + 1):
        assert H.hswa_decode_multi_workspace_size(lp, 64, n_tok) == 0
        with pytest.raises(H.HswaError) as e:
            H.hswa_decode_multi(lp, ok_layer, 16, 16, 16, 16, 1, n_tok, 1.0, 256, 1 << 20)
        assert e.value.status == H.HSWA_ERR_INVALID_ARG
    sizes = [H.hswa_decode_multi_workspace_size(lp, 64, t) for t in range(1, H.HSWA_DECODE_MAX_TOKENS + 1)]
    assert sizes[0] == H.hswa_decode_workspace_size(lp, 64)
    assert all(b > a for a, b in zip(sizes, sizes[1:]))
    H.hswa_pool_destroy(lp)


def test_empty_batches_return_before_any_launch():
    """A chunked prefill with no sequences or no query rows, and a window
    gather or scatter with no sequences, return HSWA_OK before touching a
    device pointer (the pointers given here are not device memory)."""
    cfg, lp, _ = make_pair()
    full = H.Layer(kind=H.HSWA_KIND_FULL, window=0, k_pool=16, v_pool=16)
    swa = H.Layer(kind=H.HSWA_KIND_SWA, window=128, k_pool=16, v_pool=16)
    for layer in (full, swa):
        H.hswa_prefill_chunk(lp, layer, 16, 16, 16, 16, 16, 0, 0, 0, 1.0)
        H.hswa_prefill_chunk(lp, layer, 16, 16, 16, 16, 16, 3, 0, 0, 1.0)
    H.hswa_swa_gather(lp, swa, 16, 16, 16, 0, 16)
    H.hswa_swa_scatter(lp, swa, 16, 16, 16, 0, 16)
    # but a negative count, or more rows in one sequence than in the chunk, is refused
    with pytest.raises(H.HswaError) as e:
        H.hswa_prefill_chunk(lp, full, 16, 16, 16, 16, 16, -1, 0, 0, 1.0)
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    with pytest.raises(H.HswaError) as e:
        H.hswa_prefill_chunk(lp, full, 16, 16, 16, 16, 16, 2, 3, 4, 1.0)
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    with pytest.raises(H.HswaError) as e:
        H.hswa_swa_gather(lp, swa, 16, 16, 16, -1, 16)
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    H.hswa_pool_destroy(lp)


@pytest.mark.parametrize("dtype", [H.HSWA_DTYPE_BF16, H.HSWA_DTYPE_FP8_E4M3])
def test_decode_refuses_more_rows_than_the_merge_grid_takes(dtype):
    """The partial-record merge runs one CTA row per (sequence, token): at
    most 65535 rows, so 4096 sequences of 16 tokens are refused with
    HSWA_ERR_UNSUPPORTED before any launch, and 4095 are not refused for
    that reason."""
    cfg = H.Config(window=128, page_size=64, n_q_heads=64, n_kv_heads=8, head_dim=128, dtype=dtype,
                   full_pages=64, swa_pages=64, max_seqs=4096, max_pages_per_seq=4)
    lp = H.hswa_pool_create(cfg, None, None)
    scales = dict(k_scale=16, v_scale=16) if dtype == H.HSWA_DTYPE_FP8_E4M3 else {}
    layer = H.Layer(kind=H.HSWA_KIND_FULL, window=0, k_pool=16, v_pool=16, **scales)
    with pytest.raises(H.HswaError) as e:
        H.hswa_decode_multi(lp, layer, 16, 16, 16, 16, 4096, 16, 1.0, 256, 1 << 30)
    assert e.value.status == H.HSWA_ERR_UNSUPPORTED
    H.hswa_pool_destroy(lp)


def test_prefill_workspace_sizes():
    """Only FP8 pools need a prefill workspace. Its layout: the staging table
    [n_seqs][table row], a first-copy offset per sequence [n_seqs + 1], the
    fp16 copy of the q rows, then fp16 K and V page copies. The upper bound
    holds, per sequence, its whole table row (Full layer) or
    ceil((W - 1 + max_q_len) / P) + 1 pages (SWA layer) and n_seqs * max_q_len
    query rows; the exact size holds the pages the chunk reads: logical pages
    0 .. (prefix + n - 1) / P (Full), from (prefix - W + 1) / P (SWA)."""
    cfg, lp, _ = make_pair()
    full = H.Layer(kind=H.HSWA_KIND_FULL, window=0, k_pool=16, v_pool=16)
    assert H.hswa_prefill_workspace_size(lp, full, 4, 4096) == 0
    assert H.hswa_prefill_workspace_size_exact(lp, full, [0], [0, 5]) == 0
    H.hswa_pool_destroy(lp)
    W, P, MP, hkv, d = 128, 64, 100, 8, 128
    cfg = H.Config(window=W, page_size=P, n_q_heads=64, n_kv_heads=hkv, head_dim=d, dtype=H.HSWA_DTYPE_FP8_E4M3,
                   full_pages=1000, swa_pages=100, max_seqs=8, max_pages_per_seq=MP)
    lp = H.hswa_pool_create(cfg, None, None)
    swa = H.Layer(kind=H.HSWA_KIND_SWA, window=W, k_pool=16, v_pool=16)
    page = hkv * P * d * 2  # one fp16 K (or V) page copy

    def up1k(x):
        return -(-x // 1024) * 1024

    def pages(n_bytes, n_seqs, q_rows):
        fixed = up1k(n_seqs * MP * 4) + up1k((n_seqs + 1) * 4) + up1k(q_rows * 64 * d * 2)
        return (n_bytes - fixed) / (2 * page)

    assert pages(H.hswa_prefill_workspace_size(lp, full, 8, 4096), 8, 8 * 4096) == 8 * MP
    for q in (1, 64, 65, 4096):
        per = min(MP, -(-(W - 1 + q) // P) + 1)
        assert pages(H.hswa_prefill_workspace_size(lp, swa, 8, q), 8, 8 * q) == 8 * per
    assert H.hswa_prefill_workspace_size(lp, H.Layer(kind=H.HSWA_KIND_SWA, window=0), 8, 64) == 0
    # exact sizes: prefixes around page and window edges, an empty chunk
    prefix = np.array([0, 63, 64, 127, 128, 1000, 5000, 77], np.int32)
    chunk = np.array([1, 1, 64, 130, 0, 300, 129, 64], np.int32)
    q_start = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    exp_full = sum(-(-(p + n) // P) for p, n in zip(prefix, chunk) if n > 0)
    exp_swa = sum((p + n - 1) // P - max(0, p - W + 1) // P + 1 for p, n in zip(prefix, chunk) if n > 0)
    assert pages(H.hswa_prefill_workspace_size_exact(lp, full, prefix, q_start), 8, int(q_start[-1])) == exp_full
    assert pages(H.hswa_prefill_workspace_size_exact(lp, swa, prefix, q_start), 8, int(q_start[-1])) == exp_swa
    assert H.hswa_prefill_workspace_size_exact(lp, full, prefix, q_start) < \
        H.hswa_prefill_workspace_size(lp, full, 8, int(chunk.max()))
    H.hswa_pool_destroy(lp)


@pytest.mark.parametrize("dtype", [H.HSWA_DTYPE_BF16, H.HSWA_DTYPE_F32, H.HSWA_DTYPE_FP8_E4M3])
def test_swa_window_offsets_match_oracle(dtype):
    """hswa_swa_window_offsets (host): the packed-buffer token offsets are the
    prefix sum of the oracle's in-window counts min(L, W), from given lengths
    and from the pool's own lengths after a reserve trace; the byte count
    follows the packed layout of the pool's element type."""
    W, P, hkv, d = 128, 16, 2, 128
    cfg = H.Config(window=W, page_size=P, n_q_heads=8, n_kv_heads=hkv, head_dim=d, dtype=dtype,
                   full_pages=4000, swa_pages=400, max_seqs=6, max_pages_per_seq=256)
    pool = H.hswa_pool_create(cfg, None, None)
    ora = oracle.DualPool(W, P, 4000, 400, 6, 256)
    swa = H.Layer(kind=H.HSWA_KIND_SWA, window=W)
    per_token = 2 * hkv * (d + 4) if dtype == H.HSWA_DTYPE_FP8_E4M3 else 2 * hkv * d * (4 if dtype == 0 else 2)
    try:
        lens = np.array([0, 1, 127, 128, 129, 5000], np.int32)
        off, nbytes = H.hswa_swa_window_offsets(pool, swa, len(lens), lens)
        exp = oracle.swa_window_counts(lens, W)[1]
        assert np.array_equal(off, exp) and nbytes == int(exp[-1]) * per_token
        rng = np.random.default_rng(5)
        for _ in range(20):
            ids = np.sort(rng.choice(6, size=rng.integers(1, 7), replace=False))
            n_new = rng.integers(0, 300, size=ids.size)
            H.hswa_reserve(pool, ids, n_new)
            ora.reserve(ids, n_new)
            H.hswa_swa_release(pool, ids)
            ora.swa_release(ids)
            for n in (0, 3, 6):
                off, nbytes = H.hswa_swa_window_offsets(pool, swa, n)
                exp = oracle.swa_window_counts(ora.seq_len[:n], W)[1]
                assert np.array_equal(off, exp) and nbytes == int(exp[-1]) * per_token
        full = H.Layer(kind=H.HSWA_KIND_FULL, window=W)
        with pytest.raises(H.HswaError):
            H.hswa_swa_window_offsets(pool, full, 3)
        with pytest.raises(H.HswaError):
            H.hswa_swa_window_offsets(pool, swa, 7)
        with pytest.raises(H.HswaError):
            H.hswa_swa_window_offsets(pool, swa, 1, np.array([-1], np.int32))
    finally:
        H.hswa_pool_destroy(pool)
