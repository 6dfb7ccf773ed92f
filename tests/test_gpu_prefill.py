"""Chunked-prefill parity: libhswa (GPU) against the float64 oracle.

A chunk of new tokens per sequence is reserved on both sides, appended with
hswa_append_kv, and hswa_prefill_chunk runs for a Full layer (keys [0, t])
and an SWA layer (keys [t - W + 1, t]); every output row checked is compared
element by element with the oracle. The SWA release after the chunk must
leave identical tables on both sides."""
import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
import hybrid_sliding_window_dual_gb300 as H
from scenario import Scenario, TOL, device_out, max_err, prefill_kernel, raw_host

FULL, SWA = wl.KIND_FULL, wl.KIND_SWA


def run_prefill_chunk(sc, chunk, seed, row_samples=None, expect_kernel=False):
    """chunk[s] new tokens for sequence s. row_samples: per-sequence list of
    chunk rows to check (None = all). expect_kernel: check that each layer
    ran the tensor-core kernel of its kind."""
    B = len(sc.cached)
    prefix = sc.ora.seq_len[:B].copy()
    chunk = np.asarray(chunk, np.int64)
    q_start = np.zeros(B + 1, np.int64)
    q_start[1:] = np.cumsum(chunk)
    T = int(q_start[-1])
    full_slots, swa_slots = sc.reserve(range(B), chunk)
    sc.sess.sync()
    d_prefix = torch.as_tensor(prefix.astype(np.int32), device="cuda")
    d_qs = torch.as_tensor(q_start.astype(np.int32), device="cuda")
    seqs = list(range(B))
    errs = {}
    for layer, kind in enumerate(sc.kinds):
        slots = full_slots if kind == FULL else swa_slots
        snap = sc.snapshot(layer, seqs)
        q = sc.gen((T, sc.hq, sc.d), seed + 10 * layer)
        kn = sc.gen((T, sc.hkv, sc.d), seed + 10 * layer + 1)
        vn = sc.gen((T, sc.hkv, sc.d), seed + 10 * layer + 2)
        qd = sc.to_dev(q)
        o = torch.full_like(qd, float("nan"))
        sc.sess.append(layer, sc.to_dev(kn), sc.to_dev(vn), torch.as_tensor(slots, device="cuda"))
        sc.sess.prefill(layer, qd, o, d_prefix, d_qs, B, int(chunk.max()) if B else 0, sc.scale)
        assert sc.sess.check() == 0
        if expect_kernel:
            assert H.hswa_last_kernel() == prefill_kernel(kind, sc.window(layer))
        sc.oracle_append(snap, slots, (raw_host(kn), raw_host(vn)), sc.P)
        rows, q_seq, q_pos = [], [], []
        for s in range(B):
            rs = range(int(chunk[s])) if row_samples is None else row_samples[s]
            for r in rs:
                rows.append(int(q_start[s]) + r)
                q_seq.append(s)
                q_pos.append(int(prefix[s]) + r)
        rows = np.array(rows, np.int64)
        exp = oracle.attention(raw_host(q)[rows], snap[0], snap[1], snap[2], np.array(q_seq), np.array(q_pos),
                               sc.window(layer), sc.scale)
        got = device_out(o)[rows]
        assert np.isfinite(got).all()
        errs[kind] = max_err(got, exp)
        assert errs[kind] <= TOL[sc.dtype], (kind, errs[kind])
    sc.release(range(B))
    sc.sess.sync()
    sc.assert_tables_equal(device=True)
    return errs


@pytest.mark.gpu
def test_tiny_workload_decode_then_chunk():
    """Two sequences (300 and 77 cached), 4 Q / 1 KV heads, d 64, page 16,
    fp32: one decode token each, then a 64-token chunk on the second
    sequence crossing the W = 128 boundary, then release."""
    w = wl.tiny()
    sc = Scenario(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page_size, w.window, w.dtype, w.cached, seed=w.seed)
    from test_gpu_decode import run_decode_step
    run_decode_step(sc, [0, 1], seed=11)
    sc.release([0, 1])
    run_prefill_chunk(sc, [0, 64], seed=21)
    assert sc.ora.seq_len[1] == 142


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(8, 2, 64, 16, wl.DTYPE_BF16, 40), (4, 1, 64, 16, wl.DTYPE_F32, 128)])
def test_prefill_generic_ragged(shape):
    hq, hkv, d, P, dtype, W = shape
    cached = [0, 5, 16, 200]
    sc = Scenario(hq, hkv, d, P, W, dtype, cached, seed=12, extra_tokens=300)
    run_prefill_chunk(sc, [33, 0, 100, 257], seed=5)


@pytest.mark.gpu
@pytest.mark.parametrize("permute", [False, True])
def test_prefill_bf16_d128_ragged(permute):
    """Chunks that are not multiples of the tile, prefixes that are not
    multiples of the page, an empty chunk and a chunk from position 0."""
    cached = [0, 70, 1000, 129, 4000]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=13, permute=permute, extra_tokens=700)
    run_prefill_chunk(sc, [300, 1, 0, 513, 129], seed=9)


@pytest.mark.gpu
def test_prefill_fast_path_dispatch_and_window_wider_than_chunk():
    """Tile-aligned and unaligned prefixes around the window edge."""
    cached = [127, 128, 255, 256, 60]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=14, extra_tokens=400)
    run_prefill_chunk(sc, [128, 129, 1, 256, 300], seed=3, expect_kernel=True)


@pytest.mark.gpu
@pytest.mark.parametrize("hq,hkv", [(16, 8), (24, 4), (32, 8), (48, 4)])
def test_prefill_query_heads_per_kv_head(hq, hkv):
    """2, 6, 4 and 12 query heads per kv head: a CTA takes a pair of query
    heads of one kv head, so every even group size runs on the tensor-core
    kernel. Ragged chunks and prefixes, Full and SWA layer."""
    cached = [0, 70, 1000, 129]
    sc = Scenario(hq, hkv, 128, 64, 128, wl.DTYPE_BF16, cached, seed=17, extra_tokens=600)
    run_prefill_chunk(sc, [300, 1, 513, 129], seed=6, expect_kernel=True)


@pytest.mark.gpu
def test_chunked_prefill_full_size_sampled():
    """8 sequences, cached prefix uniform in [8192, 65536], 4096-token chunk,
    64/8 heads, d 128, page 64: the chunked-prefill workload in the launch
    configuration the benchmark times. The oracle checks rows at the tile
    edges and the chunk ends of every sequence, on every head."""
    w = wl.chunked_prefill()
    sc = Scenario(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page_size, w.window, w.dtype, w.cached, seed=w.seed,
                  extra_tokens=w.n_new + 64)
    rows = [0, 1, 127, 128, 129, 1000, 2047, 4094, 4095]
    run_prefill_chunk(sc, [w.n_new] * len(w.cached), seed=77, row_samples=[rows] * len(w.cached),
                      expect_kernel=True)


@pytest.mark.gpu
def test_prefill_swa_after_release_reads_only_live_pages():
    """Prefixes built chunk by chunk with a release after each, so the SWA
    pages below the window are gone; the SWA prefill must neither read them
    nor report them (its first key tile may start below the window)."""
    cached = [1000, 777, 130, 2049]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=15, chunk=100, extra_tokens=600)
    assert (sc.ora.swa_bt[:, :10] < 0).any()
    run_prefill_chunk(sc, [200, 129, 64, 500], seed=4, expect_kernel=True)


@pytest.mark.gpu
@pytest.mark.parametrize("W", [1, 40, 127, 128, 129])
def test_prefill_swa_windows_many_sequences(W):
    """SWA windows around the two-key-tile limit of the persistent window
    kernel (W <= 128 runs it, W = 129 the general kernel), over 40 sequences
    with ragged chunks (some empty) and prefixes, so that the CTAs' shares of
    the unit list start and end inside (sequence, kv head, block) groups and
    K / V tiles are reused across head pairs and blocks; every row against
    the oracle."""
    rng = np.random.default_rng(100 + W)
    cached = [int(x) for x in rng.integers(0, 3000, size=40)]
    chunk = [int(x) for x in rng.integers(0, 400, size=40)]
    chunk[3] = 0
    sc = Scenario(16, 2, 128, 64, W, wl.DTYPE_BF16, cached, layer_kinds=(SWA,), seed=18, extra_tokens=420)
    run_prefill_chunk(sc, chunk, seed=8, expect_kernel=True)


@pytest.mark.gpu
@pytest.mark.parametrize("W", [128, 64])
def test_prefill_swa_many_short_sequences(W):
    """300 sequences with chunks of 0-150 tokens: each persistent CTA's share
    of the window kernel's unit list runs across many sequences, partial
    blocks and kv heads, so its K / V page ring is refilled at every
    sequence boundary; every row against the oracle."""
    rng = np.random.default_rng(300 + W)
    cached = [int(x) for x in rng.integers(0, 700, size=300)]
    chunk = [int(x) for x in rng.integers(0, 151, size=300)]
    sc = Scenario(16, 2, 128, 64, W, wl.DTYPE_BF16, cached, layer_kinds=(SWA,), seed=21, extra_tokens=160)
    run_prefill_chunk(sc, chunk, seed=11, expect_kernel=True)


@pytest.mark.gpu
@pytest.mark.parametrize("cached,chunk", [([1000], [5]), ([0], [1]), ([127], [130]), ([300, 0], [0, 700])])
def test_prefill_swa_few_units(cached, chunk):
    """Chunks so small that most CTAs of the persistent window kernel get no
    unit; a chunk inside one block, one from position 0, one crossing a
    block edge, an empty chunk next to a long one."""
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, layer_kinds=(SWA,), seed=19, extra_tokens=720)
    run_prefill_chunk(sc, chunk, seed=9, expect_kernel=True)


@pytest.mark.gpu
def test_prefill_many_sequences_keep_their_order():
    """70 sequences: past 64 the Full-layer grid keeps the sequences' own
    order instead of ranking them longest first; ragged chunks and prefixes,
    every row of both layers against the oracle."""
    rng = np.random.default_rng(70)
    cached = [int(x) for x in rng.integers(0, 1500, size=70)]
    chunk = [int(x) for x in rng.integers(0, 200, size=70)]
    sc = Scenario(16, 2, 128, 64, 128, wl.DTYPE_BF16, cached, seed=20, extra_tokens=210)
    run_prefill_chunk(sc, chunk, seed=10, expect_kernel=True)


@pytest.mark.gpu
def test_prefill_window_covers_whole_sequence_equals_full():
    """W >= every position: the SWA layer's chunk attends to exactly the Full
    layer's keys, so both layers give the same bits on the same history."""
    cached = [0, 100, 700, 1500]
    chunk = [130, 64, 300, 1]
    sc = Scenario(64, 8, 128, 64, 4096, wl.DTYPE_BF16, cached, layer_kinds=(FULL, SWA), seed=16,
                  extra_tokens=400, chunk=8192)
    B = len(cached)
    prefix = sc.ora.seq_len[:B].copy()
    full_slots, swa_slots = sc.reserve(range(B), chunk)
    sc.sess.sync()
    q_start = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    T = int(q_start[-1])
    kn = sc.to_dev(sc.gen((T, 8, 128), 1))
    vn = sc.to_dev(sc.gen((T, 8, 128), 2))
    q = sc.to_dev(sc.gen((T, 64, 128), 3))
    d_prefix = torch.as_tensor(prefix.astype(np.int32), device="cuda")
    d_qs = torch.as_tensor(q_start, device="cuda")
    outs = []
    for layer, slots in ((0, full_slots), (1, swa_slots)):
        if layer == 1:  # the same K/V history in both layers
            for s in range(B):
                for p in range(int(prefix[s] + 63) // 64):
                    sc.sess.k[1][sc.ora.swa_bt[s, p]] = sc.sess.k[0][sc.ora.full_bt[s, p]]
                    sc.sess.v[1][sc.ora.swa_bt[s, p]] = sc.sess.v[0][sc.ora.full_bt[s, p]]
        sc.sess.append(layer, kn, vn, torch.as_tensor(slots, device="cuda"))
        o = torch.empty_like(q)
        sc.sess.prefill(layer, q, o, d_prefix, d_qs, B, max(chunk), sc.scale)
        assert H.hswa_last_kernel() == "prefill_tc_bf16_d128"
        outs.append(o)
    assert sc.sess.check() == 0
    assert torch.equal(outs[0], outs[1])
