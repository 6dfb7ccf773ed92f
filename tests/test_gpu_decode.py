"""Decode parity: libhswa (GPU) against the float64 oracle.

Each case reserves one new token per sequence on both sides (slots must
agree bit for bit), appends its K/V through hswa_append_kv, runs hswa_decode
for a Full and an SWA layer and compares every output element with the
oracle (bf16: max abs 2e-2, fp32: 1e-5)."""
import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
import hybrid_sliding_window_dual_gb300 as H
from scenario import Scenario, TOL, device_out, max_err, raw_host

FULL, SWA = wl.KIND_FULL, wl.KIND_SWA


def run_decode_step(sc, samples, seed, expect_kernel=None):
    B = len(sc.cached)
    full_slots, swa_slots = sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    sc.assert_tables_equal(device=True)
    errs = {}
    for layer, kind in enumerate(sc.kinds):
        slots = full_slots if kind == FULL else swa_slots
        snap = sc.snapshot(layer, samples)
        q = sc.gen((B, sc.hq, sc.d), seed + 10 * layer)
        kn = sc.gen((B, sc.hkv, sc.d), seed + 10 * layer + 1)
        vn = sc.gen((B, sc.hkv, sc.d), seed + 10 * layer + 2)
        qd = sc.to_dev(q)
        o = torch.full_like(qd, float("nan"))
        sc.sess.append(layer, sc.to_dev(kn), sc.to_dev(vn), torch.as_tensor(slots, device="cuda"))
        sc.sess.decode(layer, qd, o, B, sc.scale)
        assert sc.sess.check() == 0
        if expect_kernel:
            assert H.hswa_last_kernel() == expect_kernel
        # appended rows are in the pool bit for bit
        P = sc.P
        sl = torch.as_tensor(slots.astype(np.int64), device="cuda")
        rows_k = sc.sess.k[layer][sl // P, :, sl % P, :]
        assert np.array_equal(raw_host(rows_k), raw_host(kn))
        # oracle: the snapshot (taken before the append) plus the oracle's append
        sc.oracle_append(snap, slots[samples], (raw_host(kn)[samples], raw_host(vn)[samples]), P)
        lens = sc.ora.seq_len[samples]
        exp = oracle.attention(raw_host(q)[samples], snap[0], snap[1], snap[2], np.arange(len(samples)),
                               lens - 1, sc.window(layer), sc.scale)
        got = device_out(o)[samples]
        errs[kind] = max_err(got, exp)
        assert np.isfinite(got).all()
        assert errs[kind] <= TOL[sc.dtype], (kind, errs[kind])
    return errs


@pytest.mark.gpu
@pytest.mark.parametrize("permute", [False, True])
def test_decode_fast_path_ragged_lengths(permute):
    cached = [0, 1, 62, 63, 64, 127, 128, 191, 700, 3000]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=3, permute=permute)
    run_decode_step(sc, list(range(len(cached))), seed=50, expect_kernel="decode_mma_bf16_d128")


@pytest.mark.gpu
def test_decode_fast_path_many_steps_with_release():
    """Several decode steps; release every 8 tokens; tables re-synced each step."""
    cached = [5, 130, 255, 1000, 2047]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=4)
    for step in range(20):
        run_decode_step(sc, list(range(len(cached))), seed=100 + step)
        if step % 8 == 7:
            sc.release(range(len(cached)))
            sc.sess.sync()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(8, 2, 64, 16, wl.DTYPE_BF16), (4, 1, 64, 16, wl.DTYPE_F32),
                                   (6, 3, 32, 8, wl.DTYPE_F32), (16, 4, 128, 64, wl.DTYPE_BF16)])
def test_decode_generic_path(shape):
    hq, hkv, d, P, dtype = shape
    cached = [0, 3, 17, 100, 300]
    sc = Scenario(hq, hkv, d, P, 12 if P < 64 else 128, dtype, cached, seed=5)
    run_decode_step(sc, list(range(len(cached))), seed=7)
    assert H.hswa_last_kernel().startswith("decode_generic")


@pytest.mark.gpu
def test_decode_window_covers_whole_sequence_equals_full():
    """W >= L: the SWA layer attends to exactly the Full layer's keys."""
    cached = [10, 50, 99]
    sc = Scenario(64, 8, 128, 64, 512, wl.DTYPE_BF16, cached, layer_kinds=(FULL, SWA), seed=6)
    B = len(cached)
    full_slots, swa_slots = sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    kn = sc.to_dev(sc.gen((B, 8, 128), 1))
    vn = sc.to_dev(sc.gen((B, 8, 128), 2))
    q = sc.to_dev(sc.gen((B, 64, 128), 3))
    outs = []
    for layer, slots in ((0, full_slots), (1, swa_slots)):
        # same K/V history in both layers: copy the Full pages into the SWA pages
        if layer == 1:
            for s in range(B):
                L = int(sc.ora.seq_len[s])
                for p in range((L + 63) // 64):
                    sc.sess.k[1][sc.ora.swa_bt[s, p]] = sc.sess.k[0][sc.ora.full_bt[s, p]]
                    sc.sess.v[1][sc.ora.swa_bt[s, p]] = sc.sess.v[0][sc.ora.full_bt[s, p]]
        sc.sess.append(layer, kn, vn, torch.as_tensor(slots, device="cuda"))
        o = torch.empty_like(q)
        sc.sess.decode(layer, q, o, B, sc.scale)
        outs.append(o)
    assert sc.sess.check() == 0
    assert torch.equal(outs[0], outs[1])


@pytest.mark.gpu
def test_decode_bad_table_entry_sets_bounds_and_skips():
    cached = [300, 300]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=8)
    B = 2
    sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    sc.sess.d_full_bt[1, 2] = -1           # a released / never-reserved page inside the key range
    sc.sess.d_full_bt[0, 3] = 1 << 30      # a page past the pool
    q = sc.to_dev(sc.gen((B, 64, 128), 1))
    o = torch.empty_like(q)
    sc.sess.decode(0, q, o, B, sc.scale)
    assert sc.sess.check() == H.HSWA_ERR_BOUNDS
    assert sc.sess.check() == 0            # the word was cleared
    assert torch.isfinite(o.float()).all()


@pytest.mark.gpu
def test_decode_empty_batch_is_a_no_op():
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, [10], seed=9)
    q = torch.zeros(0, 64, 128, dtype=torch.bfloat16, device="cuda")
    sc.sess.decode(0, q, q, 0, sc.scale)
    assert sc.sess.check() == 0


@pytest.mark.gpu
def test_decode_batch_full_size_sampled():
    """64 sequences, cached lengths uniform in [1024, 32768], 64/8 heads,
    d 128, page 64, permuted Full free list: the decode-batch workload in
    the launch configuration the benchmark times; the oracle checks
    sequences {0, 1, longest, last} on every head."""
    w = wl.decode_batch()
    sc = Scenario(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page_size, w.window, w.dtype, w.cached, seed=w.seed)
    B = len(w.cached)
    samples = sorted({0, 1, int(np.argmax(w.cached)), B - 1})
    run_decode_step(sc, samples, seed=1234, expect_kernel="decode_mma_bf16_d128")


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(64, 8, 128, 64, wl.DTYPE_BF16), (8, 2, 64, 16, wl.DTYPE_BF16)])
def test_decode_append_fused_matches_oracle_and_separate_calls(shape):
    """hswa_decode_append gives the oracle's result, leaves the pool exactly as
    hswa_append_kv does, and matches append + decode bit for bit."""
    hq, hkv, d, P, dtype = shape
    cached = [0, 1, 63, 64, 65, 127, 700, 3000]
    B = len(cached)
    a = Scenario(hq, hkv, d, P, 128, dtype, cached, seed=21)
    b = Scenario(hq, hkv, d, P, 128, dtype, cached, seed=21)
    fa, sa = a.reserve(range(B), [1] * B)
    fb, sb = b.reserve(range(B), [1] * B)
    a.sess.sync()
    b.sess.sync()
    for layer, kind in enumerate(a.kinds):
        slots = fa if kind == FULL else sa
        snap = a.snapshot(layer, list(range(B)))
        q = a.gen((B, hq, d), 300 + layer)
        kn = a.gen((B, hkv, d), 310 + layer)
        vn = a.gen((B, hkv, d), 320 + layer)
        ds = torch.as_tensor(slots, device="cuda")
        o_fused = torch.full((B, hq, d), float("nan"), dtype=a.sess.dtype, device="cuda")
        a.sess.decode_append(layer, a.to_dev(q), a.to_dev(kn), a.to_dev(vn), ds, o_fused, B, a.scale)
        assert a.sess.check() == 0
        o_sep = torch.full_like(o_fused, float("nan"))
        b.sess.append(layer, b.to_dev(kn), b.to_dev(vn), ds)
        b.sess.decode(layer, b.to_dev(q), o_sep, B, b.scale)
        assert b.sess.check() == 0
        assert torch.equal(o_fused.view(torch.int16), o_sep.view(torch.int16))
        assert torch.equal(a.sess.k[layer], b.sess.k[layer]) and torch.equal(a.sess.v[layer], b.sess.v[layer])
        a.oracle_append(snap, slots, (raw_host(kn), raw_host(vn)), P)
        exp = oracle.attention(raw_host(q), snap[0], snap[1], snap[2], np.arange(B), a.ora.seq_len[:B] - 1,
                               a.window(layer), a.scale)
        assert max_err(device_out(o_fused), exp) <= TOL[dtype]
