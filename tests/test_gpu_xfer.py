"""SWA-mask transfer parity: hswa_swa_gather / hswa_swa_scatter against the
oracle's pack / unpack, bit for bit, to device memory and to pinned host
memory, and a full offload -> drop -> restore -> reload round trip."""
import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
import hybrid_sliding_window_dual_gb300 as H
from scenario import Scenario, raw_host, window_offsets

SWA = wl.KIND_SWA


def gather_and_compare(sc, layer, dst_host):
    B = len(sc.cached)
    lens = sc.ora.seq_len[:B]
    off_h, nbytes = window_offsets(sc.sess, layer, lens, sc.W)
    off = torch.as_tensor(off_h, device="cuda")
    dt = sc.sess.dtype
    esize = torch.empty(0, dtype=dt).element_size()
    n_elem = int(off_h[-1]) * 2 * sc.hkv * sc.d
    assert nbytes == n_elem * esize
    if dst_host:
        buf = torch.empty(n_elem, dtype=dt, pin_memory=True)
    else:
        buf = torch.empty(n_elem, dtype=dt, device="cuda")
    sc.sess.gather(layer, off, B, buf)
    assert sc.sess.check() == 0
    snap_k = raw_host(sc.sess.k[layer])
    snap_v = raw_host(sc.sess.v[layer])
    exp = oracle.swa_pack(snap_k, snap_v, sc.ora.swa_bt, lens, sc.W)
    got = raw_host(buf)
    assert got.shape == exp.shape and np.array_equal(got, exp)
    return buf, off


@pytest.mark.gpu
@pytest.mark.parametrize("dst_host", [False, True])
@pytest.mark.parametrize("dtype", [wl.DTYPE_BF16, wl.DTYPE_F32])
def test_gather_matches_oracle_pack(dst_host, dtype):
    cached = [0, 1, 64, 127, 128, 129, 300, 5000]
    sc = Scenario(8, 2, 128 if dtype == wl.DTYPE_BF16 else 64, 64, 128, dtype, cached,
                  layer_kinds=(SWA, SWA), seed=31)
    for layer in (0, 1):
        gather_and_compare(sc, layer, dst_host)


@pytest.mark.gpu
def test_offload_drop_restore_reload_round_trip():
    cached = [3, 128, 200, 777, 64]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, layer_kinds=(SWA, SWA, SWA), seed=32)
    B = len(cached)
    bufs = [gather_and_compare(sc, layer, True) for layer in range(3)]
    before = [raw_host(b) for b, _ in bufs]
    # evict the SWA segments, shift the free list, give the windows new pages
    assert sc.sess.swa_drop(range(B)) == sc.ora.swa_drop(range(B))
    taken = sc.reserve([B - 1], [200])  # another request takes pages meanwhile
    assert sc.sess.swa_restore(range(B - 1)) == sc.ora.swa_restore(range(B - 1))
    sc.sess.sync()
    sc.assert_tables_equal(device=True)
    lens = sc.ora.seq_len[:B - 1]
    off_h, nbytes = window_offsets(sc.sess, 0, lens, sc.W)
    off = torch.as_tensor(off_h, device="cuda")
    for layer in range(3):
        n = nbytes // 2
        src = bufs[layer][0][:n]
        sc.sess.scatter(layer, off, B - 1, src)
        assert sc.sess.check() == 0
        # the pool now holds what the oracle's unpack would write
        k_exp = raw_host(sc.sess.k[layer]).copy()
        v_exp = raw_host(sc.sess.v[layer]).copy()
        oracle.swa_unpack(before[layer][:n], k_exp, v_exp, sc.ora.swa_bt, lens, sc.W)
        assert np.array_equal(raw_host(sc.sess.k[layer]), k_exp)
        assert np.array_equal(raw_host(sc.sess.v[layer]), v_exp)
        # and gathering again gives the same packed bytes
        out = torch.empty_like(src)
        sc.sess.gather(layer, off, B - 1, out)
        assert sc.sess.check() == 0
        assert torch.equal(out.view(torch.int16), src.view(torch.int16))


@pytest.mark.gpu
def test_gather_of_released_window_page_sets_bounds():
    sc = Scenario(8, 2, 128, 64, 128, wl.DTYPE_BF16, [500], layer_kinds=(SWA,), seed=33)
    sc.sess.d_swa_bt[0, 7] = -1  # a page inside the window
    off = torch.as_tensor(window_offsets(sc.sess, 0, [500], 128)[0], device="cuda")
    buf = torch.zeros(128 * 2 * 2 * 128, dtype=torch.bfloat16, device="cuda")
    sc.sess.gather(0, off, 1, buf)
    assert sc.sess.check() == H.HSWA_ERR_BOUNDS


@pytest.mark.gpu
def test_append_slot_past_pool_sets_bounds_and_skips():
    sc = Scenario(8, 2, 128, 64, 128, wl.DTYPE_BF16, [10], seed=34)
    k = torch.ones(2, 2, 128, dtype=torch.bfloat16, device="cuda")
    before = sc.sess.k[0].clone()
    slots = torch.tensor([-1, sc.cfg.full_pages * 64], dtype=torch.int32, device="cuda")
    sc.sess.append(0, k, k, slots)
    assert sc.sess.check() == H.HSWA_ERR_BOUNDS
    assert torch.equal(before, sc.sess.k[0])
