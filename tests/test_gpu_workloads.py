"""Parity on the two largest workloads, at full size, in the launch
configuration the benchmark times.

* hybrid 70-layer decode: 10 Full + 60 SWA layers (Full at every 7th),
  batch 128 at 128K cached tokens, 64/8 heads, d 128. One decode step runs
  over all 70 layers; the oracle checks sequences {0, 127} on one Full and
  two SWA layers (every head), and the slots and tables bit for bit.
* SWA-mask transfer + eviction: 256 sequences with lognormal lengths
  (median 16K, cap 256K), 60 SWA layers. Every layer's in-window tokens are
  gathered into pinned host memory and compared with the oracle's pack (two
  layers); the SWA segments are evicted, given new pages and scattered back,
  and a second gather must reproduce every layer bit for bit. Then four
  rounds of 64 decode tokens with a release after each keep the SWA pool at
  the window level, with identical tables on both sides.
"""
import math

import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
from scenario import Scenario, TOL, device_out, max_err, raw_host, window_offsets

FULL, SWA = wl.KIND_FULL, wl.KIND_SWA


@pytest.mark.gpu
def test_hybrid70_decode_step_sampled():
    w = wl.hybrid70()
    B = len(w.cached)
    sc = Scenario(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page_size, w.window, w.dtype, w.cached,
                  layer_kinds=w.layer_kinds, seed=w.seed, permute=False, extra_tokens=8,
                  swa_pages=B * 5 + 80, share_full_pool=True)
    samples = [0, B - 1]
    full_slots, swa_slots = sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    sc.assert_tables_equal(device=True)
    checked = {6: None, 0: None, 69: None}
    for layer, kind in enumerate(w.layer_kinds):
        slots = full_slots if kind == FULL else swa_slots
        q = sc.gen((B, w.n_q_heads, w.head_dim), 7000 + layer)
        kn = sc.gen((B, w.n_kv_heads, w.head_dim), 8000 + layer)
        vn = sc.gen((B, w.n_kv_heads, w.head_dim), 9000 + layer)
        snap = sc.snapshot(layer, samples) if layer in checked else None
        o = torch.full((B, w.n_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
        sc.sess.append(layer, sc.to_dev(kn), sc.to_dev(vn), torch.as_tensor(slots, device="cuda"))
        sc.sess.decode(layer, sc.to_dev(q), o, B, sc.scale)
        if snap is not None:
            assert sc.sess.check() == 0
            sc.oracle_append(snap, slots[samples], (raw_host(kn)[samples], raw_host(vn)[samples]), sc.P)
            lens = sc.ora.seq_len[samples]
            exp = oracle.attention(raw_host(q)[samples], snap[0], snap[1], snap[2], np.arange(len(samples)),
                                   lens - 1, sc.window(layer), sc.scale)
            err = max_err(device_out(o)[samples], exp)
            assert err <= TOL[w.dtype], (layer, err)
            checked[layer] = err
    assert sc.sess.check() == 0
    assert all(v is not None for v in checked.values())


@pytest.mark.gpu
def test_swa_transfer_round_trip_and_ring_release():
    w = wl.swa_transfer()
    B = len(w.cached)
    W, P = w.window, w.page_size
    sc = Scenario(w.n_q_heads, w.n_kv_heads, w.head_dim, P, W, w.dtype, w.cached,
                  layer_kinds=w.layer_kinds, seed=w.seed, extra_tokens=4 * 64 + 8, swa_pages=B * 6 + 100)
    n_layers = len(w.layer_kinds)
    lens = sc.ora.seq_len[:B].copy()
    off, nbytes = window_offsets(sc.sess, 0, lens, W)
    d_off = torch.as_tensor(off, device="cuda")
    n = int(off[-1]) * 2 * w.n_kv_heads * w.head_dim
    assert nbytes == 2 * n
    # only in-window tokens move: n_s = min(L_s, W) per sequence
    assert int(off[-1]) == int(np.minimum(lens, W).sum())
    host = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in range(n_layers)]
    for layer in range(n_layers):
        sc.sess.gather(layer, d_off, B, host[layer])
    assert sc.sess.check() == 0
    for layer in (0, n_layers - 1):
        exp = oracle.swa_pack(raw_host(sc.sess.k[layer]), raw_host(sc.sess.v[layer]), sc.ora.swa_bt, lens, W)
        assert np.array_equal(raw_host(host[layer]), exp), layer
    # evict the SWA segments (the Full segment stays) and give the windows
    # new pages: the dropped pages go to the tail of the free list, the
    # restored ones come from its head
    old = sc.ora.swa_bt.copy()
    assert sc.sess.swa_drop(range(B)) == sc.ora.swa_drop(range(B))
    assert sc.sess.swa_restore(range(B)) == sc.ora.swa_restore(range(B))
    sc.assert_tables_equal()
    live = sc.ora.swa_bt >= 0
    assert np.array_equal(live, old >= 0)
    assert (sc.ora.swa_bt[live] != old[live]).mean() > 0.9
    sc.sess.sync()
    before0 = (raw_host(sc.sess.k[0]).copy(), raw_host(sc.sess.v[0]).copy())
    for layer in range(n_layers):
        sc.sess.scatter(layer, d_off, B, host[layer])
    assert sc.sess.check() == 0
    # the pool now holds what the oracle's unpack writes
    oracle.swa_unpack(raw_host(host[0]), before0[0], before0[1], sc.ora.swa_bt, lens, W)
    assert np.array_equal(raw_host(sc.sess.k[0]), before0[0])
    assert np.array_equal(raw_host(sc.sess.v[0]), before0[1])
    again = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for layer in range(n_layers):
        sc.sess.gather(layer, d_off, B, again)
        assert sc.sess.check() == 0
        assert torch.equal(again.view(torch.int16).cpu(), host[layer].view(torch.int16)), layer
    # ring release every 64 decode tokens keeps the SWA pool at the window level
    for _ in range(4):
        for _ in range(64):
            sc.reserve(range(B), [1] * B)
        assert max(sc.ora.live_swa_pages(s) for s in range(B)) <= math.ceil((W + 64) / P) + 1
        sc.release(range(B))
        assert max(sc.ora.live_swa_pages(s) for s in range(B)) <= math.ceil(W / P) + 1
    sc.sess.sync()
    sc.assert_tables_equal(device=True)
