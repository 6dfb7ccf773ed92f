"""Layer-by-layer reload of offloaded SWA windows, overlapped with attention
(MiMo page, Sec. 2.1: asynchronous layer-by-layer pulling).

Two identical dual pools run the same decode step over a 14-layer hybrid
model (Full at every 7th layer). Pool b first offloads every SWA window to
pinned host memory, evicts the SWA segments, gives the windows new pages and
overwrites the SWA pools with a sentinel; its step then reloads each layer's
window on a side stream while earlier layers compute, waiting only right
before each SWA layer. Every layer's output must equal pool a's bit for bit.

The oracle checks the reload itself, independently of pool a: each gathered
window equals oracle.swa_pack of the pool it came from; after the step, each
reloaded SWA pool equals the poisoned pool with oracle.swa_unpack of that
window (at the pages the restore handed out) and the step's appended token,
bit for bit; and every layer's output of the reloaded step matches
oracle.attention over those pools (max abs 2e-2).
"""
import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
from hybrid_sliding_window_dual_gb300.session import LayerwiseReload
from scenario import Scenario, TOL, device_out, raw_host, window_offsets


def make(seed):
    kinds = tuple(wl.KIND_FULL if i % 7 == 6 else wl.KIND_SWA for i in range(14))
    cached = [5, 127, 128, 129, 700, 2000, 4095, 64, 1, 300, 3333, 256]
    return Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, layer_kinds=kinds, seed=seed, permute=True,
                    swa_pages=len(cached) * 8 + 40)


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["serial", "direct", "staged"])
def test_layerwise_reload_step_equals_resident_step(mode):
    a, b = make(61), make(61)
    B = len(a.cached)
    kinds = a.kinds
    swa_layers = [i for i, k in enumerate(kinds) if k == wl.KIND_SWA]
    # offload pool b's windows, evict, restore to new pages, poison the pools
    lens = b.ora.seq_len[:B].copy()
    off, nbytes = window_offsets(b.sess, swa_layers[0], lens, b.W)
    d_off = torch.as_tensor(off, device="cuda")
    n = nbytes // 2
    host = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for _ in swa_layers]
    # host copies of every pool of b before the offload (the oracle's inputs)
    pools = {ly: [raw_host(b.sess.k[ly]).copy(), raw_host(b.sess.v[ly]).copy()] for ly in range(len(kinds))}
    packed = {ly: oracle.swa_pack(pools[ly][0], pools[ly][1], b.ora.swa_bt, lens, b.W) for ly in swa_layers}
    for buf, ly in zip(host, swa_layers):
        b.sess.gather(ly, d_off, B, buf)
    assert b.sess.check() == 0
    for buf, ly in zip(host, swa_layers):
        assert np.array_equal(raw_host(buf), packed[ly]), ly
    assert b.sess.swa_drop(range(B)) == b.ora.swa_drop(range(B))
    assert b.sess.swa_restore(range(B)) == b.ora.swa_restore(range(B))
    b.sess.sync()
    for ly in swa_layers:
        b.sess.k[ly].fill_(7.0)
        b.sess.v[ly].fill_(-7.0)
        # the oracle's reloaded pool: the same poison, the window unpacked at
        # the restored pages
        pools[ly] = [np.full_like(pools[ly][0], 0x40E0), np.full_like(pools[ly][1], 0xC0E0)]
        oracle.swa_unpack(packed[ly], pools[ly][0], pools[ly][1], b.ora.swa_bt, lens, b.W)
    d_len_snap = b.sess.d_seq_len.clone()
    torch.cuda.synchronize()
    # the step on both pools
    outs, inputs = {}, {}
    side = torch.cuda.Stream()
    for name, sc in (("a", a), ("b", b)):
        fs, ss = sc.reserve(range(B), [1] * B)
        sc.sess.sync()
        d_fs = torch.as_tensor(fs, device="cuda")
        d_ss = torch.as_tensor(ss, device="cuda")
        events, staged = {}, None
        cur = torch.cuda.current_stream()
        if name == "b":
            side.wait_stream(cur)
            if mode == "direct":    # the scatter kernel reads pinned host memory, side stream
                events = sc.sess.reload_async(swa_layers, d_len_snap, d_off, B, host, side)
            elif mode == "serial":  # every window back before the first layer
                sc.sess.reload_async(swa_layers, d_len_snap, d_off, B, host, side)
                cur.wait_stream(side)
            else:                   # copy engines into a 3-buffer staging ring
                staging = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
                staged = LayerwiseReload(sc.sess, swa_layers, d_len_snap, d_off, B, host, side, staging)
                staged.start(cur)
        res = []
        for ly, kind in enumerate(kinds):
            q = sc.to_dev(sc.gen((B, 64, 128), 900 + ly))
            kn = sc.to_dev(sc.gen((B, 8, 128), 950 + ly))
            vn = sc.to_dev(sc.gen((B, 8, 128), 990 + ly))
            if name == "b":
                inputs[ly] = (raw_host(q), raw_host(kn), raw_host(vn), fs if kind == wl.KIND_FULL else ss)
            if ly in events:
                cur.wait_event(events[ly])
            if staged is not None:
                staged.before_layer(ly, cur)
            o = torch.empty_like(q)
            sc.sess.decode_append(ly, q, kn, vn, d_fs if kind == wl.KIND_FULL else d_ss, o, B, sc.scale)
            res.append(o)
        assert sc.sess.check() == 0
        outs[name] = res
    for ly in range(len(kinds)):
        assert torch.equal(outs["a"][ly].view(torch.int16), outs["b"][ly].view(torch.int16)), ly
    # the reloaded step against the oracle
    torch.cuda.synchronize()
    for ly, kind in enumerate(kinds):
        q, kn, vn, slots = inputs[ly]
        k_pool, v_pool = pools[ly]
        oracle.append_kv(k_pool, kn, slots)
        oracle.append_kv(v_pool, vn, slots)
        if kind == wl.KIND_SWA:
            assert np.array_equal(raw_host(b.sess.k[ly]), k_pool), ly
            assert np.array_equal(raw_host(b.sess.v[ly]), v_pool), ly
        bt = b.ora.full_bt if kind == wl.KIND_FULL else b.ora.swa_bt
        exp = oracle.attention(q, k_pool, v_pool, bt, np.arange(B), lens, b.window(ly), b.scale)
        got = device_out(outs["b"][ly])
        assert np.abs(got - exp).max() <= TOL[b.dtype], ly
