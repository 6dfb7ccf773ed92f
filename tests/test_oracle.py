"""Pins for the CPU oracle (no GPU).

The oracle is checked here against things other than itself:
* a library routine (torch scaled_dot_product_attention in float64 on a
  dense copy of the paged data) for Full and sliding-window masks;
* closed forms: one key gives that key's value, equal logits give the
  plain mean of the values in the key set, huge logits give the arg-max
  value, W >= L makes an SWA layer equal a Full layer;
* pool invariants and closed-form page counts for reserve / release;
* the layer layout and ratios the MiMo-V2.5 page prints (golden file);
* dense slicing for the in-window pack, and a pack/unpack round trip.
A final test compiles deliberately broken copies of the oracle source and
checks that each one fails at least one of these pins.
"""
import json
import math
import os
import re
import subprocess
import sys

import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
from oracle import DualPool, NoSpace

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def paged_from_dense(dense, page_size, page_of):
    """Place dense [S][Hkv][Lmax][d] rows into a pool [pages][Hkv][P][d]
    with logical page p of sequence s stored at physical page page_of[s][p]."""
    S, hkv, lmax, d = dense.shape
    n_lp = -(-lmax // page_size)
    pages = int(page_of.max()) + 1
    pool = np.zeros((pages, hkv, page_size, d), dense.dtype)
    for s in range(S):
        for p in range(n_lp):
            rows = dense[s, :, p * page_size:(p + 1) * page_size, :]
            pool[page_of[s, p], :, :rows.shape[1], :] = rows
    return pool


def random_case(seed, S=3, hq=8, hkv=2, d=16, P=4, lmax=37):
    rng = np.random.default_rng(seed)
    n_lp = -(-lmax // P)
    perm = rng.permutation(S * n_lp + 5)[:S * n_lp].reshape(S, n_lp).astype(np.int32)
    k = rng.standard_normal((S, hkv, lmax, d)).astype(np.float32)
    v = rng.standard_normal((S, hkv, lmax, d)).astype(np.float32)
    kp = paged_from_dense(k, P, perm)
    vp = paged_from_dense(v, P, perm)
    return k, v, kp, vp, perm


def sdpa_reference(q, k, v, s, positions, window, scale, hq):
    """torch SDPA (float64) over a dense copy: q [n][Hq][d] for sequence s."""
    hkv = k.shape[1]
    kk = torch.from_numpy(k[s]).double().repeat_interleave(hq // hkv, dim=0)  # [Hq][L][d]
    vv = torch.from_numpy(v[s]).double().repeat_interleave(hq // hkv, dim=0)
    qq = torch.from_numpy(q).double().permute(1, 0, 2)  # [Hq][n][d]
    L = k.shape[2]
    j = torch.arange(L)[None, :]
    t = torch.as_tensor(positions)[:, None]
    mask = j <= t
    if window > 0:
        mask &= j > t - window
    out = torch.nn.functional.scaled_dot_product_attention(
        qq[None], kk[None], vv[None], attn_mask=mask[None, None], scale=scale)
    return out[0].permute(1, 0, 2).numpy()


# ------------------------------------------------ pins as reusable checks
def pin_sdpa(lib=None):
    hq, hkv, d, P = 8, 2, 16, 4
    k, v, kp, vp, bt = random_case(1, hq=hq, hkv=hkv, d=d, P=P)
    rng = np.random.default_rng(7)
    worst = 0.0
    for window in (0, 1, 5, 9, 64):
        for s in range(k.shape[0]):
            pos = np.array([0, 3, 4, 17, 36], np.int64)
            q = rng.standard_normal((len(pos), hq, d)).astype(np.float32)
            got = oracle.attention(q, kp, vp, bt, np.full(len(pos), s), pos, window,
                                   1 / math.sqrt(d), lib=lib)
            ref = sdpa_reference(q, k, v, s, pos, window, 1 / math.sqrt(d), hq)
            worst = max(worst, float(np.abs(got - ref).max()))
    return worst < 1e-12, worst


def pin_single_key(lib=None):
    k, v, kp, vp, bt = random_case(2)
    ok = True
    for s in range(k.shape[0]):
        q = np.random.default_rng(s).standard_normal((2, 8, 16)).astype(np.float32)
        # Full layer at t = 0, and an SWA layer with W = 1 at t = 20
        o = oracle.attention(q, kp, vp, bt, [s, s], [0, 20], 0, 0.25, lib=lib)
        o1 = oracle.attention(q, kp, vp, bt, [s, s], [20, 20], 1, 0.25, lib=lib)
        g = np.arange(8) * 2 // 8
        ok &= np.array_equal(o[0], v[s, g, 0, :])
        ok &= np.array_equal(o1[0], v[s, g, 20, :])
    return bool(ok), None


def pin_equal_logits(lib=None):
    """q = 0: every key has the same logit, so o is the plain mean of the
    values in the key set; this fixes both window edges."""
    k, v, kp, vp, bt = random_case(3)
    worst = 0.0
    for window in (0, 1, 2, 7, 128):
        for t in (0, 5, 11, 36):
            q = np.zeros((1, 8, 16), np.float32)
            o = oracle.attention(q, kp, vp, bt, [1], [t], window, 0.3, lib=lib)
            lo = max(0, t - window + 1) if window else 0
            g = np.arange(8) * 2 // 8
            ref = v[1, g, lo:t + 1, :].astype(np.float64).mean(axis=1)
            worst = max(worst, float(np.abs(o[0] - ref).max()))
    return worst < 1e-13, worst


def pin_large_logits(lib=None):
    """scale 1e4: the softmax is one-hot at the largest logit (no overflow)."""
    k, v, kp, vp, bt = random_case(4)
    q = np.random.default_rng(9).standard_normal((1, 8, 16)).astype(np.float32)
    t = 30
    o = oracle.attention(q, kp, vp, bt, [2], [t], 0, 1e4, lib=lib)
    ok = np.isfinite(o).all()
    for h in range(8):
        g = h * 2 // 8
        s = k[2, g, :t + 1, :].astype(np.float64) @ q[0, h].astype(np.float64)
        ok &= np.allclose(o[0, h], v[2, g, int(np.argmax(s)), :], atol=1e-12, rtol=0)
    return bool(ok), None


def pin_window_covers_all(lib=None):
    k, v, kp, vp, bt = random_case(5)
    q = np.random.default_rng(3).standard_normal((4, 8, 16)).astype(np.float32)
    pos = [36, 20, 3, 0]
    full = oracle.attention(q, kp, vp, bt, [0, 1, 2, 0], pos, 0, 0.25, lib=lib)
    swa = oracle.attention(q, kp, vp, bt, [0, 1, 2, 0], pos, 37, 0.25, lib=lib)
    return bool(np.array_equal(full, swa)), None


ATTENTION_PINS = [pin_sdpa, pin_single_key, pin_equal_logits, pin_large_logits,
                  pin_window_covers_all]


@pytest.mark.parametrize("pin", ATTENTION_PINS, ids=lambda f: f.__name__)
def test_attention_pin(pin):
    ok, detail = pin()
    assert ok, detail


def test_attention_bf16_inputs_are_exact():
    """bf16 inputs are widened exactly: the same values given as fp32 give
    the same float64 result bit for bit."""
    k, v, kp, vp, bt = random_case(6)
    q = np.random.default_rng(1).standard_normal((3, 8, 16)).astype(np.float32)
    to_bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    qb, kb, vb = to_bf(q), to_bf(kp), to_bf(vp)
    o_b = oracle.attention(qb, kb, vb, bt, [0, 1, 2], [36, 10, 2], 5, 0.25)
    o_f = oracle.attention(qb.float(), kb.float(), vb.float(), bt, [0, 1, 2], [36, 10, 2], 5, 0.25)
    assert np.array_equal(o_b, o_f)


def test_attention_rejects_released_page():
    k, v, kp, vp, bt = random_case(7)
    bt = bt.copy()
    bt[0, 2] = -1
    q = np.zeros((1, 8, 16), np.float32)
    with pytest.raises(IndexError):
        oracle.attention(q, kp, vp, bt, [0], [20], 0, 0.25)
    # an SWA query whose window avoids page 2 does not touch it
    oracle.attention(q, kp, vp, bt, [0], [30], 4, 0.25)


# --------------------------------------------------------- bookkeeping
def test_reserve_identity_order_gives_consecutive_slots():
    pool = DualPool(window=128, page_size=16, full_pages=64, swa_pages=64, max_seqs=4,
                    max_pages_per_seq=32)
    f, s = pool.reserve([2], [200])
    assert np.array_equal(f, np.arange(200)) and np.array_equal(s, np.arange(200))
    f2, s2 = pool.reserve([0, 2], [3, 5])
    # seq 0 takes page 13, then seq 2 continues its page 12 (200 % 16 = 8)
    assert f2.tolist() == [208, 209, 210] + [200, 201, 202, 203, 204]


def test_reserve_follows_free_order():
    P = 8
    order = wl.permutation(40, 11)
    pool = DualPool(128, P, 40, 40, 2, 16, full_free_order=order, swa_free_order=order[::-1])
    f, s = pool.reserve([0, 1], [20, 9])
    pages_f = list(order[:3]) + list(order[3:5])
    pages_s = list(order[::-1][:3]) + list(order[::-1][3:5])
    exp_f = [pages_f[t // P] * P + t % P for t in range(20)] + \
            [pages_f[3 + t // P] * P + t % P for t in range(9)]
    exp_s = [pages_s[t // P] * P + t % P for t in range(20)] + \
            [pages_s[3 + t // P] * P + t % P for t in range(9)]
    assert f.tolist() == exp_f and s.tolist() == exp_s


def snapshot(pool):
    return (list(pool.full_free), list(pool.swa_free), pool.full_bt.copy(),
            pool.swa_bt.copy(), pool.seq_len.copy())


def same(a, b):
    return all(np.array_equal(np.asarray(x), np.asarray(y)) for x, y in zip(a, b))


@pytest.mark.parametrize("short", ["full", "swa"])
def test_reserve_is_all_or_nothing(short):
    pool = DualPool(128, 16, 10 if short == "full" else 40, 40 if short == "full" else 10,
                    4, 64)
    pool.reserve([0], [100])  # 7 pages of each
    before = snapshot(pool)
    with pytest.raises(NoSpace):
        pool.reserve([1, 3], [16, 40])  # needs 1 + 3 more pages of each
    assert same(before, snapshot(pool))


@pytest.mark.parametrize("L", [0, 1, 127, 128, 129, 191, 192, 193, 1000, 4096])
def test_release_count_closed_form(L):
    W, P = 128, 64
    pool = DualPool(W, P, 128, 128, 1, 128)
    if L:
        pool.reserve([0], [L])
    n_pages = -(-L // P)
    freed = pool.swa_release([0])
    assert freed == max(0, (L - W) // P)
    assert pool.live_swa_pages(0) == n_pages - freed
    for p in np.nonzero(pool.swa_bt[0] >= 0)[0]:
        assert (p + 1) * P > L - W and p * P < L  # page meets [L-W, L)
    assert pool.swa_release([0]) == 0  # idempotent


def check_invariants(pool, seqs):
    live_f = pool.full_bt[pool.full_bt >= 0]
    live_s = pool.swa_bt[pool.swa_bt >= 0]
    assert len(set(live_f.tolist())) == live_f.size
    assert len(set(live_s.tolist())) == live_s.size
    assert live_f.size + len(pool.full_free) == pool.full_pages
    assert live_s.size + len(pool.swa_free) == pool.swa_pages
    assert not set(live_f.tolist()) & set(pool.full_free)
    assert not set(live_s.tolist()) & set(pool.swa_free)
    for s in seqs:
        L = int(pool.seq_len[s])
        assert pool.live_full_pages(s) == -(-L // pool.P)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_swa_pool_stays_at_window_or_chunk_level(seed):
    """Random decode steps and prefill chunks; release after each chunk and
    every 64 decode tokens. Live SWA pages per sequence stay within
    ceil(W/P)+1 after a release and ceil((W+C)/P)+1 between releases."""
    rng = np.random.default_rng(seed)
    W, P, S = 128, 16, 5
    pool = DualPool(W, P, 4000, 400, S, 256,
                    full_free_order=wl.permutation(4000, seed),
                    swa_free_order=wl.permutation(400, seed + 1))
    since = np.zeros(S, np.int64)
    for _ in range(300):
        s = int(rng.integers(S))
        chunk = int(rng.choice([1, 1, 1, 37, 100]))
        if pool.seq_len[s] + chunk > 256 * P:
            continue
        pool.reserve([s], [chunk])
        since[s] += chunk
        bound = math.ceil((W + since[s]) / P) + 1
        assert pool.live_swa_pages(s) <= bound
        if chunk > 1 or since[s] >= 64:
            pool.swa_release([s])
            since[s] = 0
            assert pool.live_swa_pages(s) <= math.ceil(W / P) + 1
        check_invariants(pool, range(S))
    pool.seq_free([0, 3])
    check_invariants(pool, range(S))
    assert pool.seq_len[0] == 0 and pool.live_swa_pages(3) == 0


def test_golden_layer_layout_and_ratios():
    """The MiMo-V2.5-Pro numbers: 70 layers, 10 Full + 60 SWA, W 128; the
    dual pool holds about 1/7 of the single-pool KV and so about 7x the
    capacity, at long context."""
    g = json.load(open(os.path.join(GOLDEN, "mimo_v25_pro_layout.json")))
    w = wl.hybrid70(n_seqs=2, context=131072)
    kinds = w.layer_kinds
    assert len(kinds) == g["n_layers"]
    assert kinds.count(wl.KIND_FULL) == g["n_full_layers"]
    assert kinds.count(wl.KIND_SWA) == g["n_swa_layers"]
    assert w.window == g["window"]
    N, P = 131072, w.page_size
    pool = DualPool(w.window, P, 2 * N // P + 8, 2 * N // P + 8, 2, N // P + 2)
    for s in (0, 1):
        for start in range(0, N, 4096):  # chunked prefill with release per chunk
            pool.reserve([s], [4096])
            pool.swa_release([s])
    per_tok = 2 * w.n_kv_heads * w.head_dim * 2
    dual = oracle.kv_bytes(pool, kinds, [0, 1], per_tok)
    single = len(kinds) * 2 * N * per_tok
    ratio = dual / single
    a, b = g["approx_kv_ratio"]
    assert abs(ratio - a / b) / (a / b) < 0.05, ratio
    assert abs(1 / ratio - g["approx_capacity_gain"]) / g["approx_capacity_gain"] < 0.05
    # the exact page-granular value: 10/70 + 60/70 * (live SWA tokens) / N
    live = pool.live_swa_pages(0) * P
    assert math.isclose(ratio, 10 / 70 + 60 / 70 * live / N, rel_tol=1e-12)


# ---------------------------------------------------------------- pack
def test_pack_equals_dense_window_slices():
    rng = np.random.default_rng(0)
    S, hkv, d, P, W = 4, 2, 8, 4, 6
    lens = np.array([1, 6, 13, 40])
    k = rng.standard_normal((S, hkv, 40, d)).astype(np.float32)
    v = rng.standard_normal((S, hkv, 40, d)).astype(np.float32)
    pool = DualPool(W, P, 64, 64, S, 10, swa_free_order=wl.permutation(64, 3))
    pool.reserve(range(S), lens)
    n_lp = 10
    swa_bt = pool.swa_bt.copy()
    page_of = np.where(swa_bt >= 0, swa_bt, 63)[:, :n_lp]
    kp = paged_from_dense(np.pad(k, ((0, 0), (0, 0), (0, 0), (0, 0))), P, page_of)
    vp = paged_from_dense(v, P, page_of)
    pool.swa_release(range(S))
    packed = oracle.swa_pack(kp, vp, pool.swa_bt, lens, W)
    expect = []
    for s in range(S):
        n = min(lens[s], W)
        expect.append(k[s, :, lens[s] - n:lens[s], :].reshape(-1))
        expect.append(v[s, :, lens[s] - n:lens[s], :].reshape(-1))
    assert np.array_equal(packed, np.concatenate(expect))
    assert packed.size == 2 * hkv * d * sum(min(L, W) for L in lens)


def test_pack_unpack_round_trip_through_new_pages():
    rng = np.random.default_rng(1)
    S, hkv, d, P, W = 3, 2, 8, 4, 9
    lens = [30, 5, 17]
    pool = DualPool(W, P, 64, 32, S, 16, swa_free_order=wl.permutation(32, 5))
    pool.reserve(range(S), lens)
    pool.swa_release(range(S))
    kp = rng.standard_normal((32, hkv, P, d)).astype(np.float32)
    vp = rng.standard_normal((32, hkv, P, d)).astype(np.float32)
    packed = oracle.swa_pack(kp, vp, pool.swa_bt, lens, W)
    old = pool.swa_bt.copy()
    pool.swa_drop(range(S))
    assert (pool.swa_bt < 0).all()
    pool.reserve([0], [0])
    # take a few pages first so the restored pages differ from the old ones
    pool.swa_free.rotate(-7)
    n = pool.swa_restore(range(S))
    assert n == int((old >= 0).sum())
    assert not np.array_equal(old, pool.swa_bt)
    kp2 = np.zeros_like(kp)
    vp2 = np.zeros_like(vp)
    oracle.swa_unpack(packed, kp2, vp2, pool.swa_bt, lens, W)
    again = oracle.swa_pack(kp2, vp2, pool.swa_bt, lens, W)
    assert np.array_equal(packed.view(np.uint32), again.view(np.uint32))


def test_append_then_read_through_table():
    P, hkv, d = 4, 2, 3
    pool = DualPool(8, P, 16, 16, 2, 8, full_free_order=wl.permutation(16, 2))
    f, _ = pool.reserve([0, 1], [6, 3])
    kp = np.zeros((16, hkv, P, d), np.float32)
    new = np.arange(9 * hkv * d, dtype=np.float32).reshape(9, hkv, d)
    oracle.append_kv(kp, new, f)
    for i, (s, t) in enumerate([(0, t) for t in range(6)] + [(1, t) for t in range(3)]):
        assert np.array_equal(kp[pool.full_bt[s, t // P], :, t % P, :], new[i])


# ------------------------------------------------------------ mutations
MUTATIONS = {
    "window_off_by_one": ("t - window + 1 > 0) ? t - window + 1", "t - window > 0) ? t - window"),
    "gqa_interleaved": ("(((int64_t)h * n_kv_heads) / n_q_heads)", "(h % n_kv_heads)"),
    "row_in_page": ("j % page_size) * head_dim", "(j + 1) % page_size) * head_dim"),
    "scale_dropped": ("score[j - lo] = scale * dot", "score[j - lo] = dot"),
    "no_max_subtract": ("exp(score[j] - m)", "exp(score[j])"),
    "causal_excludes_self": ("j <= t; ++j", "j < t; ++j"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "hswa_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new)
    c = tmp_path / "mut.c"
    so = tmp_path / "mut.so"
    c.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"])
    # run the pins in a child process: a broken oracle may also crash
    code = ("import sys; sys.path[:0] = [%r, %r]; import oracle, test_oracle as t\n"
            "lib = oracle.load_library(%r)\n"
            "for pin in t.ATTENTION_PINS:\n"
            "    try:\n"
            "        ok, _ = pin(lib)\n"
            "    except Exception:\n"
            "        ok = False\n"
            "    print(pin.__name__, 'ok' if ok else 'FAILED')\n"
            % (os.path.dirname(os.path.dirname(__file__)), os.path.dirname(__file__), str(so)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    caught = r.returncode != 0 or "FAILED" in r.stdout
    assert caught, "no pin caught mutation %s:\n%s" % (name, r.stdout)
