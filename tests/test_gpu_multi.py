"""Multi-token decode parity: hswa_decode_multi (GPU) against the float64 oracle.

Each case reserves n_tok new tokens per sequence, appends their K/V, and
runs one decode over all n_tok query tokens of every sequence: token w sits
at position L - n_tok + w and sees keys up to itself (Full) or the W keys
ending at itself (SWA). Every output element is compared with the oracle
evaluated at those positions (bf16: max abs 2e-2, fp32: 1e-5)."""
import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
import hybrid_sliding_window_dual_gb300 as H
from scenario import Scenario, TOL, device_out, max_err, raw_host

FULL, SWA = wl.KIND_FULL, wl.KIND_SWA


def run_multi_step(sc, n_tok, seed, samples=None, expect_kernel=None):
    B = len(sc.cached)
    samples = list(range(B)) if samples is None else samples
    full_slots, swa_slots = sc.reserve(range(B), [n_tok] * B)
    sc.sess.sync()
    errs = {}
    for layer, kind in enumerate(sc.kinds):
        slots = full_slots if kind == FULL else swa_slots
        kn = sc.gen((B * n_tok, sc.hkv, sc.d), seed + 10 * layer + 1)
        vn = sc.gen((B * n_tok, sc.hkv, sc.d), seed + 10 * layer + 2)
        sc.sess.append(layer, sc.to_dev(kn), sc.to_dev(vn), torch.as_tensor(slots, device="cuda"))
        q = sc.gen((B * n_tok, sc.hq, sc.d), seed + 10 * layer)
        qd = sc.to_dev(q)
        o = torch.full_like(qd, float("nan"))
        sc.sess.decode_multi(layer, qd, o, B, n_tok, sc.scale)
        assert sc.sess.check() == 0
        if expect_kernel:
            assert H.hswa_last_kernel() in expect_kernel
        snap = sc.snapshot(layer, samples)
        lens = sc.ora.seq_len[samples]
        rows = (np.asarray(samples)[:, None] * n_tok + np.arange(n_tok)[None, :]).reshape(-1)
        q_seq = np.repeat(np.arange(len(samples)), n_tok)
        q_pos = (lens[:, None] - n_tok + np.arange(n_tok)[None, :]).reshape(-1)
        exp = oracle.attention(raw_host(q)[rows], snap[0], snap[1], snap[2], q_seq, q_pos, sc.window(layer),
                               sc.scale)
        got = device_out(o)[rows]
        assert np.isfinite(got).all()
        errs[kind] = max_err(got, exp)
        assert errs[kind] <= TOL[sc.dtype], (kind, n_tok, errs[kind])
    return errs


FAST = ("decode_mma_bf16_d128", "decode_tc_bf16_d128")


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [1, 2, 3, 4, 5, 7, 8, 9, 12, 15, 16])
def test_multi_token_decode_ragged_lengths(n_tok):
    # lengths around page edges and the window (W = 128, P = 64), one empty
    # sequence whose first new token sees only itself
    cached = [0, 1, 61, 62, 63, 64, 125, 126, 127, 128, 129, 191, 700, 3000]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=7, extra_tokens=16)
    run_multi_step(sc, n_tok, seed=300 + n_tok, expect_kernel=FAST)
    if n_tok > 3:  # past what the mma.sync kernel serves
        assert H.hswa_last_kernel() == "decode_tc_bf16_d128"


@pytest.mark.gpu
def test_multi_token_decode_steps_with_release():
    """Verification steps of 3 tokens; release before each reserve."""
    cached = [5, 130, 255, 1000, 2047]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=8, extra_tokens=64)
    for step in range(12):
        sc.release(range(len(cached)))
        sc.sess.sync()
        run_multi_step(sc, 3, seed=400 + step)


@pytest.mark.gpu
def test_multi_token_one_equals_single_token_decode_bitwise():
    """n_tok = 1 runs the same kernel as hswa_decode: identical bytes."""
    cached = [3, 64, 300, 5000]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=9)
    B = len(cached)
    full_slots, swa_slots = sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    for layer, kind in enumerate(sc.kinds):
        q = sc.to_dev(sc.gen((B, sc.hq, sc.d), 70 + layer))
        a = torch.empty_like(q)
        b = torch.empty_like(q)
        sc.sess.decode(layer, q, a, B, sc.scale)
        sc.sess.decode_multi(layer, q, b, B, 1, sc.scale)
        assert sc.sess.check() == 0
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(4, 1, 64, 16, wl.DTYPE_F32), (16, 4, 128, 64, wl.DTYPE_BF16)])
def test_multi_token_generic_path(shape):
    hq, hkv, d, P, dtype = shape
    cached = [0, 3, 17, 100, 300]
    sc = Scenario(hq, hkv, d, P, 40, dtype, cached, seed=11, extra_tokens=16)
    run_multi_step(sc, 4, seed=500)


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [4, 8, 16])
def test_multi_token_full_size_batch_sampled(n_tok):
    """The decode_batch shape (Hq 64, Hkv 8, d 128, P 64, W 128) with 256
    sequences of mixed lengths, n_tok tokens each; oracle on sampled
    sequences. Most (sequence, kv head) segments are cut between CTAs here,
    so the partial records and their merge are exercised."""
    rng = np.random.default_rng(12)
    cached = list(rng.integers(1, 16384, 256))
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=12, permute=True, chunk=8192)
    samples = sorted(set(rng.integers(0, 256, 12).tolist()) | {0, 255})
    run_multi_step(sc, n_tok, seed=600 + n_tok, samples=samples)


@pytest.mark.gpu
@pytest.mark.parametrize("T", [3, 6, 12])
def test_multi_token_steps_large_max_jumps(T):
    """Scores whose row max jumps by far more than 2^8 between pages (the
    lazy rescale of O in the tensor-core kernel must fire), several
    verification steps of T tokens with releases in between."""
    cached = [40, 300, 1500, 4000]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=14, extra_tokens=64)
    B = len(cached)
    for step in range(3):
        sc.release(range(B))
        sc.sess.sync()
        full_slots, swa_slots = sc.reserve(range(B), [T] * B)
        sc.sess.sync()
        for layer, kind in enumerate(sc.kinds):
            slots = full_slots if kind == FULL else swa_slots
            # keys grow in magnitude with position: later pages win by far
            kn = sc.gen((B * T, sc.hkv, sc.d), 900 + 10 * step + layer)
            grow = (1.0 + torch.arange(B * T) % T).view(-1, 1, 1)
            kn = (kn.float() * grow).to(kn.dtype)
            vn = sc.gen((B * T, sc.hkv, sc.d), 950 + 10 * step + layer)
            sc.sess.append(layer, sc.to_dev(kn), sc.to_dev(vn), torch.as_tensor(slots, device="cuda"))
            q = sc.gen((B * T, sc.hq, sc.d), 990 + 10 * step + layer)
            q = (q.float() * 4.0).to(q.dtype)
            qd = sc.to_dev(q)
            o = torch.full_like(qd, float("nan"))
            sc.sess.decode_multi(layer, qd, o, B, T, sc.scale)
            assert sc.sess.check() == 0
            snap = sc.snapshot(layer, list(range(B)))
            lens = sc.ora.seq_len[:B]
            q_seq = np.repeat(np.arange(B), T)
            q_pos = (lens[:, None] - T + np.arange(T)[None, :]).reshape(-1)
            exp = oracle.attention(raw_host(q), snap[0], snap[1], snap[2], q_seq, q_pos, sc.window(layer), sc.scale)
            got = device_out(o)
            assert np.isfinite(got).all()
            assert max_err(got, exp) <= TOL[sc.dtype], (kind, step, max_err(got, exp))


@pytest.mark.gpu
def test_multi_token_rejects_bad_token_counts_and_small_workspace():
    cached = [10, 20]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=13)
    q = sc.to_dev(sc.gen((2 * 8, sc.hq, sc.d), 1))
    o = torch.empty_like(q)
    ws = sc.sess.workspace(2, 8)
    for n_tok in (0, H.HSWA_DECODE_MAX_TOKENS + 1):
        assert H.hswa_decode_multi_workspace_size(sc.sess.pool, 2, n_tok) == 0
        with pytest.raises(H.HswaError) as e:
            H.hswa_decode_multi(sc.sess.pool, sc.sess.layers[0], q, o, sc.sess.bt(0), sc.sess.d_seq_len, 2, n_tok,
                                sc.scale, ws, ws.numel())
        assert e.value.status == H.HSWA_ERR_INVALID_ARG
    # 8 tokens with only the bytes a 1-token decode needs
    small = H.hswa_decode_multi_workspace_size(sc.sess.pool, 2, 1)
    assert H.hswa_decode_multi_workspace_size(sc.sess.pool, 2, 8) > small
    with pytest.raises(H.HswaError) as e:
        H.hswa_decode_multi(sc.sess.pool, sc.sess.layers[0], q, o, sc.sess.bt(0), sc.sess.d_seq_len, 2, 8,
                            sc.scale, ws, small)
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    assert sc.sess.check() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [3, 8, 16])
def test_multi_token_positions_before_the_sequence_start(n_tok):
    """Sequences shorter than n_tok: query token w sits at t = L - n_tok + w,
    and a token with t < 0 has no key to attend and gets o = 0; the others
    match the oracle at their positions (both kernels)."""
    cached = [0, 1, 2, 5, 70]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=15, extra_tokens=16)
    B = len(cached)
    full_slots, swa_slots = sc.reserve(range(B), [1] * B)  # L = cached + 1
    sc.sess.sync()
    lens = sc.ora.seq_len[:B]
    assert (lens < n_tok).any()
    for layer, kind in enumerate(sc.kinds):
        slots = full_slots if kind == FULL else swa_slots
        kn = sc.gen((B, sc.hkv, sc.d), 1100 + layer)
        vn = sc.gen((B, sc.hkv, sc.d), 1110 + layer)
        sc.sess.append(layer, sc.to_dev(kn), sc.to_dev(vn), torch.as_tensor(slots, device="cuda"))
        q = sc.gen((B * n_tok, sc.hq, sc.d), 1120 + layer)
        o = torch.full_like(sc.to_dev(q), float("nan"))
        sc.sess.decode_multi(layer, sc.to_dev(q), o, B, n_tok, sc.scale)
        assert sc.sess.check() == 0
        got = device_out(o)
        pos = (lens[:, None] - n_tok + np.arange(n_tok)[None, :]).reshape(-1)
        seq = np.repeat(np.arange(B), n_tok)
        before = pos < 0
        assert np.all(got[before] == 0.0)
        snap = sc.snapshot(layer, list(range(B)))
        exp = oracle.attention(raw_host(q)[~before], snap[0], snap[1], snap[2], seq[~before], pos[~before],
                               sc.window(layer), sc.scale)
        assert max_err(got[~before], exp) <= TOL[sc.dtype], (kind, n_tok)


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [2, 8])
def test_multi_token_bad_table_entries_set_bounds_and_skip(n_tok):
    """Invalid block-table entries inside the key range (the first page of a
    segment, a page past the pool, every page of one sequence) are skipped,
    the call reports HSWA_ERR_BOUNDS and the output stays finite."""
    cached = [300, 300, 60]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=16, extra_tokens=16)
    B = len(cached)
    sc.reserve(range(B), [n_tok] * B)
    sc.sess.sync()
    sc.sess.d_full_bt[0, 0] = -1
    sc.sess.d_full_bt[1, 3] = 1 << 30
    sc.sess.d_full_bt[2, 0] = -1
    sc.sess.d_full_bt[2, 1] = -1
    q = sc.to_dev(sc.gen((B * n_tok, 64, 128), 1))
    o = torch.full_like(q, float("nan"))
    sc.sess.decode_multi(0, q, o, B, n_tok, sc.scale)
    assert sc.sess.check() == H.HSWA_ERR_BOUNDS
    assert sc.sess.check() == 0
    assert torch.isfinite(o.float()).all()
    assert torch.equal(o[2 * n_tok:].float(), torch.zeros_like(o[2 * n_tok:].float()))  # no key left


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [3, 8, 16])
def test_multi_token_decode_window_shorter_than_the_draft(n_tok):
    """A window of 8 keys (W < n_tok for the longer drafts): each token's
    keys end at itself and start W - 1 before it, so the first drafts fall
    out of the later tokens' windows; both kernels, ragged lengths."""
    cached = [0, 5, 60, 63, 64, 200, 1000]
    sc = Scenario(64, 8, 128, 64, 8, wl.DTYPE_BF16, cached, seed=17, extra_tokens=16)
    run_multi_step(sc, n_tok, seed=1700 + n_tok, expect_kernel=FAST)


@pytest.mark.gpu
def test_multi_token_empty_batch_is_a_no_op():
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, [10], seed=18)
    q = torch.zeros(0, 64, 128, dtype=torch.bfloat16, device="cuda")
    for n_tok in (2, 8, 16):
        sc.sess.decode_multi(0, q, q, 0, n_tok, sc.scale)
    assert sc.sess.check() == 0


@pytest.mark.gpu
def test_multi_token_largest_batch_the_combine_grid_takes():
    """n_seqs x n_tok up to 65535 rows (the merge kernel's grid rows): 4095
    short sequences of 16 tokens, oracle on samples (the refusal past the
    limit is checked without a GPU in test_abi.py)."""
    rng = np.random.default_rng(19)
    cached = list(rng.integers(0, 150, 4095))
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=19, extra_tokens=16, chunk=4096)
    run_multi_step(sc, 16, seed=1900, samples=[0, 1, 2047, 4093, 4094], expect_kernel=FAST)
