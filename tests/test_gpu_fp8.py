"""FP8 (E4M3) KV cache on the GPU against the oracle.

The cached history is seeded random E4M3 codes (no NaN pattern) with seeded
positive scales; new tokens are bf16 and quantized by hswa_append_kv. The
codes and scales the library writes must equal the oracle's quantizer bit
for bit, and hswa_decode / hswa_decode_append over the FP8 pools must match
the oracle's float64 attention over the exactly dequantized pools (max abs
2e-2, the bf16 I/O tolerance)."""
import math

import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
import hybrid_sliding_window_dual_gb300 as H
from hybrid_sliding_window_dual_gb300.session import DualPoolSession
from scenario import prefill_kernel, raw_host

FULL, SWA = wl.KIND_FULL, wl.KIND_SWA
HQ, HKV, D, P, W = 64, 8, 128, 64, 128


class Fp8Case:
    def __init__(self, cached, seed, kinds=(FULL, SWA), extra=8):
        B = len(cached)
        full_pages = sum(math.ceil((L + extra) / P) for L in cached) + 4
        swa_pages = B * (5 + math.ceil(extra / P)) + 80
        mp = max(math.ceil((L + extra) / P) for L in cached) + 1
        self.cfg = H.Config(window=W, page_size=P, n_q_heads=HQ, n_kv_heads=HKV, head_dim=D,
                            dtype=H.HSWA_DTYPE_FP8_E4M3, full_pages=full_pages, swa_pages=swa_pages, max_seqs=B,
                            max_pages_per_seq=mp)
        fo, so = wl.permutation(full_pages, seed), wl.permutation(swa_pages, seed + 1)
        self.sess = DualPoolSession(self.cfg, kinds, fo, so)
        self.ora = oracle.DualPool(W, P, full_pages, swa_pages, B, mp, fo, so)
        self.kinds, self.B, self.cached = list(kinds), B, list(cached)
        for s, L in enumerate(cached):
            for start in range(0, L, 4096):
                n = min(4096, L - start)
                a = self.sess.reserve([s], [n])
                b = self.ora.reserve([s], [n])
                assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
                assert self.sess.release([s]) == self.ora.swa_release([s])
        self.sess.sync()
        for i in range(len(kinds)):  # seeded on the device (the full-size pools hold GBs of codes)
            for t, seed_i in ((self.sess.k[i], 10), (self.sess.v[i], 20)):
                g = torch.Generator(device="cuda")
                g.manual_seed(seed * 100 + seed_i + i)
                flat = t.view(-1)
                for j in range(0, flat.numel(), 1 << 28):
                    n = min(1 << 28, flat.numel() - j)
                    mag = torch.randint(0, 0x7F, (n,), generator=g, device="cuda", dtype=torch.uint8)
                    sgn = torch.randint(0, 2, (n,), generator=g, device="cuda", dtype=torch.uint8)
                    flat[j:j + n] = mag | (sgn << 7)
            for t, seed_i in ((self.sess.ks[i], 30), (self.sess.vs[i], 40)):
                g = torch.Generator(device="cuda")
                g.manual_seed(seed * 100 + seed_i + i)
                t.copy_(0.001 + 0.01 * torch.rand(t.shape, generator=g, device="cuda"))
        torch.cuda.synchronize()
        self.host = [[x.cpu().numpy().copy() for x in (self.sess.k[i], self.sess.ks[i], self.sess.v[i],
                                                        self.sess.vs[i])] for i in range(len(kinds))]

    def table(self, layer):
        return self.ora.full_bt if self.kinds[layer] == FULL else self.ora.swa_bt


@pytest.mark.gpu
@pytest.mark.parametrize("fused", [False, True])
def test_fp8_append_and_decode_match_oracle(fused):
    cached = [0, 1, 63, 64, 65, 127, 128, 700, 3000, 9000]
    c = Fp8Case(cached, seed=71)
    B = c.B
    fs, ss = c.sess.reserve(range(B), [1] * B)
    efs, ess = c.ora.reserve(range(B), [1] * B)
    assert np.array_equal(fs, efs) and np.array_equal(ss, ess)
    c.sess.sync()
    scale = 1 / math.sqrt(D)
    for layer, kind in enumerate(c.kinds):
        slots = fs if kind == FULL else ss
        q = wl.normal((B, HQ, D), 500 + layer, wl.DTYPE_BF16)
        kn = wl.normal((B, HKV, D), 510 + layer, wl.DTYPE_BF16) * 3
        vn = wl.normal((B, HKV, D), 520 + layer, wl.DTYPE_BF16) * 0.5
        o = torch.full((B, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        ds = torch.as_tensor(slots, device="cuda")
        if fused:
            c.sess.decode_append(layer, q.cuda(), kn.cuda(), vn.cuda(), ds, o, B, scale)
        else:
            c.sess.append(layer, kn.cuda(), vn.cuda(), ds)
            c.sess.decode(layer, q.cuda(), o, B, scale)
        assert c.sess.check() == 0
        assert H.hswa_last_kernel().endswith("decode_mma_fp8_d128")
        kc, ks, vc, vs = c.host[layer]
        oracle.append_kv_fp8(kc, ks, vc, vs, kn.float().numpy(), vn.float().numpy(), slots)
        # the library's quantized rows and scales, bit for bit
        assert np.array_equal(c.sess.k[layer].cpu().numpy(), kc)
        assert np.array_equal(c.sess.v[layer].cpu().numpy(), vc)
        assert np.array_equal(c.sess.ks[layer].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(c.sess.vs[layer].cpu().numpy().view(np.uint32), vs.view(np.uint32))
        exp = oracle.attention_fp8(raw_host(q), kc, ks, vc, vs, c.table(layer), np.arange(B),
                                   c.ora.seq_len[:B] - 1, 0 if kind == FULL else W, scale)
        got = o.float().cpu().numpy()
        assert np.isfinite(got).all()
        err = float(np.abs(got - exp).max())
        assert err <= 2e-2, (layer, err)


@pytest.mark.gpu
def test_fp8_unsupported_calls_say_so():
    c = Fp8Case([100], seed=72, kinds=(SWA,))
    # prefill over an FP8 pool needs the workspace variant
    q = torch.zeros(1, HQ, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(H.HswaError) as e:
        H.hswa_prefill_chunk(c.sess.pool, c.sess.layers[0], q, q.clone(), c.sess.bt(0),
                             torch.zeros(1, dtype=torch.int32, device="cuda"),
                             torch.tensor([0, 1], dtype=torch.int32, device="cuda"), 1, 1, 1, 0.1)
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    assert c.sess.check() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("swa_first", [False, True])
def test_fp8_prefill_chunk_matches_oracle(swa_first):
    """A ragged chunk over FP8 pools: the new tokens are quantized by the
    append, the staging pass dequantizes every page the chunk reads, and the
    tensor-core kernel attends; every output row against the oracle."""
    cached = [0, 5, 63, 64, 127, 128, 129, 700, 3000]
    chunk = [1, 60, 64, 65, 128, 200, 7, 129, 300]
    kinds = (SWA, FULL) if swa_first else (FULL, SWA)
    c = Fp8Case(cached, seed=74 + swa_first, kinds=kinds, extra=max(chunk) + 8)
    B = c.B
    fs, ss = c.sess.reserve(range(B), chunk)
    efs, ess = c.ora.reserve(range(B), chunk)
    assert np.array_equal(fs, efs) and np.array_equal(ss, ess)
    c.sess.sync()
    n_tot = sum(chunk)
    q_start = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    d_prefix = torch.tensor(cached, dtype=torch.int32, device="cuda")
    d_qs = torch.as_tensor(q_start, device="cuda")
    q_seq = np.repeat(np.arange(B), chunk)
    q_pos = np.concatenate([np.arange(L, L + n) for L, n in zip(cached, chunk)])
    scale = 1 / math.sqrt(D)
    for layer, kind in enumerate(c.kinds):
        slots = fs if kind == FULL else ss
        q = wl.normal((n_tot, HQ, D), 800 + layer, wl.DTYPE_BF16)
        kn = wl.normal((n_tot, HKV, D), 810 + layer, wl.DTYPE_BF16) * 2
        vn = wl.normal((n_tot, HKV, D), 820 + layer, wl.DTYPE_BF16)
        c.sess.append(layer, kn.cuda(), vn.cuda(), torch.as_tensor(slots, device="cuda"))
        o = torch.full((n_tot, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        c.sess.prefill(layer, q.cuda(), o, d_prefix, d_qs, B, max(chunk), scale, prefix_host=np.array(cached),
                       q_start_host=q_start)
        assert c.sess.check() == 0
        assert H.hswa_last_kernel() == prefill_kernel(kind, 0 if kind == FULL else W, fp8=True)
        kc, ks, vc, vs = c.host[layer]
        oracle.append_kv_fp8(kc, ks, vc, vs, kn.float().numpy(), vn.float().numpy(), slots)
        assert np.array_equal(c.sess.k[layer].cpu().numpy(), kc)
        exp = oracle.attention_fp8(raw_host(q), kc, ks, vc, vs, c.table(layer), q_seq, q_pos,
                                   0 if kind == FULL else W, scale)
        got = o.float().cpu().numpy()
        assert np.isfinite(got).all()
        err = float(np.abs(got - exp).max())
        assert err <= 2e-2, (layer, kind, err)


@pytest.mark.gpu
def test_fp8_prefill_workspace_too_small():
    """A workspace without room for the tables, the q copy and one page copy
    is refused before any launch; one short of the chunk's page copies
    stages what fits, reads the rest as zeros and reports HSWA_ERR_BOUNDS."""
    c = Fp8Case([100, 300], seed=76, extra=80)
    B = c.B
    c.sess.reserve(range(B), [64, 64])
    c.ora.reserve(range(B), [64, 64])
    c.sess.sync()
    lay = c.sess.layers[0]
    prefix, q_start = np.array([100, 300], np.int32), np.array([0, 64, 128], np.int32)
    need = H.hswa_prefill_workspace_size_exact(c.sess.pool, lay, prefix, q_start)
    assert 0 < need < H.hswa_prefill_workspace_size(c.sess.pool, lay, B, 64)
    page = HKV * 64 * D * 2
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    q = wl.normal((128, HQ, D), 77, wl.DTYPE_BF16).cuda()
    args = (c.sess.pool, lay, q, torch.empty_like(q), c.sess.bt(0), torch.as_tensor(prefix, device="cuda"),
            torch.as_tensor(q_start, device="cuda"), B, 128, 64, 0.1, ws)
    with pytest.raises(H.HswaError) as e:
        H.hswa_prefill_chunk_ws(*args, need - 2 * page * ((100 + 64 + 63) // 64 + (300 + 64 + 63) // 64))
    assert e.value.status == H.HSWA_ERR_INVALID_ARG
    assert c.sess.check() == 0
    o = torch.full_like(q, float("nan"))
    H.hswa_prefill_chunk_ws(*(args[:3] + (o,) + args[4:]), need - 2 * page)
    assert c.sess.check() == H.HSWA_ERR_BOUNDS
    assert torch.isfinite(o.float()).all()
    H.hswa_prefill_chunk_ws(*(args[:3] + (o,) + args[4:]), need)
    assert c.sess.check() == 0


def fp8_multi_step(c, n_tok, seed, samples=None, grow=False):
    """Reserve n_tok tokens per sequence, append them (quantized), run one
    multi-token decode per layer and compare the given sequences' rows with
    the oracle at positions L - n_tok + w (tokens before position 0: o = 0).
    grow: new keys scaled by 1 + their draft position and q by 4, so that the
    row max jumps by far more than 2^8 on the last page."""
    B = c.B
    samples = list(range(B)) if samples is None else samples
    fs, ss = c.sess.reserve(range(B), [n_tok] * B)
    efs, ess = c.ora.reserve(range(B), [n_tok] * B)
    assert np.array_equal(fs, efs) and np.array_equal(ss, ess)
    c.sess.sync()
    scale = 1 / math.sqrt(D)
    for layer, kind in enumerate(c.kinds):
        slots = fs if kind == FULL else ss
        kn = wl.normal((B * n_tok, HKV, D), seed + 10 * layer + 1, wl.DTYPE_BF16)
        vn = wl.normal((B * n_tok, HKV, D), seed + 10 * layer + 2, wl.DTYPE_BF16)
        q = wl.normal((B * n_tok, HQ, D), seed + 10 * layer, wl.DTYPE_BF16)
        if grow:
            kn = (kn.float() * (1.0 + torch.arange(B * n_tok) % n_tok).view(-1, 1, 1)).to(torch.bfloat16)
            q = (q.float() * 4.0).to(torch.bfloat16)
        c.sess.append(layer, kn.cuda(), vn.cuda(), torch.as_tensor(slots, device="cuda"))
        o = torch.full((B * n_tok, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        c.sess.decode_multi(layer, q.cuda(), o, B, n_tok, scale)
        assert c.sess.check() == 0
        assert H.hswa_last_kernel() in ("decode_mma_fp8_d128", "decode_tc_fp8_d128")
        kc, ks, vc, vs = (x.cpu().numpy() for x in (c.sess.k[layer], c.sess.ks[layer], c.sess.v[layer],
                                                     c.sess.vs[layer]))
        lens = c.ora.seq_len[samples]
        rows = (np.asarray(samples)[:, None] * n_tok + np.arange(n_tok)[None, :]).reshape(-1)
        seq = np.repeat(np.asarray(samples), n_tok)
        pos = (lens[:, None] - n_tok + np.arange(n_tok)[None, :]).reshape(-1)
        got = o.float().cpu().numpy()[rows]
        assert np.isfinite(got).all()
        before = pos < 0
        assert np.all(got[before] == 0.0)
        exp = oracle.attention_fp8(raw_host(q)[rows[~before]], kc, ks, vc, vs, c.table(layer), seq[~before],
                                   pos[~before], 0 if kind == FULL else W, scale)
        err = float(np.abs(got[~before] - exp).max())
        assert err <= 2e-2, (layer, n_tok, err)


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [2, 3, 4, 5, 8, 9, 16])
def test_fp8_multi_token_decode_matches_oracle(n_tok):
    """Multi-token decode over FP8 pools (passes of two tokens on mma.sync,
    or one pass on the tensor cores with the pages converted to f16 in
    shared memory), lengths around page edges and the window."""
    cached = [0, 1, 62, 63, 64, 125, 126, 127, 128, 700, 3000]
    c = Fp8Case(cached, seed=73, extra=24)
    fp8_multi_step(c, n_tok, seed=1300 + n_tok)


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [2, 3, 8, 16])
def test_fp8_multi_token_large_max_jumps(n_tok):
    """Keys growing with the draft position and a scaled query: the row max
    jumps by far more than 2^8 on the last page, so the lazy O rescale fires
    in each kernel variant (two tokens per mma.sync pass; the tensor-core
    kernel with 4, 2 and 1 copies of the rows), over steps with releases."""
    c = Fp8Case([40, 300, 1500, 4000], seed=91, extra=3 * n_tok + 8)
    for step in range(3):
        assert c.sess.release(range(c.B)) == c.ora.swa_release(range(c.B))
        c.sess.sync()
        fp8_multi_step(c, n_tok, seed=1600 + 10 * step, grow=True)


@pytest.mark.gpu
def test_fp8_multi_token_decode_steps_with_release():
    """Verification steps of 3 tokens over FP8 pools, a release before each."""
    c = Fp8Case([5, 130, 255, 1000, 2047], seed=74, extra=64)
    for step in range(6):
        assert c.sess.release(range(c.B)) == c.ora.swa_release(range(c.B))
        c.sess.sync()
        fp8_multi_step(c, 3, seed=1400 + 10 * step)


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [2, 4, 8, 16])
def test_fp8_multi_token_full_size_sampled(n_tok):
    """The decode-batch workload over FP8 pools with n_tok query tokens per
    sequence, oracle on sampled sequences: two tokens per mma.sync pass, and
    the tensor-core kernel with 4, 2 and 1 copies of the rows."""
    w = wl.decode_batch()
    c = Fp8Case(list(w.cached), seed=82, extra=max(8, n_tok))
    fp8_multi_step(c, n_tok, seed=1500 + n_tok, samples=[0, 1, 17, 31, 32, 50, 63])


def fp8_window_pack(c, layer, lens):
    kc, ks, vc, vs = (x.cpu().numpy() for x in (c.sess.k[layer], c.sess.ks[layer], c.sess.v[layer], c.sess.vs[layer]))
    return oracle.swa_pack_fp8(kc, ks, vc, vs, c.ora.swa_bt, lens, W)


@pytest.mark.gpu
@pytest.mark.parametrize("dst_host", [False, True])
def test_fp8_gather_scatter_round_trip(dst_host):
    """Gather the windows of FP8 SWA layers (to device or pinned host memory)
    and compare with the oracle's pack byte for byte; then drop the SWA
    segments, give the windows other pages and scatter the buffers back: the
    pools pack to the same bytes again."""
    from scenario import window_offsets
    cached = [0, 1, 63, 64, 65, 127, 128, 129, 700, 3000]
    c = Fp8Case(cached, seed=77, kinds=(SWA, SWA))
    B = len(cached)
    lens = c.ora.seq_len[:B]
    offs, nbytes = window_offsets(c.sess, 0, lens, W)
    off = torch.as_tensor(offs, device="cuda")
    assert nbytes == int(offs[-1]) * 2 * HKV * (D + 4)
    bufs = []
    for layer in range(2):
        buf = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) if dst_host else \
            torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        c.sess.gather(layer, off, B, buf)
        assert c.sess.check() == 0
        assert H.hswa_last_kernel() == "swa_gather_fp8"
        exp = fp8_window_pack(c, layer, lens)
        assert np.array_equal(buf.cpu().numpy(), exp)
        bufs.append((buf, exp))
    assert c.sess.swa_drop(range(B)) == c.ora.swa_drop(range(B))
    assert c.sess.swa_restore(range(B)) == c.ora.swa_restore(range(B))
    c.sess.sync()
    for layer in range(2):
        c.sess.scatter(layer, off, B, bufs[layer][0])
        assert c.sess.check() == 0
        assert H.hswa_last_kernel() == "swa_scatter_fp8"
        assert np.array_equal(fp8_window_pack(c, layer, lens), bufs[layer][1])


@pytest.mark.gpu
def test_fp8_decode_batch_full_size_sampled():
    """The decode-batch workload (64 sequences, cached lengths uniform in
    [1024, 32768], 64/8 heads) over FP8 pools, in the launch configuration
    the benchmark times: one fused append + decode step per layer, oracle on
    sampled sequences."""
    w = wl.decode_batch()
    c = Fp8Case(list(w.cached), seed=81)
    B = c.B
    fs, ss = c.sess.reserve(range(B), [1] * B)
    efs, ess = c.ora.reserve(range(B), [1] * B)
    assert np.array_equal(fs, efs) and np.array_equal(ss, ess)
    c.sess.sync()
    samples = [0, 1, 17, 31, 32, 50, 63]
    scale = 1 / math.sqrt(D)
    for layer, kind in enumerate(c.kinds):
        slots = fs if kind == FULL else ss
        q = wl.normal((B, HQ, D), 900 + layer, wl.DTYPE_BF16)
        kn = wl.normal((B, HKV, D), 910 + layer, wl.DTYPE_BF16)
        vn = wl.normal((B, HKV, D), 920 + layer, wl.DTYPE_BF16)
        o = torch.full((B, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        c.sess.decode_append(layer, q.cuda(), kn.cuda(), vn.cuda(), torch.as_tensor(slots, device="cuda"), o, B,
                             scale)
        assert c.sess.check() == 0
        kc, ks, vc, vs = (x.cpu().numpy() for x in (c.sess.k[layer], c.sess.ks[layer], c.sess.v[layer],
                                                     c.sess.vs[layer]))
        exp = oracle.attention_fp8(raw_host(q)[samples], kc, ks, vc, vs, c.table(layer), np.array(samples),
                                   c.ora.seq_len[samples] - 1, 0 if kind == FULL else W, scale)
        got = o.float().cpu().numpy()[samples]
        assert np.isfinite(got).all()
        assert float(np.abs(got - exp).max()) <= 2e-2, layer


@pytest.mark.gpu
def test_fp8_chunked_prefill_full_size_sampled():
    """The chunked-prefill workload (8 sequences, prefixes uniform in
    [8192, 65536], a 4096-token chunk each) over FP8 pools: the staging pass
    and the fp16 tensor-core kernel at full size, oracle on rows at the tile
    edges and the chunk ends of every sequence."""
    w = wl.chunked_prefill()
    C = w.n_new
    c = Fp8Case(list(w.cached), seed=82, extra=C + 8)
    B = c.B
    fs, ss = c.sess.reserve(range(B), [C] * B)
    efs, ess = c.ora.reserve(range(B), [C] * B)
    assert np.array_equal(fs, efs) and np.array_equal(ss, ess)
    c.sess.sync()
    prefix = np.array(w.cached, np.int64)
    d_prefix = torch.as_tensor(prefix.astype(np.int32), device="cuda")
    d_qs = torch.arange(0, B * C + 1, C, dtype=torch.int32, device="cuda")
    rows_in_chunk = [0, 1, 127, 128, 129, 2047, 4094, 4095]
    rows = np.array([s * C + r for s in range(B) for r in rows_in_chunk])
    q_seq = np.repeat(np.arange(B), len(rows_in_chunk))
    q_pos = np.array([prefix[s] + r for s in range(B) for r in rows_in_chunk])
    scale = 1 / math.sqrt(D)
    for layer, kind in enumerate(c.kinds):
        slots = fs if kind == FULL else ss
        q = wl.normal((B * C, HQ, D), 930 + layer, wl.DTYPE_BF16)
        kn = wl.normal((B * C, HKV, D), 940 + layer, wl.DTYPE_BF16)
        vn = wl.normal((B * C, HKV, D), 950 + layer, wl.DTYPE_BF16)
        c.sess.append(layer, kn.cuda(), vn.cuda(), torch.as_tensor(slots, device="cuda"))
        o = torch.full((B * C, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        c.sess.prefill(layer, q.cuda(), o, d_prefix, d_qs, B, C, scale, prefix_host=prefix,
                       q_start_host=np.arange(0, B * C + 1, C))
        assert c.sess.check() == 0
        assert H.hswa_last_kernel() == prefill_kernel(kind, 0 if kind == FULL else W, fp8=True)
        kc, ks, vc, vs = (x.cpu().numpy() for x in (c.sess.k[layer], c.sess.ks[layer], c.sess.v[layer],
                                                     c.sess.vs[layer]))
        exp = oracle.attention_fp8(raw_host(q)[rows], kc, ks, vc, vs, c.table(layer), q_seq, q_pos,
                                   0 if kind == FULL else W, scale)
        got = o.float().cpu().numpy()[rows]
        assert np.isfinite(got).all()
        assert float(np.abs(got - exp).max()) <= 2e-2, layer


@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [2, 8])
def test_fp8_multi_token_bad_table_entries_set_bounds_and_skip(n_tok):
    """Invalid block-table entries inside the key range of an FP8 multi-token
    decode (the first page of a segment, a page past the pool, every page of
    one sequence): HSWA_ERR_BOUNDS, pages skipped, output finite, zeros where
    no key is left. Three sequences leave most CTAs without work."""
    c = Fp8Case([300, 300, 60], seed=75, extra=16)
    B = c.B
    c.sess.reserve(range(B), [n_tok] * B)
    c.sess.sync()
    c.sess.d_full_bt[0, 0] = -1
    c.sess.d_full_bt[1, 3] = 1 << 30
    c.sess.d_full_bt[2, 0] = -1
    c.sess.d_full_bt[2, 1] = -1
    q = wl.normal((B * n_tok, HQ, D), 1600, wl.DTYPE_BF16).cuda()
    o = torch.full_like(q, float("nan"))
    c.sess.decode_multi(0, q, o, B, n_tok, 1 / math.sqrt(D))
    assert c.sess.check() == H.HSWA_ERR_BOUNDS
    assert c.sess.check() == 0
    assert torch.isfinite(o.float()).all()
    assert torch.equal(o[2 * n_tok:].float(), torch.zeros_like(o[2 * n_tok:].float()))
