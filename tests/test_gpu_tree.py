"""Prefix reuse on the GPU: attention over pages shared through the SWA-aware
prefix cache tree, against the float64 oracle.

Request A prefills 4096 + 1000 tokens in two chunks; after each chunk's SWA
release its prefix is stored in the tree. Request B repeats A's first 4096
tokens and adds its own: the tree hits 64 pages (the window of A's first
chunk end is still held), B shares them and prefills only its 300 new tokens,
whose Full and SWA attention read A's pages; then B decodes a token. Request
C repeats A's first 3000 tokens: the same tokens, but the SWA slots of their
last W positions were released, so the hit is trimmed to nothing (the pages'
pseudo-match). Every table, slot and match is checked against the oracle
bit for bit and every output row against the oracle's attention."""
import numpy as np
import pytest
import torch

import hswa_workloads as wl
import oracle
from oracle import prefix_tree as PT
import hybrid_sliding_window_dual_gb300 as H
from hybrid_sliding_window_dual_gb300.session import DualPoolSession
from scenario import TOL, device_out, max_err, prefill_kernel, raw_host

FULL, SWA = wl.KIND_FULL, wl.KIND_SWA
HQ, HKV, D, P, W = 64, 8, 128, 64, 128


class Case:
    def __init__(self, seed):
        full_pages, swa_pages, S, MP = 200, 160, 4, 96
        fo, so = wl.permutation(full_pages, seed), wl.permutation(swa_pages, seed + 1)
        self.cfg = H.Config(window=W, page_size=P, n_q_heads=HQ, n_kv_heads=HKV, head_dim=D,
                            dtype=H.HSWA_DTYPE_BF16, full_pages=full_pages, swa_pages=swa_pages, max_seqs=S,
                            max_pages_per_seq=MP)
        self.sess = DualPoolSession(self.cfg, [FULL, SWA], fo, so)
        self.ora = oracle.DualPool(W, P, full_pages, swa_pages, S, MP, fo, so)
        self.otree = PT.PrefixTree(self.ora)
        self.seed = seed
        self.scale = D ** -0.5

    def check_tables(self):
        f, s, lens = self.sess.tables()
        assert np.array_equal(f, self.ora.full_bt) and np.array_equal(s, self.ora.swa_bt)
        assert np.array_equal(lens.astype(np.int64), self.ora.seq_len)

    def match(self, tokens):
        got = self.sess.match_prefix(tokens)
        exp = self.otree.match(tokens)
        assert got[0] == exp[0] and got[3] == exp[3]
        assert list(got[1]) == list(exp[1]) and list(got[2]) == list(exp[2])
        return got

    def chunk(self, s, n, seed, check=True):
        """Reserve, append and attend n new tokens of sequence s (both layers)."""
        prefix = int(self.ora.seq_len[s])
        fs, ss = self.sess.reserve([s], [n])
        efs, ess = self.ora.reserve([s], [n])
        assert np.array_equal(fs, efs) and np.array_equal(ss, ess)
        self.sess.sync()
        d_prefix = torch.full((1,), prefix, dtype=torch.int32, device="cuda")
        d_qs = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        # the kernels address sequence s as row 0 of the tables they get
        rows = {FULL: self.sess.d_full_bt[s:s + 1], SWA: self.sess.d_swa_bt[s:s + 1]}
        errs = []
        for layer, kind in enumerate((FULL, SWA)):
            q = wl.normal((n, HQ, D), seed + 10 * layer, wl.DTYPE_BF16)
            kn = wl.normal((n, HKV, D), seed + 10 * layer + 1, wl.DTYPE_BF16)
            vn = wl.normal((n, HKV, D), seed + 10 * layer + 2, wl.DTYPE_BF16)
            slots = fs if kind == FULL else ss
            self.sess.append(layer, kn.cuda(), vn.cuda(), torch.as_tensor(slots, device="cuda"))
            o = torch.full((n, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
            H.hswa_prefill_chunk(self.sess.pool, self.sess.layers[layer], q.cuda(), o, rows[kind], d_prefix, d_qs,
                                 1, n, n, self.scale, self.sess.stream)
            assert self.sess.check() == 0
            if not check:
                continue
            assert H.hswa_last_kernel() == prefill_kernel(kind, 0 if kind == FULL else W)
            bt = self.ora.full_bt if kind == FULL else self.ora.swa_bt
            exp = oracle.attention(raw_host(q), raw_host(self.sess.k[layer]), raw_host(self.sess.v[layer]), bt,
                                   np.full(n, s), np.arange(prefix, prefix + n), 0 if kind == FULL else W,
                                   self.scale)
            got = device_out(o)
            assert np.isfinite(got).all()
            errs.append(max_err(got, exp))
            assert errs[-1] <= TOL[wl.DTYPE_BF16], (layer, errs[-1])
        return errs

    def release(self, s):
        assert self.sess.release([s]) == self.ora.swa_release([s])

    def store(self, s, tokens):
        assert self.sess.store_prefix(s, tokens) == self.otree.insert(s, tokens)

    def free(self, s):
        self.sess.seq_free([s])
        self.ora.seq_free([s])


@pytest.mark.gpu
def test_shared_prefix_attention_matches_oracle():
    c = Case(21)
    rng = np.random.default_rng(21)
    a = rng.integers(0, 32000, 5096).tolist()
    # request A: two chunks, release then store after each
    assert c.match(a)[0] == 0
    c.chunk(0, 4096, 100, check=False)
    c.release(0)
    c.store(0, a[:4096])
    c.chunk(0, 1000, 200)
    c.release(0)
    c.store(0, a)
    c.free(0)
    c.check_tables()
    # request B: A's first chunk + 300 own tokens
    b = a[:4096] + rng.integers(0, 32000, 300).tolist()
    m, full, swa, raw = c.match(b)
    assert (m, raw) == (64, 64)
    c.sess.share_prefix(1, full, swa)
    c.ora.share_prefix(1, list(full), list(swa))
    c.check_tables()
    c.chunk(1, 300, 300)  # attention over A's shared pages and B's own
    c.release(1)
    c.check_tables()
    # one decode token for B on top of the shared prefix
    c.chunk(1, 1, 400)
    # request C: equal tokens whose window was released: no hit
    m, _, _, raw = c.match(a[:3000])
    assert (m, raw) == (0, 46)
    c.store(1, b)
    c.free(1)
    c.check_tables()
    # every page the tree holds is still valid; evicting everything empties the pools' holders
    ff, fs = c.sess.evict(10 ** 6, 10 ** 6)
    assert (ff, fs) == c.otree.evict(10 ** 6, 10 ** 6)
    assert len(H.hswa_get_free_list(c.sess.pool, H.HSWA_KIND_FULL)) == c.cfg.full_pages
    assert len(H.hswa_get_free_list(c.sess.pool, H.HSWA_KIND_SWA)) == c.cfg.swa_pages
    c.sess.close()
