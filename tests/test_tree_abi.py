"""The native SWA-aware prefix cache tree against the oracle (no GPU).

Random request traces (match, share the hit, prefill in chunks with
releases, store at the end, free; evictions when a pool runs short, and on
their own) drive libhswa and the oracle side by side; after every call the
match results, block tables, free lists, page holder counts and tree nodes
must be identical."""
import numpy as np
import pytest

import hswa_workloads as wl
import oracle
from oracle import prefix_tree as PT
import hybrid_sliding_window_dual_gb300 as H


def oracle_nodes(tree):
    return np.array([[nd.id, -1 if nd.parent is tree.root else nd.parent.id, nd.index, nd.full, nd.swa]
                     for nd in tree.nodes()], np.int32).reshape(-1, 5)


class Pair:
    def __init__(self, W, P, full, swa, S, MP, seed):
        fo, so = wl.permutation(full, seed), wl.permutation(swa, seed + 1)
        self.cfg = H.Config(window=W, page_size=P, n_q_heads=4, n_kv_heads=1, head_dim=16,
                            dtype=H.HSWA_DTYPE_BF16, full_pages=full, swa_pages=swa, max_seqs=S,
                            max_pages_per_seq=MP)
        self.pool = H.hswa_pool_create(self.cfg, fo, so)
        self.tree = H.hswa_tree_create(self.pool)
        self.opool = oracle.DualPool(W, P, full, swa, S, MP, fo, so)
        self.otree = PT.PrefixTree(self.opool)
        self.P, self.MP = P, MP

    def check(self):
        f, s, lens = H.hswa_get_tables(self.pool, self.cfg)
        assert np.array_equal(f, self.opool.full_bt) and np.array_equal(s, self.opool.swa_bt)
        assert np.array_equal(lens.astype(np.int64), self.opool.seq_len)
        assert list(H.hswa_get_free_list(self.pool, H.HSWA_KIND_FULL)) == list(self.opool.full_free)
        assert list(H.hswa_get_free_list(self.pool, H.HSWA_KIND_SWA)) == list(self.opool.swa_free)
        assert np.array_equal(H.hswa_get_page_refs(self.pool, H.HSWA_KIND_FULL, self.cfg.full_pages),
                              self.opool.full_ref)
        assert np.array_equal(H.hswa_get_page_refs(self.pool, H.HSWA_KIND_SWA, self.cfg.swa_pages),
                              self.opool.swa_ref)
        assert np.array_equal(H.hswa_tree_nodes(self.tree), oracle_nodes(self.otree))
        assert H.hswa_tree_stats(self.tree) == self.otree.stats()

    def match(self, tokens):
        got = H.hswa_tree_match(self.tree, tokens, self.MP)
        exp = self.otree.match(tokens)
        assert got[0] == exp[0] and got[3] == exp[3]
        assert list(got[1]) == list(exp[1]) and list(got[2]) == list(exp[2])
        return got

    def reserve(self, s, n):
        try:
            exp = self.opool.reserve([s], [n])
        except oracle.NoSpace:
            with pytest.raises(H.NoSpace):
                H.hswa_reserve(self.pool, [s], [n])
            return None
        got = H.hswa_reserve(self.pool, [s], [n])
        assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])
        return got

    def close(self):
        H.hswa_tree_destroy(self.tree)
        self.otree.clear()
        assert list(H.hswa_get_free_list(self.pool, H.HSWA_KIND_FULL)) == list(self.opool.full_free)
        assert list(H.hswa_get_free_list(self.pool, H.HSWA_KIND_SWA)) == list(self.opool.swa_free)
        H.hswa_pool_destroy(self.pool)


def random_tokens(rng, bases, P):
    """A request that continues a whole earlier one (a follow-up turn), cuts
    one at a random page, or is new."""
    base = bases[rng.integers(len(bases))] if bases and rng.random() < 0.8 else []
    if rng.random() < 0.5:
        keep = len(base)
    else:
        keep = int(rng.integers(0, len(base) // P + 1)) * P if base else 0
    tail = rng.integers(0, 3, int(rng.integers(1, 48))).tolist()
    return base[:keep] + tail


@pytest.mark.parametrize("seed,W,P,full,swa", [(0, 8, 4, 160, 120), (1, 6, 4, 200, 60), (2, 12, 4, 120, 200),
                                              (3, 5, 2, 300, 300), (4, 16, 8, 90, 60)])
def test_native_tree_matches_oracle_on_random_traces(seed, W, P, full, swa):
    rng = np.random.default_rng(100 + seed)
    S, MP = 6, 64 // P + 8
    x = Pair(W, P, full, swa, S, MP, seed)
    bases, live = [], {}
    for step in range(250):
        op = rng.random()
        free_seqs = [s for s in range(S) if s not in live]
        if op < 0.45 and free_seqs:
            s = free_seqs[0]
            tokens = random_tokens(rng, bases, P)[:MP * P - 1]
            m, fpages, spages, raw = x.match(tokens)
            if m:
                H.hswa_seq_share_prefix(x.pool, s, fpages, spages)
                x.opool.share_prefix(s, list(fpages), list(spages))
            L, ok = m * P, True
            while L < len(tokens):
                n = min(int(rng.integers(1, 12)), len(tokens) - L)
                if x.reserve(s, n) is None:
                    want = n // P + 2
                    assert H.hswa_tree_evict(x.tree, want, want) == x.otree.evict(want, want)
                    x.check()
                    if x.reserve(s, n) is None:
                        ok = False
                        break
                if rng.random() < 0.7:
                    assert H.hswa_swa_release(x.pool, [s]) == x.opool.swa_release([s])
                L += n
            if ok:
                live[s] = tokens
                bases.append(tokens)
            else:  # could not admit it: give its pages back
                H.hswa_seq_free(x.pool, [s])
                x.opool.seq_free([s])
        elif op < 0.75 and live:
            s = sorted(live)[int(rng.integers(len(live)))]
            n = len(live[s]) if rng.random() < 0.8 else int(rng.integers(0, len(live[s]) + 1))
            assert H.hswa_tree_insert(x.tree, s, live[s][:n]) == x.otree.insert(s, live[s][:n])
            H.hswa_seq_free(x.pool, [s])
            x.opool.seq_free([s])
            del live[s]
        else:
            wf, ws = int(rng.integers(0, 5)), int(rng.integers(0, 5))
            assert H.hswa_tree_evict(x.tree, wf, ws) == x.otree.evict(wf, ws)
        x.check()
    for s in sorted(live):
        H.hswa_seq_free(x.pool, [s])
        x.opool.seq_free([s])
    x.check()
    x.close()


def test_pseudo_match_and_reuse_through_the_abi():
    """The pages' case at W = 128, P = 64: a stored 1000-token request hits
    15 pages for the same tokens and none for its first 700."""
    x = Pair(128, 64, 64, 64, 4, 32, 0)
    tokens = list(range(1000))
    for L in range(0, 1000, 256):
        x.reserve(0, min(256, 1000 - L))
        assert H.hswa_swa_release(x.pool, [0]) == x.opool.swa_release([0])
    assert H.hswa_tree_insert(x.tree, 0, tokens) == x.otree.insert(0, tokens) == 15
    H.hswa_seq_free(x.pool, [0])
    x.opool.seq_free([0])
    m, fpages, spages, raw = x.match(tokens)
    assert (m, raw) == (15, 15)
    assert x.match(tokens[:700])[0] == 0
    H.hswa_seq_share_prefix(x.pool, 1, fpages, spages)
    x.opool.share_prefix(1, list(fpages), list(spages))
    x.check()
    assert x.reserve(1, 40) is not None
    x.check()
    x.close()


def test_tree_argument_errors_change_nothing():
    x = Pair(8, 4, 32, 32, 2, 8, 0)
    x.reserve(0, 10)
    x.check()
    with pytest.raises(H.HswaError):  # more tokens than the sequence holds
        H.hswa_tree_insert(x.tree, 0, list(range(11)))
    with pytest.raises(H.HswaError):  # cap below the query's pages
        H.hswa_tree_match(x.tree, list(range(12)), 2)
    with pytest.raises(H.HswaError):  # sequence not empty
        H.hswa_seq_share_prefix(x.pool, 0, [1], [1])
    with pytest.raises(H.HswaError):  # pages held by no one
        free_page = int(H.hswa_get_free_list(x.pool, H.HSWA_KIND_FULL)[0])
        H.hswa_seq_share_prefix(x.pool, 1, [free_page], [0])
    with pytest.raises(H.HswaError):  # a pool with a live tree
        H.hswa_pool_destroy(x.pool)
    with pytest.raises(H.HswaError):
        H.hswa_tree_evict(x.tree, -1, 0)
    x.check()
    H.hswa_seq_free(x.pool, [0])
    x.opool.seq_free([0])
    x.close()


def test_depth_updates_on_a_prompt_shared_by_branches():
    """One prompt shared by branches of different depths, checked against
    the oracle after every call. Evicting the shallowest branch makes the
    prompt's shallowest leaf deeper (its children are looked at again); a new
    shallower branch makes it shallower; a branch that extends a stored leaf
    turns that leaf into an inner node; SWA evictions in between take pages
    on both sides of the window as leaves go."""
    W, P = 8, 4
    x = Pair(W, P, 400, 400, 4, 40, 7)
    prompt = list(range(100, 100 + 6 * P))  # 6 pages

    def store(tokens):
        m, fpages, spages, raw = x.match(tokens)
        if m:
            H.hswa_seq_share_prefix(x.pool, 0, fpages, spages)
            x.opool.share_prefix(0, list(fpages), list(spages))
        L = m * P
        while L < len(tokens):
            n = min(5, len(tokens) - L)
            assert x.reserve(0, n) is not None
            assert H.hswa_swa_release(x.pool, [0]) == x.opool.swa_release([0])
            L += n
        assert H.hswa_tree_insert(x.tree, 0, tokens) == x.otree.insert(0, tokens)
        H.hswa_seq_free(x.pool, [0])
        x.opool.seq_free([0])
        x.check()

    # branches 1, 3, 5 and 2 pages below the prompt, the shallowest stored first (oldest)
    for b, k in ((1, 1), (2, 3), (3, 5), (4, 2)):
        store(prompt + [b] * (P * k))
    for _ in range(6):  # leaves oldest first: the one-page branch goes first
        assert H.hswa_tree_evict(x.tree, 1, 0) == x.otree.evict(1, 0)
        x.check()
        assert H.hswa_tree_evict(x.tree, 0, 1) == x.otree.evict(0, 1)
        x.check()
    store(prompt + [5] * P)                    # shallower than every branch left
    store(prompt + [4] * (P * 2) + [6] * P)    # extends the two-page branch's leaf
    for _ in range(30):
        assert H.hswa_tree_evict(x.tree, 2, 1) == x.otree.evict(2, 1)
        x.check()
    assert H.hswa_tree_stats(x.tree)[0] == 0
    x.close()
