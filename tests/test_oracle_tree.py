"""Pins for the oracle's SWA-aware prefix cache tree (no GPU).

* the window-safety rule ("MiMo-V2.5 Series Inference Full-Link
  Optimization", Sec. 2.1, SWA-aware prefix cache tree, item 1) on hand
  cases, and the pages' pseudo-match: equal tokens whose SWA tail has been
  released give no hit;
* on random request traces: every match against a brute-force restatement
  (the deepest stored node whose token path equals the query's prefix,
  found by comparing full paths, then the largest end e = m*P such that
  every position in [e - W, e) sits on a page with an SWA slot); and the
  holder invariants: each page's count equals the tables and tree nodes
  naming it, a free page is named by nobody, nothing is lost or doubled;
* eviction: it frees only pages the tree alone holds, out-of-window SWA
  before in-window SWA, oldest leaves first;
* planted mistakes in the oracle fail these pins.
"""
import importlib.util
import os
import sys

import numpy as np
import pytest

import oracle
from oracle import prefix_tree as PT

HERE = os.path.dirname(__file__)


def test_window_safe_pages_hand_cases():
    f = PT.window_safe_pages
    assert f([], 64, 128) == 0
    assert f([1] * 15, 64, 128) == 15
    # released head, window pages 13 and 14 kept (positions [832, 960))
    assert f([-1] * 13 + [5, 6], 64, 128) == 15
    # a 10-page prefix whose pages 8 and 9 have no SWA page is trimmed to 8
    # pages: the window of that end, positions [384, 512), is pages 6 and 7
    assert f([1] * 8 + [-1, -1], 64, 128) == 8
    # only the last page missing: trimmed to the first m whose window is whole
    assert f([1] * 9 + [-1], 64, 128) == 9
    # W not a multiple of P: m = 5 needs positions [40, 80) = pages 2, 3, 4
    assert f([-1, -1, 1, 1, 1], 16, 40) == 5
    # page 2 missing: every m from 5 down to 1 has a window meeting a missing page
    assert f([-1, -1, -1, 1, 1], 16, 40) == 0
    assert f([1, -1, -1, 1, 1], 16, 40) == 1
    # m = 4 with P = 2, W = 5 needs positions [3, 8): page 1 holds position 3
    assert f([1, -1, 1, 1], 2, 5) == 1
    assert f([-1, 1, 1, 1], 2, 5) == 4


def make_pool(W=128, P=64, full=64, swa=64, S=4, MP=32):
    return oracle.DualPool(W, P, full, swa, S, MP)


def run_request(pool, tree, s, tokens, chunk, release=True):
    """A request: match, share the hit, prefill the rest in chunks with a
    release after each, then store the result in the tree."""
    m, full, swa, raw = tree.match(tokens)
    if m:
        pool.share_prefix(s, full, swa)
    L = m * pool.P
    while L < len(tokens):
        n = min(chunk, len(tokens) - L)
        pool.reserve([s], [n])
        if release:
            pool.swa_release([s])
        L += n
    tree.insert(s, tokens)
    return m, raw


def test_pseudo_match_of_the_pages():
    """A 1000-token request ends with its out-of-window SWA released. The
    same 1000 tokens hit 15 pages; its first 700 tokens are equal tokens too,
    but the SWA slots of their last W positions are gone, so the hit is 0."""
    pool, tokens = make_pool(), list(range(1000))
    tree = PT.PrefixTree(pool)
    assert run_request(pool, tree, 0, tokens, 256) == (0, 0)
    pool.seq_free([0])
    m, full, swa, raw = tree.match(tokens)
    assert (m, raw) == (15, 15)
    assert swa[13] >= 0 and swa[14] >= 0 and all(x < 0 for x in swa[:13])
    m, _, _, raw = tree.match(tokens[:700])
    assert (m, raw) == (0, 10)
    # the hit is reusable: a new request shares 15 pages and computes 40 tokens
    assert run_request(pool, tree, 1, tokens + [7] * 40, 256)[0] == 15
    assert pool.seq_len[1] == 1040
    assert np.array_equal(pool.full_bt[1, :15], full)


# ------------------------------------------------------------ brute force
def node_paths(tree):
    """Token path (concatenated page tokens from the root) of every node."""
    out = {}
    for nd in tree.nodes():
        chain, x = [], nd
        while x is not tree.root:
            chain.append(x)
            x = x.parent
        chain.reverse()
        out[nd.id] = (sum((list(c.tokens) for c in chain), []), chain)
    return out


def brute_match(tree, tokens):
    P, W = tree.pool.P, tree.pool.W
    best = []
    for path, chain in node_paths(tree).values():
        if len(path) <= len(tokens) and tokens[:len(path)] == path and len(chain) > len(best):
            best = chain
    raw = len(best)
    for m in range(raw, -1, -1):
        e = m * P
        if all(best[t // P].swa >= 0 for t in range(max(0, e - W), e)):
            return m, [c.full for c in best[:m]], [c.swa for c in best[:m]], raw
    raise AssertionError("m = 0 always qualifies")


def check_holders(pool, tree):
    full_cnt = np.zeros(pool.full_pages, np.int64)
    swa_cnt = np.zeros(pool.swa_pages, np.int64)
    for x in pool.full_bt[pool.full_bt >= 0]:
        full_cnt[x] += 1
    for x in pool.swa_bt[pool.swa_bt >= 0]:
        swa_cnt[x] += 1
    for nd in tree.nodes():
        full_cnt[nd.full] += 1
        if nd.swa >= 0:
            swa_cnt[nd.swa] += 1
    assert np.array_equal(full_cnt, pool.full_ref)
    assert np.array_equal(swa_cnt, pool.swa_ref)
    for free, cnt, n in ((pool.full_free, full_cnt, pool.full_pages), (pool.swa_free, swa_cnt, pool.swa_pages)):
        free = list(free)
        assert len(set(free)) == len(free)
        assert set(free) == set(np.flatnonzero(cnt == 0).tolist())
        assert len(free) + int(np.count_nonzero(cnt)) == n
    # two nodes never store the same Full page; a node's page matches its tokens' position
    fulls = [nd.full for nd in tree.nodes()]
    assert len(set(fulls)) == len(fulls)


def random_tokens(rng, bases, P):
    """A request sharing a random whole-page prefix with an earlier one."""
    base = bases[rng.integers(len(bases))] if bases and rng.random() < 0.8 else []
    keep = int(rng.integers(0, len(base) // P + 1)) * P if base else 0
    tail = rng.integers(0, 3, int(rng.integers(1, 40))).tolist()
    return base[:keep] + tail


@pytest.mark.parametrize("seed,W,P", [(0, 8, 4), (1, 6, 4), (2, 12, 4), (3, 5, 2)])
def test_random_traces_match_brute_force_and_keep_holders(seed, W, P, module=PT):
    rng = np.random.default_rng(seed)
    pool = oracle.DualPool(W, P, 400, 400, 6, 40)
    tree = module.PrefixTree(pool)
    bases, live = [], {}
    for step in range(160):
        op = rng.random()
        free_seqs = [s for s in range(6) if s not in live]
        if op < 0.5 and free_seqs:
            s = free_seqs[0]
            tokens = random_tokens(rng, bases, P)
            exp = brute_match(tree, tokens)
            got = tree.match(tokens)
            assert got[0] == exp[0] and got[3] == exp[3], (step, got, exp)
            assert list(got[1]) == exp[1] and list(got[2]) == exp[2]
            if got[0]:
                pool.share_prefix(s, got[1], got[2])
            L = got[0] * P
            while L < len(tokens):
                n = min(int(rng.integers(1, 9)), len(tokens) - L)
                try:
                    pool.reserve([s], [n])
                except oracle.NoSpace:
                    tree.evict(n, n)
                    pool.reserve([s], [n])
                if rng.random() < 0.7:
                    pool.swa_release([s])
                L += n
            live[s] = tokens
            bases.append(tokens)
        elif op < 0.8 and live:
            s = sorted(live)[int(rng.integers(len(live)))]
            tree.insert(s, live[s])
            pool.seq_free([s])
            del live[s]
        else:
            before_f, before_s = len(pool.full_free), len(pool.swa_free)
            held = {int(x) for x in pool.full_bt[pool.full_bt >= 0]}
            held_s = {int(x) for x in pool.swa_bt[pool.swa_bt >= 0]}
            ff, fs = tree.evict(int(rng.integers(0, 4)), int(rng.integers(0, 4)))
            assert len(pool.full_free) - before_f == ff and len(pool.swa_free) - before_s == fs
            assert not held & set(pool.full_free) and not held_s & set(pool.swa_free)
        check_holders(pool, tree)
    tree.clear()
    for s in sorted(live):
        pool.seq_free([s])
    assert len(pool.full_free) == 400 and len(pool.swa_free) == 400


def test_swa_eviction_takes_out_of_window_pages_first():
    """One stored 16-page sequence with every SWA page kept (no release):
    W = 8, P = 4, so pages 14 and 15 meet the window of its end. Evicting 14
    SWA pages takes pages 0..13 (oldest first among equals: creation
    order), keeps the tail and so the full 16-page hit; one more takes the
    tail and the hit shrinks."""
    pool = oracle.DualPool(8, 4, 64, 64, 2, 20)
    tree = PT.PrefixTree(pool)
    tokens = list(range(64))
    run_request(pool, tree, 0, tokens, 64, release=False)
    pool.seq_free([0])
    assert tree.stats() == (16, 16, 16)
    assert tree.evict(0, 14) == (0, 14)
    assert [nd.swa >= 0 for nd in tree.nodes()] == [False] * 14 + [True, True]
    assert tree.match(tokens)[0] == 16
    assert tree.evict(0, 1) == (0, 1)
    assert tree.match(tokens)[0] == 0  # page 14 or 15 gone: no end keeps a whole window
    check_holders(pool, tree)


def test_insert_adopts_the_window_of_a_recomputed_prefix():
    """A request whose prefix was a pseudo-match recomputes it; storing it
    gives the tree's nodes the SWA pages they had lost, so the same prefix
    hits afterwards."""
    pool, tokens = make_pool(), list(range(1000))
    tree = PT.PrefixTree(pool)
    run_request(pool, tree, 0, tokens, 256)
    pool.seq_free([0])
    c = tokens[:704] + [5] * 30
    assert run_request(pool, tree, 1, c, 256) == (0, 11)  # pseudo-match, recomputed
    pool.seq_free([1])
    m, _, swa, _ = tree.match(tokens[:704])
    assert m == 11 and swa[9] >= 0 and swa[10] >= 0
    check_holders(pool, tree)


def test_full_eviction_is_least_recently_used():
    pool = oracle.DualPool(8, 4, 64, 64, 2, 20)
    tree = PT.PrefixTree(pool)
    a, b = [1] * 12, [2] * 12
    run_request(pool, tree, 0, a, 12)
    pool.seq_free([0])
    run_request(pool, tree, 1, b, 12)
    pool.seq_free([1])
    tree.match(a)  # a is now the more recent
    assert tree.evict(1, 0)[0] == 1
    assert [(list(nd.tokens), nd.index) for nd in tree.nodes()] == \
        [([1] * 4, 0), ([1] * 4, 1), ([1] * 4, 2), ([2] * 4, 0), ([2] * 4, 1)]
    check_holders(pool, tree)


def test_full_eviction_takes_the_oldest_leaves_and_spares_held_pages():
    pool = oracle.DualPool(8, 4, 64, 64, 3, 20)
    tree = PT.PrefixTree(pool)
    a, b = [1] * 12, [2] * 12
    run_request(pool, tree, 0, a, 12)
    pool.seq_free([0])
    run_request(pool, tree, 1, b, 12)
    pool.seq_free([1])
    # a request now shares b's prefix: b's pages are held, a's are not
    m, full, swa, _ = tree.match(b + [3] * 4)
    assert m == 3
    pool.share_prefix(2, full, swa)
    assert tree.evict(2, 0)[0] == 2  # a's two deepest pages, oldest leaf first
    assert [list(nd.tokens) for nd in tree.nodes()] == [[1] * 4, [2] * 4, [2] * 4, [2] * 4]
    assert tree.evict(10, 0)[0] == 1  # a's last page; b's are held by sequence 2
    assert [list(nd.tokens) for nd in tree.nodes()] == [[2] * 4] * 3  # and stay cached
    check_holders(pool, tree)


# ------------------------------------------------------------------ mutants
MUTATIONS = {
    "window_off_by_one": ("first = max(0, m * P - W) // P", "first = max(0, m * P - W + 1) // P"),
    "no_trim": ("return m, [nd.full for nd in path[:m]]", "m = len(path)\n        return m, [nd.full for nd in path[:m]]"),
    "no_adopt": ("elif nxt.swa < 0 and pool.swa_bt[s, p] >= 0:", "elif False:"),
    "in_window_first": ("key=lambda nd: (in_window[nd.id], nd.last, nd.id)",
                        "key=lambda nd: (not in_window[nd.id], nd.last, nd.id)"),
    "evict_held_leaves": ("if not nd.children and pool.full_ref[nd.full] == 1]", "if not nd.children]"),
    "newest_leaf_first": ("nd = min(leaves, key=lambda nd: (nd.last, nd.id))",
                          "nd = max(leaves, key=lambda nd: (nd.last, nd.id))"),
}


def mutant_module(name):
    src = open(PT.__file__).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, name
    spec = importlib.util.spec_from_loader("mutant_tree_" + name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src.replace(old, new), "mutant", "exec"), mod.__dict__)
    return mod


def all_pins(mod):
    """Run every pin above against a tree module; True if all hold."""
    saved = PT.PrefixTree, PT.window_safe_pages
    PT.PrefixTree, PT.window_safe_pages = mod.PrefixTree, mod.window_safe_pages
    try:
        for fn in (test_window_safe_pages_hand_cases, test_pseudo_match_of_the_pages,
                   test_swa_eviction_takes_out_of_window_pages_first,
                   test_insert_adopts_the_window_of_a_recomputed_prefix,
                   test_full_eviction_is_least_recently_used,
                   test_full_eviction_takes_the_oldest_leaves_and_spares_held_pages):
            fn()
        for args in [(0, 8, 4), (1, 6, 4), (2, 12, 4), (3, 5, 2)]:
            test_random_traces_match_brute_force_and_keep_holders(*args, module=mod)
        return True
    except (AssertionError, ValueError, KeyError, IndexError):
        return False
    finally:
        PT.PrefixTree, PT.window_safe_pages = saved


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_tree_pins_catch_planted_mistake(name):
    assert not all_pins(mutant_module(name)), name
