"""CPU oracle of the SWA-aware prefix cache tree.

TEST INFRASTRUCTURE ONLY: used by tests/ (see oracle/__init__.py). It
shares no code with the CUDA library.

"MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 2.1, SWA-aware
prefix cache tree. Equal tokens no longer mean reusable KV, because the SWA
pool drops out-of-window slots; the tree therefore

1. trims every match to the window-safety length: besides equal tokens,
   the last W positions of the matched prefix must still have SWA slots;
   the part past that boundary counts as a miss;
2. (release bound to the request lifecycle: the pool's swa_release);
3. keeps two indexes per node, the Full segment and the SWA mapping, and
   evicts them apart: out-of-window SWA segments alone (the Full prefix
   stays reusable) or whole segments.

Readings taken where the page is silent:
* granularity: one node per page of P tokens; a node holds the page's
  tokens, its Full page and its SWA page (-1: none); matches and inserts
  are whole pages;
* the tree holds one reference on each page it stores (the pool counts
  holders, see oracle/pool.py); a hit gives a sequence the prefix's Full
  pages and its SWA window pages (DualPool.share_prefix);
* recency: a logical clock advanced by every match and insert; a match
  stamps the nodes of its untrimmed token match, an insert the nodes of its
  whole path;
* insert keeps the tree's page where one exists for the same tokens (the
  sequence's duplicate is freed with the sequence) and adopts the
  sequence's SWA page where the tree's node has none;
* SWA eviction frees SWA pages that only the tree holds: first those
  outside the window of every stored sequence end below them (a node at
  page index i is inside that window when i >= (D*P - W) // P for the
  shallowest leaf below or at it, D pages deep), oldest first (clock, then
  creation order), then the in-window ones; Full eviction removes, oldest
  first, leaf nodes whose Full page only the tree holds (their SWA page
  goes too), until enough pages are free or no leaf qualifies.
"""
from __future__ import annotations


class Node:
    __slots__ = ("tokens", "full", "swa", "parent", "children", "last", "id", "index")

    def __init__(self, tokens, full, swa, parent, node_id, index):
        self.tokens = tokens      # tuple of the page's P token ids
        self.full = full          # Full page
        self.swa = swa            # SWA page or -1
        self.parent = parent
        self.children = {}        # tokens tuple -> Node
        self.last = 0             # clock of the last match / insert through it
        self.id = node_id         # creation order
        self.index = index        # logical page index (depth - 1)


def window_safe_pages(swa, P, W):
    """Largest m <= len(swa) such that every logical page meeting the last W
    positions [m*P - W, m*P) has an SWA page (swa[p] >= 0); 0 always is."""
    for m in range(len(swa), -1, -1):
        first = max(0, m * P - W) // P
        if all(swa[p] >= 0 for p in range(first, m)):
            return m
    return 0


class PrefixTree:
    def __init__(self, pool):
        self.pool = pool
        self.root = Node((), -1, -1, None, -1, -1)
        self.clock = 0
        self.next_id = 0

    # ---------------------------------------------------------- traversal
    def nodes(self):
        """Every node but the root, in creation order."""
        out, stack = [], [self.root]
        while stack:
            nd = stack.pop()
            for ch in nd.children.values():
                out.append(ch)
                stack.append(ch)
        return sorted(out, key=lambda nd: nd.id)

    def _page_keys(self, tokens):
        P = self.pool.P
        return [tuple(int(x) for x in tokens[i * P:(i + 1) * P]) for i in range(len(tokens) // P)]

    # -------------------------------------------------------------- match
    def match(self, tokens):
        """Window-safe hit for a token sequence: returns (m, full_pages,
        swa_pages, raw) with m whole pages usable, the pages of logical pages
        [0, m), and raw the pages whose tokens matched before trimming."""
        self.clock += 1
        node, path = self.root, []
        for key in self._page_keys(tokens):
            nxt = node.children.get(key)
            if nxt is None:
                break
            path.append(nxt)
            node = nxt
        for nd in path:
            nd.last = self.clock
        m = window_safe_pages([nd.swa for nd in path], self.pool.P, self.pool.W)
        return m, [nd.full for nd in path[:m]], [nd.swa for nd in path[:m]], len(path)

    # ------------------------------------------------------------- insert
    def insert(self, seq, tokens):
        """Store the whole pages of sequence seq's first len(tokens) tokens
        (its Full pages must all be present). Returns the new node count."""
        pool, s = self.pool, int(seq)
        keys = self._page_keys(tokens)
        if len(tokens) > pool.seq_len[s]:
            raise ValueError("more tokens than the sequence holds")
        for p in range(len(keys)):
            if pool.full_bt[s, p] < 0:
                raise ValueError("sequence page without a Full page")
        self.clock += 1
        node, created = self.root, 0
        for p, key in enumerate(keys):
            nxt = node.children.get(key)
            if nxt is None:
                full, swa = int(pool.full_bt[s, p]), int(pool.swa_bt[s, p])
                nxt = Node(key, full, swa, node, self.next_id, p)
                self.next_id += 1
                pool.ref_full(full)
                if swa >= 0:
                    pool.ref_swa(swa)
                node.children[key] = nxt
                created += 1
            elif nxt.swa < 0 and pool.swa_bt[s, p] >= 0:
                nxt.swa = int(pool.swa_bt[s, p])
                pool.ref_swa(nxt.swa)
            nxt.last = self.clock
            node = nxt
        return created

    # -------------------------------------------------------------- evict
    def _shallowest_leaf(self):
        """Pages D of the shallowest leaf at or below each node (by id)."""
        out = {}

        def visit(nd):
            if not nd.children:
                d = nd.index + 1
            else:
                d = min(visit(ch) for ch in nd.children.values())
            out[nd.id] = d
            return d

        for ch in self.root.children.values():
            visit(ch)
        return out

    def evict(self, want_full, want_swa):
        """Free at least want_swa SWA pages and want_full Full pages held by
        the tree alone, if it can. Returns (freed_full, freed_swa)."""
        pool, P, W = self.pool, self.pool.P, self.pool.W
        freed_full = freed_swa = 0
        if want_swa > 0:
            dmin = self._shallowest_leaf()
            cands = [nd for nd in self.nodes() if nd.swa >= 0 and pool.swa_ref[nd.swa] == 1]
            in_window = {nd.id: nd.index >= max(0, dmin[nd.id] * P - W) // P for nd in cands}
            for nd in sorted(cands, key=lambda nd: (in_window[nd.id], nd.last, nd.id)):
                if freed_swa >= want_swa:
                    break
                freed_swa += pool.unref_swa(nd.swa)
                nd.swa = -1
        while freed_full < want_full:
            leaves = [nd for nd in self.nodes() if not nd.children and pool.full_ref[nd.full] == 1]
            if not leaves:
                break
            nd = min(leaves, key=lambda nd: (nd.last, nd.id))
            freed_full += pool.unref_full(nd.full)
            if nd.swa >= 0:
                freed_swa += pool.unref_swa(nd.swa)
            del nd.parent.children[nd.tokens]
        return freed_full, freed_swa

    # ------------------------------------------------------------ release
    def clear(self):
        """Drop every node: the tree lets go of its pages, nodes in creation
        order, each Full page before its SWA page."""
        for nd in self.nodes():
            self.pool.unref_full(nd.full)
            if nd.swa >= 0:
                self.pool.unref_swa(nd.swa)
        self.root.children.clear()

    def stats(self):
        """(nodes, Full pages held, SWA pages held)."""
        nodes = self.nodes()
        return len(nodes), len(nodes), sum(nd.swa >= 0 for nd in nodes)
