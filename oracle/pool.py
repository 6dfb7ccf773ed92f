"""CPU oracle for the dual KV pool bookkeeping.

TEST INFRASTRUCTURE ONLY: used by tests/, __graft_entry__.smoke() and
bench.py's CPU baseline. It shares no code with the CUDA library.

Follows "MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 2.1
(KVCache Dual Pool; SWA-aware prefix cache tree):

* two physical pools, Full and SWA, each a set of pages of P token slots;
* one logical sequence view: logical page p of a sequence covers positions
  [p*P, (p+1)*P); the Full table ``full_bt[s][p]`` is authoritative and the
  Full->SWA mapping is the same logical index in ``swa_bt[s][p]`` (-1 when
  that page of the sequence holds no SWA slot);
* admission checks both capacities together (all or nothing);
* out-of-window SWA pages are released after a prefill chunk, at request
  end and every N decode tokens, keeping at least the last W tokens
  (the window-safety rule).

Readings taken where the pages are silent:
* free lists are FIFO queues initialised from a caller-given order;
  allocation pops from the head in ascending (sequence id, logical page);
  frees are appended in the same ascending order;
* a page is released when every token on it is older than the last W:
  (p + 1) * P <= L - W;
* a page may be held by several owners (a sequence's table and the prefix
  tree, or several sequences sharing a cached prefix): it counts its
  holders and goes back to the tail of its free list when the last one lets
  go. Without sharing every count is 1 and the rules above are unchanged.
"""
from __future__ import annotations

import collections

import numpy as np


class NoSpace(Exception):
    """Either pool lacks the pages a call needs; no state was changed."""


class DualPool:
    def __init__(self, window, page_size, full_pages, swa_pages, max_seqs,
                 max_pages_per_seq, full_free_order=None, swa_free_order=None):
        self.W = int(window)
        self.P = int(page_size)
        self.full_pages = int(full_pages)
        self.swa_pages = int(swa_pages)
        order_f = range(full_pages) if full_free_order is None else full_free_order
        order_s = range(swa_pages) if swa_free_order is None else swa_free_order
        self.full_free = collections.deque(int(x) for x in order_f)
        self.swa_free = collections.deque(int(x) for x in order_s)
        self.full_bt = np.full((max_seqs, max_pages_per_seq), -1, np.int32)
        self.swa_bt = np.full((max_seqs, max_pages_per_seq), -1, np.int32)
        self.seq_len = np.zeros(max_seqs, np.int64)
        self.full_ref = np.zeros(full_pages, np.int64)  # holders of each page
        self.swa_ref = np.zeros(swa_pages, np.int64)

    # ------------------------------------------------------------ holders
    def ref_full(self, page):
        self.full_ref[page] += 1

    def ref_swa(self, page):
        self.swa_ref[page] += 1

    def unref_full(self, page):
        """One holder lets go; True if the page went back to the free list."""
        self.full_ref[page] -= 1
        assert self.full_ref[page] >= 0
        if self.full_ref[page] == 0:
            self.full_free.append(int(page))
            return True
        return False

    def unref_swa(self, page):
        self.swa_ref[page] -= 1
        assert self.swa_ref[page] >= 0
        if self.swa_ref[page] == 0:
            self.swa_free.append(int(page))
            return True
        return False

    # ------------------------------------------------------------------ a1
    def reserve(self, seq_ids, n_new):
        """Reserve slots for n_new[i] new tokens of sequence seq_ids[i].

        seq_ids must be strictly ascending. Returns (full_slot, swa_slot),
        one int32 entry per new token, sequences concatenated in order:
        slot = physical_page * P + position mod P.
        """
        seq_ids = [int(s) for s in seq_ids]
        n_new = [int(n) for n in n_new]
        assert all(a < b for a, b in zip(seq_ids, seq_ids[1:]))
        P = self.P
        need_full, need_swa = [], []
        for s, n in zip(seq_ids, n_new):
            L = int(self.seq_len[s])
            if L + n > self.full_bt.shape[1] * P:
                raise ValueError("sequence exceeds max_pages_per_seq")
            if n == 0:
                continue
            for p in range(L // P, (L + n - 1) // P + 1):
                if self.full_bt[s, p] < 0:
                    need_full.append((s, p))
                if self.swa_bt[s, p] < 0:
                    need_swa.append((s, p))
        if len(need_full) > len(self.full_free) or len(need_swa) > len(self.swa_free):
            raise NoSpace()
        for s, p in need_full:
            self.full_bt[s, p] = self.full_free.popleft()
            self.full_ref[self.full_bt[s, p]] = 1
        for s, p in need_swa:
            self.swa_bt[s, p] = self.swa_free.popleft()
            self.swa_ref[self.swa_bt[s, p]] = 1
        full_slot, swa_slot = [], []
        for s, n in zip(seq_ids, n_new):
            L = int(self.seq_len[s])
            t = np.arange(L, L + n, dtype=np.int64)  # positions of the new tokens
            full_slot.append(self.full_bt[s, t // P].astype(np.int64) * P + t % P)
            swa_slot.append(self.swa_bt[s, t // P].astype(np.int64) * P + t % P)
            self.seq_len[s] = L + n
        if not full_slot:
            return np.zeros(0, np.int32), np.zeros(0, np.int32)
        return np.concatenate(full_slot).astype(np.int32), np.concatenate(swa_slot).astype(np.int32)

    # ------------------------------------------------------------------ a7
    def swa_release(self, seq_ids):
        """Free SWA pages whose tokens all lie before the last W tokens."""
        freed = 0
        for s in sorted(int(x) for x in seq_ids):
            L = int(self.seq_len[s])
            for p in range(self.swa_bt.shape[1]):
                if self.swa_bt[s, p] >= 0 and (p + 1) * self.P <= L - self.W:
                    freed += self.unref_swa(int(self.swa_bt[s, p]))
                    self.swa_bt[s, p] = -1
        return freed

    def seq_free(self, seq_ids):
        """Request end: return every page of the sequences to both pools."""
        for s in sorted(int(x) for x in seq_ids):
            for p in range(self.full_bt.shape[1]):
                if self.full_bt[s, p] >= 0:
                    self.unref_full(int(self.full_bt[s, p]))
                    self.full_bt[s, p] = -1
            for p in range(self.swa_bt.shape[1]):
                if self.swa_bt[s, p] >= 0:
                    self.unref_swa(int(self.swa_bt[s, p]))
                    self.swa_bt[s, p] = -1
            self.seq_len[s] = 0

    def swa_drop(self, seq_ids):
        """Evict the SWA segment alone; the Full segment stays."""
        freed = 0
        for s in sorted(int(x) for x in seq_ids):
            for p in range(self.swa_bt.shape[1]):
                if self.swa_bt[s, p] >= 0:
                    freed += self.unref_swa(int(self.swa_bt[s, p]))
                    self.swa_bt[s, p] = -1
        return freed

    def swa_restore(self, seq_ids):
        """Give SWA pages back to the in-window logical pages of each sequence
        (positions [L - min(L, W), L)) that hold none; all or nothing."""
        need = []
        for s in sorted(int(x) for x in seq_ids):
            L = int(self.seq_len[s])
            n = min(L, self.W)
            if n == 0:
                continue
            for p in range((L - n) // self.P, (L - 1) // self.P + 1):
                if self.swa_bt[s, p] < 0:
                    need.append((s, p))
        if len(need) > len(self.swa_free):
            raise NoSpace()
        for s, p in need:
            self.swa_bt[s, p] = self.swa_free.popleft()
            self.swa_ref[self.swa_bt[s, p]] = 1
        return len(need)

    # ------------------------------------------------------ shared prefix
    def share_prefix(self, s, full_pages, swa_pages):
        """Start empty sequence s on a cached prefix of n = len(full_pages)
        whole pages (MiMo Sec. 2.1, SWA-aware prefix cache tree: a hit reuses
        the Full segment and the SWA window). The sequence holds every Full
        page and the SWA pages of the logical pages that meet the last W
        positions [n*P - W, n*P); each must be held already (by the tree).
        Its length becomes n*P."""
        s = int(s)
        n = len(full_pages)
        if self.seq_len[s] != 0 or (self.full_bt[s] >= 0).any() or (self.swa_bt[s] >= 0).any():
            raise ValueError("sequence not empty")
        if n > self.full_bt.shape[1]:
            raise ValueError("prefix exceeds max_pages_per_seq")
        first = max(0, n * self.P - self.W) // self.P
        for p in range(n):
            if not (0 <= full_pages[p] < self.full_pages) or self.full_ref[full_pages[p]] == 0:
                raise ValueError("Full page not held")
        for p in range(first, n):
            if not (0 <= swa_pages[p] < self.swa_pages) or self.swa_ref[swa_pages[p]] == 0:
                raise ValueError("SWA window page not held")
        for p in range(n):
            self.full_bt[s, p] = full_pages[p]
            self.ref_full(int(full_pages[p]))
        for p in range(first, n):
            self.swa_bt[s, p] = swa_pages[p]
            self.ref_swa(int(swa_pages[p]))
        self.seq_len[s] = n * self.P

    # ------------------------------------------------------------ queries
    def live_swa_pages(self, s):
        return int(np.count_nonzero(self.swa_bt[s] >= 0))

    def live_full_pages(self, s):
        return int(np.count_nonzero(self.full_bt[s] >= 0))
