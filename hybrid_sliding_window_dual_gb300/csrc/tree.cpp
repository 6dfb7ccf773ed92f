// SWA-aware prefix cache tree on the host.
//
// "MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 2.1, SWA-aware
// prefix cache tree: with an SWA pool that drops out-of-window slots, equal
// tokens no longer mean reusable KV. The tree
//   1. trims a match to the window-safety length: the last W positions of
//      the matched prefix must still have SWA slots; past that is a miss;
//   2. (its pages are released with the request lifecycle by the pool);
//   3. keeps two indexes per node, a Full page and an SWA page, evicted
//      apart: out-of-window SWA pages alone (the Full prefix stays reusable)
//      or whole nodes.
//
// One node per page of P tokens. The tree holds one reference on every page
// it stores; a page goes back to its pool's free list when no sequence and
// no node holds it. Every choice is deterministic (a logical clock advanced
// by each match and insert, then creation order), so the tree and the pool
// tables are a function of the call sequence.
//
// Eviction is incremental: the leaves are kept ordered by (clock, id) and
// the nodes holding an SWA page by (inside a window, clock, id), where
// "inside a window" depends on the shallowest leaf below the node, which is
// kept per node and updated upward only when the tree's shape changes. A
// call then costs O((pages freed + held pages passed over) log n) instead of
// a pass over the whole tree.
#include <algorithm>
#include <map>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "internal.h"

namespace {

struct TreeNode {
    int32_t id = -1;     // creation order (a child is always newer than its parent)
    int32_t index = -1;  // logical page index of the page in its sequences
    int32_t full = -1, swa = -1;
    uint64_t last = 0;   // clock of the last match or insert through the node
    int64_t dmin = 0;    // pages of the shallowest leaf at or below the node
    TreeNode *parent = nullptr;
    std::vector<int32_t> tokens;  // the page's P tokens
    uint64_t hash = 0;            // of tokens
    std::unordered_multimap<uint64_t, TreeNode *> children;  // by token hash
};

// 64-bit hash of a page's tokens (FNV-1a over the 32-bit values, then a
// final mix); equal hashes are confirmed by comparing the tokens.
uint64_t page_hash(const int32_t *t, int64_t n) {
    uint64_t h = 1469598103934665603ull;
    for (int64_t i = 0; i < n; ++i) {
        h ^= (uint32_t)t[i];
        h *= 1099511628211ull;
    }
    h ^= h >> 33;
    h *= 0xff51afd7ed558ccdull;
    h ^= h >> 33;
    return h;
}

TreeNode *find_child(TreeNode *node, const int32_t *t, int64_t n, uint64_t h) {
    auto range = node->children.equal_range(h);
    for (auto it = range.first; it != range.second; ++it)
        if (std::equal(t, t + n, it->second->tokens.begin())) return it->second;
    return nullptr;
}

using LeafKey = std::pair<uint64_t, int32_t>;       // (last, id)
using SwaKey = std::tuple<int, uint64_t, int32_t>;  // (inside a window, last, id)

}  // namespace

struct hswa_tree {
    hswa_pool *pool = nullptr;
    TreeNode root;
    uint64_t clock = 0;
    int32_t next_id = 0;
    int32_t n_swa = 0;                    // nodes holding an SWA page
    std::map<int32_t, TreeNode *> nodes;  // every node but the root, by id
    std::set<LeafKey> leaves;             // every leaf
    std::set<SwaKey> swa_nodes;           // every node holding an SWA page
};

namespace {

bool in_window(const hswa_tree *t, const TreeNode *nd) {
    const int64_t P = t->pool->cfg.page_size, W = t->pool->cfg.window;
    return nd->index >= std::max<int64_t>(0, nd->dmin * P - W) / P;
}

// Take a node out of the ordered sets before one of its keys (last, dmin,
// SWA page, children) changes, and put it back afterwards.
void unindex(hswa_tree *t, const TreeNode *nd) {
    if (nd->children.empty()) t->leaves.erase(LeafKey(nd->last, nd->id));
    if (nd->swa >= 0) t->swa_nodes.erase(SwaKey(in_window(t, nd) ? 1 : 0, nd->last, nd->id));
}

void reindex(hswa_tree *t, const TreeNode *nd) {
    if (nd->children.empty()) t->leaves.insert(LeafKey(nd->last, nd->id));
    if (nd->swa >= 0) t->swa_nodes.insert(SwaKey(in_window(t, nd) ? 1 : 0, nd->last, nd->id));
}

constexpr int64_t kNoLeaf = INT64_MAX;

// One child of nd went from shallowest-leaf depth a to b (a = kNoLeaf: the
// child is new; b = kNoLeaf: it was removed). Update the depths from nd up
// to the root, stopping where they no longer change. A node's children are
// scanned only when the changed child held its minimum and got deeper or
// went; otherwise the new minimum follows from the old one (a prompt shared
// by many requests has many children).
void update_dmin_up(hswa_tree *t, TreeNode *nd, int64_t a, int64_t b) {
    for (; nd && nd != &t->root; nd = nd->parent) {
        const int64_t D = nd->dmin;
        int64_t d;
        if (nd->children.empty()) {
            d = (int64_t)nd->index + 1;  // a leaf now
        } else if (a == kNoLeaf && nd->children.size() == 1) {
            d = b;  // a leaf until this child came
        } else if (b <= D) {
            d = b;  // the changed child is (one of) the shallowest
        } else if (a > D) {
            d = D;  // the changed child did not hold the minimum
        } else {
            d = kNoLeaf;
            for (auto &ch : nd->children) d = std::min(d, ch.second->dmin);
        }
        if (d == D) return;
        // the leaf-set key (last, id) holds no depth; the SWA-node key moves
        // only if the node's window side flips (near the leaf it is over)
        const bool was_in = in_window(t, nd);
        nd->dmin = d;
        if (nd->swa >= 0 && in_window(t, nd) != was_in) {
            t->swa_nodes.erase(SwaKey(was_in ? 1 : 0, nd->last, nd->id));
            t->swa_nodes.insert(SwaKey(was_in ? 0 : 1, nd->last, nd->id));
        }
        a = D;
        b = d;
    }
}

void touch(hswa_tree *t, TreeNode *nd, uint64_t clock) {
    if (nd->last == clock) return;
    unindex(t, nd);
    nd->last = clock;
    reindex(t, nd);
}

// Largest m <= n with an SWA page on every logical page that meets the last
// W positions [m*P - W, m*P) of an m-page prefix.
int32_t window_safe_pages(const std::vector<TreeNode *> &path, int64_t P, int64_t W) {
    const int32_t n = (int32_t)path.size();
    // missing[p]: pages without an SWA page among the first p, for O(1) range checks
    std::vector<int32_t> missing(n + 1, 0);
    for (int32_t p = 0; p < n; ++p) missing[p + 1] = missing[p] + (path[p]->swa < 0);
    for (int32_t m = n; m > 0; --m) {
        const int64_t first = std::max<int64_t>(0, m * P - W) / P;
        if (missing[m] - missing[first] == 0) return m;
    }
    return 0;
}

// Remove a leaf (its pages already let go of) and update its parent.
void remove_leaf(hswa_tree *t, TreeNode *nd) {
    unindex(t, nd);
    if (nd->swa >= 0) --t->n_swa;
    TreeNode *parent = nd->parent;
    const int64_t gone = nd->dmin;
    if (parent != &t->root) unindex(t, parent);
    auto range = parent->children.equal_range(nd->hash);
    for (auto it = range.first; it != range.second; ++it)
        if (it->second == nd) {
            parent->children.erase(it);
            break;
        }
    t->nodes.erase(nd->id);
    delete nd;
    if (parent != &t->root) {
        reindex(t, parent);  // a leaf now, if that was its last child
        update_dmin_up(t, parent, gone, kNoLeaf);
    }
}

}  // namespace

extern "C" int hswa_tree_create(hswa_pool *pool, hswa_tree **out) {
    if (!pool || !out) return HSWA_ERR_INVALID_ARG;
    hswa_tree *t = new (std::nothrow) hswa_tree();
    if (!t) return HSWA_ERR_INVALID_ARG;
    t->pool = pool;
    ++pool->trees;
    *out = t;
    return HSWA_OK;
}

extern "C" int hswa_tree_destroy(hswa_tree *t) {
    if (!t) return HSWA_ERR_INVALID_ARG;
    // let go of every page, nodes in creation order, Full page before SWA page
    for (auto &kv : t->nodes) {
        t->pool->unref_full(kv.second->full);
        if (kv.second->swa >= 0) t->pool->unref_swa(kv.second->swa);
    }
    for (auto &kv : t->nodes) delete kv.second;
    --t->pool->trees;
    delete t;
    return HSWA_OK;
}

extern "C" int hswa_tree_match(hswa_tree *t, const int32_t *tokens, int64_t n_tokens, int32_t *full_pages_out,
                               int32_t *swa_pages_out, int32_t cap_pages, int32_t *n_pages_out,
                               int32_t *raw_pages_out) {
    if (!t || n_tokens < 0 || (n_tokens > 0 && !tokens) || cap_pages < 0) return HSWA_ERR_INVALID_ARG;
    const int64_t P = t->pool->cfg.page_size, W = t->pool->cfg.window;
    const int64_t n_pages = n_tokens / P;
    if (cap_pages < std::min<int64_t>(n_pages, t->pool->cfg.max_pages_per_seq) ||
        (cap_pages > 0 && (!full_pages_out || !swa_pages_out)))
        return HSWA_ERR_INVALID_ARG;
    ++t->clock;
    std::vector<TreeNode *> path;
    TreeNode *node = &t->root;
    for (int64_t p = 0; p < n_pages; ++p) {
        const int32_t *pt = tokens + p * P;
        node = find_child(node, pt, P, page_hash(pt, P));
        if (!node) break;
        path.push_back(node);
    }
    for (TreeNode *nd : path) touch(t, nd, t->clock);
    const int32_t m = window_safe_pages(path, P, W);
    for (int32_t p = 0; p < m; ++p) {
        full_pages_out[p] = path[p]->full;
        swa_pages_out[p] = path[p]->swa;
    }
    if (n_pages_out) *n_pages_out = m;
    if (raw_pages_out) *raw_pages_out = (int32_t)path.size();
    return HSWA_OK;
}

extern "C" int hswa_tree_insert(hswa_tree *t, int32_t seq_id, const int32_t *tokens, int64_t n_tokens,
                                int32_t *n_new_out) {
    if (!t || n_tokens < 0 || (n_tokens > 0 && !tokens)) return HSWA_ERR_INVALID_ARG;
    hswa_pool *pool = t->pool;
    if (seq_id < 0 || seq_id >= pool->cfg.max_seqs || n_tokens > pool->seq_len[seq_id]) return HSWA_ERR_INVALID_ARG;
    const int64_t P = pool->cfg.page_size, MP = pool->cfg.max_pages_per_seq;
    const int64_t n_pages = n_tokens / P;
    const int32_t *frow = &pool->full_bt[(int64_t)seq_id * MP];
    const int32_t *srow = &pool->swa_bt[(int64_t)seq_id * MP];
    for (int64_t p = 0; p < n_pages; ++p)
        if (frow[p] < 0) return HSWA_ERR_INVALID_ARG;
    const uint64_t clock = ++t->clock;
    TreeNode *node = &t->root;
    TreeNode *attach = nullptr;  // the existing node the new chain hangs from
    int32_t created = 0;
    for (int64_t p = 0; p < n_pages; ++p) {
        const int32_t *pt = tokens + p * P;
        const uint64_t h = page_hash(pt, P);
        TreeNode *nxt = find_child(node, pt, P, h);
        if (!nxt) {
            nxt = new TreeNode();
            nxt->id = t->next_id++;
            nxt->index = (int32_t)p;
            nxt->full = frow[p];
            nxt->swa = srow[p];
            nxt->parent = node;
            nxt->tokens.assign(pt, pt + P);
            nxt->hash = h;
            nxt->last = clock;
            nxt->dmin = n_pages;  // new nodes form one chain down to the leaf at page n_pages - 1
            pool->ref_full(nxt->full);
            if (nxt->swa >= 0) {
                pool->ref_swa(nxt->swa);
                ++t->n_swa;
            }
            if (node != &t->root) unindex(t, node);  // it may stop being a leaf
            node->children.emplace(h, nxt);
            if (node != &t->root) reindex(t, node);
            reindex(t, nxt);
            t->nodes.emplace(nxt->id, nxt);
            if (!created) attach = node;
            ++created;
        } else {
            if (nxt->swa < 0 && srow[p] >= 0) {  // the sequence recomputed a lost window page
                unindex(t, nxt);
                nxt->swa = srow[p];
                pool->ref_swa(nxt->swa);
                ++t->n_swa;
                reindex(t, nxt);
            }
            touch(t, nxt, clock);
        }
        node = nxt;
    }
    // the node the chain hangs from gained a child whose shallowest leaf is
    // n_pages deep
    if (created) update_dmin_up(t, attach, kNoLeaf, n_pages);
    if (n_new_out) *n_new_out = created;
    return HSWA_OK;
}

extern "C" int hswa_tree_evict(hswa_tree *t, int32_t want_full, int32_t want_swa, int32_t *freed_full_out,
                               int32_t *freed_swa_out) {
    if (!t || want_full < 0 || want_swa < 0) return HSWA_ERR_INVALID_ARG;
    hswa_pool *pool = t->pool;
    int32_t freed_full = 0, freed_swa = 0;
    // SWA pages only the tree holds: outside every window below them first,
    // then inside; oldest first, then creation order. Freeing one node's SWA
    // page moves no other node in the order.
    for (auto it = t->swa_nodes.begin(); freed_swa < want_swa && it != t->swa_nodes.end();) {
        TreeNode *nd = t->nodes.at(std::get<2>(*it));
        if (pool->swa_ref[nd->swa] != 1) {
            ++it;
            continue;
        }
        it = t->swa_nodes.erase(it);
        freed_swa += pool->unref_swa(nd->swa);
        nd->swa = -1;
        --t->n_swa;
    }
    // leaves whose Full page only the tree holds, oldest first; a parent left
    // without children becomes a leaf and a candidate. Leaves held by a
    // sequence are set aside for the rest of the call.
    std::vector<LeafKey> held;
    while (freed_full < want_full && !t->leaves.empty()) {
        const LeafKey k = *t->leaves.begin();
        TreeNode *nd = t->nodes.at(k.second);
        if (pool->full_ref[nd->full] != 1) {
            held.push_back(k);
            t->leaves.erase(t->leaves.begin());
            continue;
        }
        freed_full += pool->unref_full(nd->full);
        if (nd->swa >= 0) freed_swa += pool->unref_swa(nd->swa);
        remove_leaf(t, nd);
    }
    for (const LeafKey &k : held) t->leaves.insert(k);
    if (freed_full_out) *freed_full_out = freed_full;
    if (freed_swa_out) *freed_swa_out = freed_swa;
    return HSWA_OK;
}

extern "C" int hswa_tree_stats(const hswa_tree *t, int32_t *n_nodes, int32_t *full_held, int32_t *swa_held) {
    if (!t) return HSWA_ERR_INVALID_ARG;
    if (n_nodes) *n_nodes = (int32_t)t->nodes.size();
    if (full_held) *full_held = (int32_t)t->nodes.size();
    if (swa_held) *swa_held = t->n_swa;
    return HSWA_OK;
}

extern "C" int hswa_tree_nodes(const hswa_tree *t, int32_t *out, int32_t cap, int32_t *count) {
    if (!t || cap < 0 || (cap > 0 && !out)) return HSWA_ERR_INVALID_ARG;
    // per node, in creation order: id, parent id (-1 = root), logical page, Full page, SWA page
    int32_t i = 0;
    for (auto &kv : t->nodes) {
        const TreeNode *nd = kv.second;
        if ((int64_t)(i + 1) * 5 <= cap) {
            int32_t *r = out + (int64_t)i * 5;
            r[0] = nd->id;
            r[1] = nd->parent == &t->root ? -1 : nd->parent->id;
            r[2] = nd->index;
            r[3] = nd->full;
            r[4] = nd->swa;
        }
        ++i;
    }
    if (count) *count = i;
    return HSWA_OK;
}
