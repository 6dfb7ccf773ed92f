// Dual KV pool bookkeeping on the host.
//
// "MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 2.1:
//  * KVCache Dual Pool -- separate Full and SWA pools behind one logical
//    sequence view; the Full index is authoritative and the Full -> SWA
//    mapping shares its logical page index; admission checks both capacities.
//  * SWA-aware prefix cache tree -- out-of-window SWA slots are released
//    after prefill chunks, at request end and every N decode tokens, keeping
//    at least the last W tokens; the SWA segment can be evicted alone.
//
// Free lists are FIFO queues; pages are taken from the head and returned to
// the tail, always in ascending (sequence id, logical page) order, so that
// the tables are a deterministic function of the call sequence. A page can
// have several holders (sequence tables and prefix-tree nodes, which share
// cached prefixes); it returns to its free list when the last one lets go.
#include <algorithm>
#include <cstring>
#include <new>

#include "internal.h"

namespace {

bool valid_config(const hswa_config *c) {
    return c && c->window > 0 && c->page_size > 0 && c->n_q_heads > 0 && c->n_kv_heads > 0 &&
           c->n_q_heads % c->n_kv_heads == 0 && c->head_dim > 0 &&
           (c->dtype == HSWA_DTYPE_F32 || c->dtype == HSWA_DTYPE_BF16 || c->dtype == HSWA_DTYPE_FP8_E4M3) &&
           c->full_pages > 0 &&
           c->swa_pages > 0 && c->max_seqs > 0 && c->max_pages_per_seq > 0 &&
           (int64_t)c->max_pages_per_seq * c->page_size <= INT32_MAX &&
           (int64_t)c->full_pages * c->page_size <= INT32_MAX &&
           (int64_t)c->swa_pages * c->page_size <= INT32_MAX;
}

bool valid_order(const int32_t *order, int32_t n) {
    if (!order) return true;
    std::vector<uint8_t> seen(n, 0);
    for (int32_t i = 0; i < n; ++i) {
        if (order[i] < 0 || order[i] >= n || seen[order[i]]) return false;
        seen[order[i]] = 1;
    }
    return true;
}

// Sorted copy of seq_ids, or false if an id is out of range or repeated.
bool sorted_ids(const hswa_pool *pool, int n, const int32_t *seq_ids, std::vector<int32_t> &out) {
    if (n < 0 || (n > 0 && !seq_ids)) return false;
    out.assign(seq_ids, seq_ids + n);
    std::sort(out.begin(), out.end());
    for (int i = 0; i < n; ++i) {
        if (out[i] < 0 || out[i] >= pool->cfg.max_seqs) return false;
        if (i > 0 && out[i] == out[i - 1]) return false;
    }
    return true;
}

}  // namespace

extern "C" int hswa_pool_create(const hswa_config *cfg, const int32_t *full_free_order,
                                const int32_t *swa_free_order, hswa_pool **out) {
    if (!out || !valid_config(cfg)) return HSWA_ERR_INVALID_ARG;
    if (!valid_order(full_free_order, cfg->full_pages) || !valid_order(swa_free_order, cfg->swa_pages))
        return HSWA_ERR_INVALID_ARG;
    hswa_pool *p = new (std::nothrow) hswa_pool();
    if (!p) return HSWA_ERR_INVALID_ARG;
    p->cfg = *cfg;
    p->full_free.init(cfg->full_pages, full_free_order);
    p->swa_free.init(cfg->swa_pages, swa_free_order);
    const int64_t entries = p->table_entries();
    p->full_bt.assign(entries, -1);
    p->swa_bt.assign(entries, -1);
    p->seq_len.assign(cfg->max_seqs, 0);
    p->swa_low.assign(cfg->max_seqs, 0);
    p->full_ref.assign(cfg->full_pages, 0);
    p->swa_ref.assign(cfg->swa_pages, 0);
    p->dirty_flag.assign(2 * entries + cfg->max_seqs, 0);
    *out = p;
    return HSWA_OK;
}

extern "C" int hswa_pool_destroy(hswa_pool *pool) {
    if (!pool || pool->trees > 0) return HSWA_ERR_INVALID_ARG;  // destroy its prefix trees first
    hswa_pool_release_device(pool);
    delete pool;
    return HSWA_OK;
}

extern "C" int hswa_reserve(hswa_pool *pool, int n, const int32_t *seq_ids, const int32_t *n_new,
                            int32_t *full_slot_out, int32_t *swa_slot_out) {
    HSWA_NVTX("hswa_reserve");
    if (!pool || n < 0 || (n > 0 && (!seq_ids || !n_new))) return HSWA_ERR_INVALID_ARG;
    const int32_t P = pool->cfg.page_size, MP = pool->cfg.max_pages_per_seq;
    // validate and count the pages each pool must give
    int64_t need_full = 0, need_swa = 0;
    for (int i = 0; i < n; ++i) {
        const int32_t s = seq_ids[i];
        if (s < 0 || s >= pool->cfg.max_seqs || n_new[i] < 0) return HSWA_ERR_INVALID_ARG;
        if (i > 0 && s <= seq_ids[i - 1]) return HSWA_ERR_INVALID_ARG;
        const int64_t L = pool->seq_len[s];
        if (L + n_new[i] > (int64_t)MP * P) return HSWA_ERR_INVALID_ARG;
        if (n_new[i] == 0) continue;
        const int32_t *frow = &pool->full_bt[(int64_t)s * MP];
        const int32_t *srow = &pool->swa_bt[(int64_t)s * MP];
        for (int64_t p = L / P; p <= (L + n_new[i] - 1) / P; ++p) {
            need_full += frow[p] < 0;
            need_swa += srow[p] < 0;
        }
    }
    if (need_full > pool->full_free.count || need_swa > pool->swa_free.count)
        return HSWA_ERR_NO_SPACE;
    // allocate: ascending (sequence, logical page), Full and SWA lists apart
    int64_t out = 0;
    for (int i = 0; i < n; ++i) {
        const int32_t s = seq_ids[i];
        const int64_t L = pool->seq_len[s];
        if (n_new[i] == 0) continue;
        for (int64_t p = L / P; p <= (L + n_new[i] - 1) / P; ++p) {
            if (pool->full_bt[(int64_t)s * MP + p] < 0) pool->set_full(s, (int32_t)p, pool->take_full());
            if (pool->swa_bt[(int64_t)s * MP + p] < 0) pool->set_swa(s, (int32_t)p, pool->take_swa());
        }
        for (int64_t t = L; t < L + n_new[i]; ++t, ++out) {
            if (full_slot_out)
                full_slot_out[out] = pool->full_bt[(int64_t)s * MP + t / P] * P + (int32_t)(t % P);
            if (swa_slot_out)
                swa_slot_out[out] = pool->swa_bt[(int64_t)s * MP + t / P] * P + (int32_t)(t % P);
        }
        pool->set_len(s, (int32_t)(L + n_new[i]));
    }
    return HSWA_OK;
}

extern "C" int hswa_swa_release(hswa_pool *pool, int n, const int32_t *seq_ids, int32_t *n_freed_out) {
    HSWA_NVTX("hswa_swa_release");
    std::vector<int32_t> ids;
    if (!pool || !sorted_ids(pool, n, seq_ids, ids)) return HSWA_ERR_INVALID_ARG;
    const int64_t P = pool->cfg.page_size, W = pool->cfg.window, MP = pool->cfg.max_pages_per_seq;
    int32_t freed = 0;
    for (int32_t s : ids) {
        const int64_t L = pool->seq_len[s];
        // pages p with (p + 1) * P <= L - W hold only tokens older than the window
        const int64_t n_old = std::min<int64_t>(L - W > 0 ? (L - W) / P : 0, MP);
        for (int64_t p = pool->swa_low[s]; p < n_old; ++p) {  // pages below hold none
            const int32_t page = pool->swa_bt[s * MP + p];
            if (page < 0) continue;
            freed += pool->unref_swa(page);
            pool->set_swa(s, (int32_t)p, -1);
        }
        if (n_old > pool->swa_low[s]) pool->swa_low[s] = (int32_t)n_old;
    }
    if (n_freed_out) *n_freed_out = freed;
    return HSWA_OK;
}

extern "C" int hswa_seq_free(hswa_pool *pool, int n, const int32_t *seq_ids) {
    HSWA_NVTX("hswa_seq_free");
    std::vector<int32_t> ids;
    if (!pool || !sorted_ids(pool, n, seq_ids, ids)) return HSWA_ERR_INVALID_ARG;
    const int64_t MP = pool->cfg.max_pages_per_seq;
    for (int32_t s : ids) {
        for (int64_t p = 0; p < MP; ++p) {
            const int32_t page = pool->full_bt[s * MP + p];
            if (page >= 0) {
                pool->unref_full(page);
                pool->set_full(s, (int32_t)p, -1);
            }
        }
        for (int64_t p = 0; p < MP; ++p) {
            const int32_t page = pool->swa_bt[s * MP + p];
            if (page >= 0) {
                pool->unref_swa(page);
                pool->set_swa(s, (int32_t)p, -1);
            }
        }
        pool->set_len(s, 0);
    }
    return HSWA_OK;
}

extern "C" int hswa_swa_drop(hswa_pool *pool, int n, const int32_t *seq_ids, int32_t *n_freed_out) {
    HSWA_NVTX("hswa_swa_drop");
    std::vector<int32_t> ids;
    if (!pool || !sorted_ids(pool, n, seq_ids, ids)) return HSWA_ERR_INVALID_ARG;
    const int64_t MP = pool->cfg.max_pages_per_seq;
    int32_t freed = 0;
    for (int32_t s : ids) {
        for (int64_t p = 0; p < MP; ++p) {
            const int32_t page = pool->swa_bt[s * MP + p];
            if (page < 0) continue;
            freed += pool->unref_swa(page);
            pool->set_swa(s, (int32_t)p, -1);
        }
    }
    if (n_freed_out) *n_freed_out = freed;
    return HSWA_OK;
}

extern "C" int hswa_swa_restore(hswa_pool *pool, int n, const int32_t *seq_ids, int32_t *n_alloc_out) {
    HSWA_NVTX("hswa_swa_restore");
    std::vector<int32_t> ids;
    if (!pool || !sorted_ids(pool, n, seq_ids, ids)) return HSWA_ERR_INVALID_ARG;
    const int64_t P = pool->cfg.page_size, W = pool->cfg.window, MP = pool->cfg.max_pages_per_seq;
    int64_t need = 0;
    for (int32_t s : ids) {
        const int64_t L = pool->seq_len[s], nw = std::min(L, W);
        if (nw == 0) continue;
        for (int64_t p = (L - nw) / P; p <= (L - 1) / P; ++p) need += pool->swa_bt[s * MP + p] < 0;
    }
    if (need > pool->swa_free.count) return HSWA_ERR_NO_SPACE;
    for (int32_t s : ids) {
        const int64_t L = pool->seq_len[s], nw = std::min(L, W);
        if (nw == 0) continue;
        for (int64_t p = (L - nw) / P; p <= (L - 1) / P; ++p)
            if (pool->swa_bt[s * MP + p] < 0) pool->set_swa(s, (int32_t)p, pool->take_swa());
    }
    if (n_alloc_out) *n_alloc_out = (int32_t)need;
    return HSWA_OK;
}

extern "C" int hswa_seq_share_prefix(hswa_pool *pool, int32_t seq_id, int32_t n_pages, const int32_t *full_pages,
                                     const int32_t *swa_pages) {
    if (!pool || seq_id < 0 || seq_id >= pool->cfg.max_seqs || n_pages < 0 ||
        n_pages > pool->cfg.max_pages_per_seq || (n_pages > 0 && (!full_pages || !swa_pages)))
        return HSWA_ERR_INVALID_ARG;
    const int64_t P = pool->cfg.page_size, W = pool->cfg.window, MP = pool->cfg.max_pages_per_seq;
    if (pool->seq_len[seq_id] != 0) return HSWA_ERR_INVALID_ARG;
    for (int64_t p = 0; p < MP; ++p)
        if (pool->full_bt[seq_id * MP + p] >= 0 || pool->swa_bt[seq_id * MP + p] >= 0) return HSWA_ERR_INVALID_ARG;
    // logical pages meeting the last W positions [n*P - W, n*P) of the prefix
    const int64_t first = std::max<int64_t>(0, n_pages * P - W) / P;
    for (int32_t p = 0; p < n_pages; ++p)
        if (full_pages[p] < 0 || full_pages[p] >= pool->cfg.full_pages || pool->full_ref[full_pages[p]] == 0)
            return HSWA_ERR_INVALID_ARG;
    for (int64_t p = first; p < n_pages; ++p)
        if (swa_pages[p] < 0 || swa_pages[p] >= pool->cfg.swa_pages || pool->swa_ref[swa_pages[p]] == 0)
            return HSWA_ERR_INVALID_ARG;
    for (int32_t p = 0; p < n_pages; ++p) {
        pool->set_full(seq_id, p, full_pages[p]);
        pool->ref_full(full_pages[p]);
    }
    for (int64_t p = first; p < n_pages; ++p) {
        pool->set_swa(seq_id, (int32_t)p, swa_pages[p]);
        pool->ref_swa(swa_pages[p]);
    }
    pool->set_len(seq_id, (int32_t)(n_pages * P));
    return HSWA_OK;
}

extern "C" int hswa_get_page_refs(const hswa_pool *pool, int kind, int32_t *out, int32_t cap) {
    if (!pool || (kind != HSWA_KIND_FULL && kind != HSWA_KIND_SWA) || cap < 0 || (cap > 0 && !out))
        return HSWA_ERR_INVALID_ARG;
    const std::vector<int32_t> &r = kind == HSWA_KIND_FULL ? pool->full_ref : pool->swa_ref;
    for (int64_t i = 0; i < (int64_t)r.size() && i < cap; ++i) out[i] = r[i];
    return HSWA_OK;
}

extern "C" int hswa_get_tables(const hswa_pool *pool, int32_t *full_bt, int32_t *swa_bt, int32_t *seq_len) {
    if (!pool) return HSWA_ERR_INVALID_ARG;
    const size_t bytes = sizeof(int32_t) * (size_t)pool->table_entries();
    if (full_bt) std::memcpy(full_bt, pool->full_bt.data(), bytes);
    if (swa_bt) std::memcpy(swa_bt, pool->swa_bt.data(), bytes);
    if (seq_len) std::memcpy(seq_len, pool->seq_len.data(), sizeof(int32_t) * pool->cfg.max_seqs);
    return HSWA_OK;
}

extern "C" int hswa_get_free_list(const hswa_pool *pool, int kind, int32_t *out, int32_t cap, int32_t *count) {
    if (!pool || (kind != HSWA_KIND_FULL && kind != HSWA_KIND_SWA) || cap < 0) return HSWA_ERR_INVALID_ARG;
    const PageQueue &q = kind == HSWA_KIND_FULL ? pool->full_free : pool->swa_free;
    if (count) *count = (int32_t)q.count;
    if (out)
        for (int64_t i = 0; i < q.count && i < cap; ++i) out[i] = q.at(i);
    return HSWA_OK;
}

extern "C" const char *hswa_status_string(int status) {
    switch (status) {
        case HSWA_OK: return "ok";
        case HSWA_ERR_INVALID_ARG: return "invalid argument";
        case HSWA_ERR_NO_SPACE: return "no space in the Full or SWA pool";
        case HSWA_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or head ratio";
        case HSWA_ERR_CUDA: return "CUDA error";
        case HSWA_ERR_TIMEOUT: return "bounded device wait timed out";
        case HSWA_ERR_BOUNDS: return "device index check failed";
        default: return "unknown status";
    }
}
