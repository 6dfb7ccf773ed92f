// Internal declarations shared by the host-side sources of libhswa.
#pragma once

#include <cstdint>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "hswa.h"

// An NVTX range around one ABI call, so that a profile of a serving step can
// be split by call (the kernels each call launches sit inside its range).
// Without a profiler attached a push / pop costs a function-pointer test.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define HSWA_NVTX(name) NvtxRange hswa_nvtx_range_(name)

// FIFO free list of page indices (ring buffer; never holds more than the
// pool's page count).
struct PageQueue {
    std::vector<int32_t> ring;
    int64_t head = 0;
    int64_t count = 0;

    void init(int32_t capacity, const int32_t *order) {
        ring.assign(capacity, 0);
        for (int32_t i = 0; i < capacity; ++i) ring[i] = order ? order[i] : i;
        head = 0;
        count = capacity;
    }
    int32_t pop() {
        int32_t v = ring[head];
        head = (head + 1) % (int64_t)ring.size();
        --count;
        return v;
    }
    void push(int32_t v) {
        ring[(head + count) % (int64_t)ring.size()] = v;
        ++count;
    }
    int32_t at(int64_t i) const { return ring[(head + i) % (int64_t)ring.size()]; }
};

struct hswa_pool {
    hswa_config cfg;
    PageQueue full_free, swa_free;
    std::vector<int32_t> full_bt, swa_bt;  // [max_seqs][max_pages_per_seq]
    std::vector<int32_t> seq_len;          // [max_seqs]
    // per sequence: no logical page below holds an SWA page (set_swa lowers
    // it, a release raises it), so a release scans only the pages it frees
    std::vector<int32_t> swa_low;          // [max_seqs]
    // holders of each page (sequence tables and prefix-tree nodes); a page
    // is on its free list exactly when its count is 0
    std::vector<int32_t> full_ref, swa_ref;
    int32_t trees = 0;  // prefix trees bound to this pool

    void ref_full(int32_t page) { ++full_ref[page]; }
    void ref_swa(int32_t page) { ++swa_ref[page]; }
    // one holder lets go; true if the page went back to the free list
    bool unref_full(int32_t page) {
        if (--full_ref[page] > 0) return false;
        full_free.push(page);
        return true;
    }
    bool unref_swa(int32_t page) {
        if (--swa_ref[page] > 0) return false;
        swa_free.push(page);
        return true;
    }
    int32_t take_full() {
        const int32_t page = full_free.pop();
        full_ref[page] = 1;
        return page;
    }
    int32_t take_swa() {
        const int32_t page = swa_free.pop();
        swa_ref[page] = 1;
        return page;
    }

    // Entries changed since the last hswa_sync_tables, as flat indices into
    // the concatenation [full_bt | swa_bt | seq_len]; each index listed once.
    std::vector<uint8_t> dirty_flag;
    std::vector<int64_t> dirty_list;
    bool need_full_upload = true;
    const void *last_dev[3] = {nullptr, nullptr, nullptr};

    // pinned staging for the table upload, and the event that says when the
    // last copy out of it has finished
    void *staging = nullptr;
    size_t staging_bytes = 0;
    void *staging_event = nullptr;  // cudaEvent_t
    int device = -1;

    int64_t table_entries() const { return (int64_t)cfg.max_seqs * cfg.max_pages_per_seq; }
    void mark(int64_t flat) {
        if (!dirty_flag[flat]) {
            dirty_flag[flat] = 1;
            dirty_list.push_back(flat);
        }
    }
    void set_full(int32_t s, int32_t p, int32_t v) {
        int64_t i = (int64_t)s * cfg.max_pages_per_seq + p;
        full_bt[i] = v;
        mark(i);
    }
    void set_swa(int32_t s, int32_t p, int32_t v) {
        int64_t i = (int64_t)s * cfg.max_pages_per_seq + p;
        swa_bt[i] = v;
        if (v >= 0 && p < swa_low[s]) swa_low[s] = p;
        mark(table_entries() + i);
    }
    void set_len(int32_t s, int32_t v) {
        seq_len[s] = v;
        mark(2 * table_entries() + s);
    }
};

// Releases the CUDA resources of a pool (defined with the CUDA sources).
void hswa_pool_release_device(hswa_pool *pool);
