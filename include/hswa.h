/*
 * hswa.h -- Hybrid sliding-window attention over a dual KV pool (GB300, sm_103a).
 *
 * C ABI of libhswa.so. Plain pointers and sizes only.
 *
 * Method: "MiMo-V2.5 Series Inference Full-Link Optimization: Pushing Hybrid
 * SWA Efficiency to the Extreme".
 *   Sec. 1.1 (Computational Complexity Analysis): most layers attend only to
 *     a sliding window of W = 128 tokens, a few (10 of 70) to the whole
 *     sequence; prefill is close to compute-bound.
 *   Sec. 1.2 (KVCache Storage Analysis): SWA layers keep only the window;
 *     decode is close to memory-bandwidth-bound.
 *   Sec. 2.1 (KVCache Dual Pool): a Full pool (O(N) per sequence) and an SWA
 *     pool (O(W)), one logical sequence view with the Full index
 *     authoritative and a Full -> SWA mapping, a joint capacity check at
 *     admission, cross-tier transfer of SWA-mask data only, and release of
 *     out-of-window SWA slots tied to the request lifecycle (after each
 *     prefill chunk, at request end, every N decode tokens) with at least the
 *     last W tokens kept (window-safety rule).
 *
 * Conventions shared by every call
 * --------------------------------
 * Pool layout. A layer's K pool and V pool are each
 *     [num_pages][n_kv_heads][page_size][head_dim]
 * elements of the pool dtype (fp32 or bf16), row-major. num_pages is
 * cfg.full_pages for a Full layer and cfg.swa_pages for an SWA layer. All
 * layers of one kind share one block table: a page index means the same
 * page in every layer of that kind.
 *
 * Logical pages. Token position t of a sequence lies on logical page
 * t / page_size, row t % page_size. full_bt[s][p] is the Full page of
 * logical page p of sequence s; swa_bt[s][p] is its SWA page, or -1 when
 * that logical page holds no SWA slot (released, or never reserved). Both
 * tables are int32 [max_seqs][max_pages_per_seq], row-major. A slot is
 * page * page_size + t % page_size.
 *
 * Sequences. Sequence ids are 0 .. max_seqs-1. Batched device calls work on
 * sequences 0 .. n_seqs-1: row i of q / o belongs to table row i.
 *
 * GQA. Query head h reads kv head h / (n_q_heads / n_kv_heads).
 *
 * Ownership. The caller allocates and owns every device and host buffer
 * (pools, q, o, tables, workspace, staging). The library owns only the
 * host-side state behind hswa_pool (free lists and host mirrors of the
 * tables) and never keeps a caller pointer beyond the call, except that
 * hswa_sync_tables remembers which device tables it last wrote to.
 *
 * Ordering. Device calls enqueue work on the given stream and return
 * without waiting. Host calls (reserve, release, ...) act on host state
 * at once. Pool memory must hold finite values beyond a sequence's last
 * token (allocate it zeroed): masked keys get probability exactly 0, but
 * 0 * NaN would still be NaN.
 *
 * Errors. Every call checks its arguments before launching anything and
 * returns one of the HSWA_* status codes below; no exception crosses the
 * ABI. Device-side index checks and bounded waits do not trap: they set a
 * device error word that hswa_check reads back.
 *
 * Device lifetime. The library looks up, once per device, the addresses of
 * its own device variables (the error word, the no-allocation decode
 * scratch) and sets its kernels' shared-memory attributes. Do not use it on
 * a device after cudaDeviceReset of that device in the same process: the
 * cached addresses and attributes belong to the context that was reset.
 */
#ifndef HSWA_H
#define HSWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status */
#define HSWA_OK 0
#define HSWA_ERR_INVALID_ARG 1 /* bad pointer, size, id or ordering          */
#define HSWA_ERR_NO_SPACE 2    /* Full or SWA pool short of pages; no change  */
#define HSWA_ERR_UNSUPPORTED 3 /* dtype / head_dim / head ratio not built     */
#define HSWA_ERR_CUDA 4        /* a CUDA runtime call or launch failed        */
#define HSWA_ERR_TIMEOUT 5     /* a bounded device wait gave up               */
#define HSWA_ERR_BOUNDS 6      /* a device index check failed (access skipped)*/

#define HSWA_KIND_FULL 0
#define HSWA_KIND_SWA 1

#define HSWA_DTYPE_F32 0
#define HSWA_DTYPE_BF16 1
/* FP8 KV cache ("Baidu AI Cloud: Day-0 support for hybrid-architecture
 * LLMs", Optimization 2, KV Cache FP8 Tiled Quantization): K and V are E4M3
 * codes with one fp32 scale per (token, kv head, 128-element tile), value =
 * code * scale. Layout per layer: k_pool [pages][Hkv][P][d] bytes, v_pool
 * [pages][Hkv][d][P] bytes (each page stored transposed), k_scale and
 * v_scale [pages][Hkv][P][d / 128] fp32. q, o and the new K/V handed to the
 * append stay bf16; the append quantizes: scale = amax / 448 (1 if amax is
 * 0), code = round-to-nearest-even(x / scale) saturating at 448. Supported
 * by hswa_append_kv, hswa_decode, hswa_decode_append, hswa_decode_multi
 * (d = 128, 8 query heads per kv head, P = 64), hswa_prefill_chunk_ws (d = 128, an even
 * number of query heads per kv head, P = 64) and hswa_swa_gather /
 * hswa_swa_scatter (d = 128, P = 64); other calls return
 * HSWA_ERR_UNSUPPORTED. */
#define HSWA_DTYPE_FP8_E4M3 2

/* A CUDA stream (the same handle as cudaStream_t); NULL = default stream. */
typedef struct CUstream_st *hswa_stream_t;

typedef struct hswa_pool hswa_pool; /* opaque host-side bookkeeping */

typedef struct hswa_config {
    int32_t window;            /* W: tokens kept by release (> 0)               */
    int32_t page_size;         /* P: token slots per page (> 0)                 */
    int32_t n_q_heads;         /* Hq                                            */
    int32_t n_kv_heads;        /* Hkv, divides Hq                               */
    int32_t head_dim;          /* d                                             */
    int32_t dtype;             /* HSWA_DTYPE_* of the pools                     */
    int32_t full_pages;        /* pages in the Full pool                        */
    int32_t swa_pages;         /* pages in the SWA pool                         */
    int32_t max_seqs;          /* rows of each block table                      */
    int32_t max_pages_per_seq; /* columns of each block table                   */
} hswa_config;

typedef struct hswa_layer {
    int32_t kind;   /* HSWA_KIND_FULL or HSWA_KIND_SWA                          */
    int32_t window; /* keys per query for an SWA layer (> 0); ignored for Full  */
    void *k_pool;   /* device [num_pages][Hkv][P][d], caller-owned             */
    void *v_pool;   /* device, same shape ([num_pages][Hkv][d][P] for FP8)     */
    float *k_scale; /* FP8 only: device [num_pages][Hkv][P][d/128], else NULL  */
    float *v_scale; /* FP8 only: same shape                                    */
} hswa_layer;

/* ------------------------------------------------ pool bookkeeping (host) */

/* Create the bookkeeping of a dual pool (Sec. 2.1, KVCache Dual Pool).
 * full_free_order / swa_free_order: the initial FIFO free lists, a
 * permutation of 0..full_pages-1 (resp. swa_pages-1); NULL means ascending.
 * Every table entry starts at -1 and every length at 0. *out receives the
 * pool; free it with hswa_pool_destroy. */
int hswa_pool_create(const hswa_config *cfg, const int32_t *full_free_order,
                     const int32_t *swa_free_order, hswa_pool **out);
int hswa_pool_destroy(hswa_pool *pool);

/* Reserve slots for new tokens (Sec. 2.1: the access request checks the Full
 * and the SWA capacity together). seq_ids[0..n) strictly ascending; n_new[i]
 * tokens (>= 0) are added at positions L_i .. L_i + n_new[i] - 1. Every
 * logical page those tokens touch that has no Full page takes one from the
 * head of the Full free list, and likewise for SWA, in ascending (sequence,
 * logical page) order. full_slot_out / swa_slot_out (host, sum(n_new)
 * entries, may be NULL) receive the slots of the new tokens, sequences
 * concatenated in argument order. If either pool is short, returns
 * HSWA_ERR_NO_SPACE and changes nothing. Lengths grow by n_new. */
int hswa_reserve(hswa_pool *pool, int n, const int32_t *seq_ids, const int32_t *n_new,
                 int32_t *full_slot_out, int32_t *swa_slot_out);

/* Release out-of-window SWA pages (Sec. 2.1, SWA-aware prefix cache tree:
 * release after each prefill chunk, at request end and every N decode
 * tokens; keep at least the last W tokens). For each listed sequence of
 * length L, every SWA page on logical page p with (p + 1) * P <= L - W is
 * let go and its entry becomes -1; a page no one else holds (see Page
 * holders below) goes to the tail of the SWA free list, in ascending
 * (sequence, page) order. seq_ids need not be sorted (they are processed in
 * ascending order). *n_freed_out (may be NULL) gets the number of pages
 * that went back to the free list. */
int hswa_swa_release(hswa_pool *pool, int n, const int32_t *seq_ids, int32_t *n_freed_out);

/* Request end: let go of all Full and SWA pages of the sequences
 * (ascending sequence, then page; pages no one else holds return to the
 * free lists) and set their lengths to 0. */
int hswa_seq_free(hswa_pool *pool, int n, const int32_t *seq_ids);

/* Evict the SWA segment of each sequence alone, keeping its Full pages
 * (Sec. 2.1: the out-of-window SWA segment can be evicted while the Full
 * segment stays). Used after hswa_swa_gather has copied the window out.
 * *n_freed_out counts the pages that went back to the free list. */
int hswa_swa_drop(hswa_pool *pool, int n, const int32_t *seq_ids, int32_t *n_freed_out);

/* Give SWA pages to every in-window logical page (positions
 * [L - min(L, W), L)) of each sequence that has none, from the head of the
 * SWA free list in ascending (sequence, page) order; all or nothing
 * (HSWA_ERR_NO_SPACE). Used before hswa_swa_scatter reloads a window. */
int hswa_swa_restore(hswa_pool *pool, int n, const int32_t *seq_ids, int32_t *n_alloc_out);

/* Host mirrors, for inspection: copies the Full table, the SWA table
 * (int32 [max_seqs][max_pages_per_seq] each) and lengths (int32
 * [max_seqs]); any pointer may be NULL. */
int hswa_get_tables(const hswa_pool *pool, int32_t *full_bt, int32_t *swa_bt, int32_t *seq_len);

/* Free lists in FIFO order: kind HSWA_KIND_FULL or HSWA_KIND_SWA. *count
 * gets the length; out (may be NULL) receives up to cap entries. */
int hswa_get_free_list(const hswa_pool *pool, int kind, int32_t *out, int32_t cap, int32_t *count);

/* ------------------------------------ SWA-aware prefix cache tree (host)
 *
 * Page holders. A page can be held by several owners at once: the table
 * rows of sequences that share a cached prefix, and the prefix tree. The
 * pool counts the holders of each page; a page returns to the tail of its
 * free list only when the last one lets go. Without sharing every count is
 * 1 and the calls above behave as described there.
 *
 * The tree (Sec. 2.1, SWA-aware prefix cache tree) stores whole pages of
 * finished sequences, one node per page of P tokens holding its Full page
 * and its SWA page (-1: none), and keeps one hold on each. Three rules
 * differ from a plain prefix cache:
 *   1. window-safety length: a match of m pages needs, besides equal
 *      tokens, an SWA page on every logical page that meets the last W
 *      positions [m*P - W, m*P); the match is trimmed to the largest such
 *      m, the rest is a miss;
 *   2. release follows the request lifecycle (hswa_swa_release above);
 *   3. two indexes per node, evicted apart: SWA pages alone (the Full
 *      prefix stays reusable) or whole nodes.
 * Recency is a logical clock advanced by every match and insert. All
 * choices are deterministic (clock, then node creation order). */
typedef struct hswa_tree hswa_tree; /* opaque, host-owned */

/* Start holding the first n_pages cached pages for empty sequence seq_id
 * (length 0, no pages): its table row gets every Full page and the SWA
 * pages of the logical pages that meet the last W positions
 * [n_pages*P - W, n_pages*P); each of those must be held already (by a
 * tree or another sequence), else HSWA_ERR_INVALID_ARG and no change. The
 * length becomes n_pages * P; new tokens start on a fresh page. */
int hswa_seq_share_prefix(hswa_pool *pool, int32_t seq_id, int32_t n_pages, const int32_t *full_pages,
                          const int32_t *swa_pages);

/* Holder counts of the pool's pages (kind HSWA_KIND_FULL / HSWA_KIND_SWA),
 * up to cap entries. */
int hswa_get_page_refs(const hswa_pool *pool, int kind, int32_t *out, int32_t cap);

/* A tree over one pool. Destroy every tree of a pool before the pool
 * (hswa_pool_destroy returns HSWA_ERR_INVALID_ARG while one exists). */
int hswa_tree_create(hswa_pool *pool, hswa_tree **out);
/* Let go of every stored page (nodes in creation order, each Full page
 * before its SWA page) and free the tree. */
int hswa_tree_destroy(hswa_tree *tree);

/* Window-safe hit for n_tokens tokens (whole pages only). *n_pages_out
 * gets m, the usable pages; full_pages_out / swa_pages_out (host, cap_pages
 * >= min(n_tokens / P, max_pages_per_seq) entries) the pages of logical
 * pages [0, m); *raw_pages_out (may be NULL) the pages whose tokens matched
 * before trimming. Stamps the nodes of the untrimmed match as used. Pass
 * the pages to hswa_seq_share_prefix to reuse them. */
int hswa_tree_match(hswa_tree *tree, const int32_t *tokens, int64_t n_tokens, int32_t *full_pages_out,
                    int32_t *swa_pages_out, int32_t cap_pages, int32_t *n_pages_out, int32_t *raw_pages_out);

/* Store the whole pages of the first n_tokens tokens of sequence seq_id
 * (n_tokens <= its length; each of those pages must have a Full page):
 * pages new to the tree become nodes holding the sequence's Full and SWA
 * pages; where a node exists for the same tokens the tree keeps its own
 * pages (the sequence's copy is freed with the sequence) and takes the
 * sequence's SWA page if the node has none. Stamps the whole path as used.
 * *n_new_out (may be NULL) gets the number of new nodes. Call before
 * hswa_seq_free at request end. */
int hswa_tree_insert(hswa_tree *tree, int32_t seq_id, const int32_t *tokens, int64_t n_tokens,
                     int32_t *n_new_out);

/* Make room: free at least want_swa SWA pages and want_full Full pages
 * that only the tree holds, if it can. SWA pages first: those outside the
 * window of every stored end below their node (a node on logical page i is
 * inside it when i >= (D*P - W) / P for the shallowest leaf below or at it,
 * D pages deep), oldest first, then the rest. Then whole leaf nodes whose
 * Full page only the tree holds, oldest first, until want_full pages are
 * free (their SWA pages go too). *freed_full_out / *freed_swa_out (may be
 * NULL) get the pages that went back to the free lists. */
int hswa_tree_evict(hswa_tree *tree, int32_t want_full, int32_t want_swa, int32_t *freed_full_out,
                    int32_t *freed_swa_out);

/* Nodes and pages held: *n_nodes = *full_held = nodes, *swa_held = nodes
 * with an SWA page (any may be NULL). */
int hswa_tree_stats(const hswa_tree *tree, int32_t *n_nodes, int32_t *full_held, int32_t *swa_held);

/* The nodes in creation order, 5 int32 each: id, parent id (-1 = root),
 * logical page, Full page, SWA page; up to cap / 5 nodes written, *count
 * gets the node count. */
int hswa_tree_nodes(const hswa_tree *tree, int32_t *out, int32_t cap, int32_t *count);

/* ------------------------------------------------- device-side calls */

/* Bring the device tables (int32 [max_seqs][max_pages_per_seq] each, and
 * lengths int32 [max_seqs]) up to date with the host state, enqueued on
 * stream: the changed entries are packed into a pinned staging buffer owned
 * by the pool and one small kernel reads them from there (device-mapped host
 * memory) and writes them. The staging buffer is reused only after that
 * kernel has finished. The first call, or a call with other device pointers
 * than the last one, uploads the whole tables and waits for the copy. */
int hswa_sync_tables(hswa_pool *pool, int32_t *d_full_bt, int32_t *d_swa_bt, int32_t *d_seq_len,
                     hswa_stream_t stream);

/* KV append (Sec. 2.1, dual pool: Full layers write only the Full pool and
 * SWA layers only the SWA pool). For each token t < n_tokens with
 * d_slots[t] >= 0: pool[slot / P][g][slot % P][:] = new[t][g][:] for K and V.
 * k, v: device [n_tokens][Hkv][d] in the pool dtype. d_slots: device int32,
 * the full_slot (Full layer) or swa_slot (SWA layer) array from
 * hswa_reserve. A slot past the pool sets HSWA_ERR_BOUNDS on the device
 * and is skipped. */
int hswa_append_kv(const hswa_pool *pool, const hswa_layer *layer, const void *k, const void *v,
                   const int32_t *d_slots, int n_tokens, hswa_stream_t stream);

/* Bytes of workspace hswa_decode needs for a batch of n_seqs sequences. */
size_t hswa_decode_workspace_size(const hswa_pool *pool, int n_seqs);

/* One decode step of attention (Sec. 1.2: decode is memory-bound; Sec. 5.1:
 * decode reads the SWA pool). For sequence i < n_seqs with L = d_seq_len[i]
 * keys (the new token already appended), query q[i][h] at position L - 1
 * attends keys [0, L) for a Full layer and [max(0, L - W), L) for an SWA
 * layer, W = layer->window:
 *     o[i][h] = softmax_j(scale * <q[i][h], k_j>) v_j.
 * q, o: device [n_seqs][Hq][d] in the pool dtype. d_bt: device table of the
 * layer's kind. L = 0 gives o = 0. ws: device workspace of at least
 * hswa_decode_workspace_size bytes (split-K partial results), caller-owned,
 * not read before it is written. A table entry outside the pool sets
 * HSWA_ERR_BOUNDS on the device; that page is skipped. */
int hswa_decode(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                const int32_t *d_bt, const int32_t *d_seq_len, int n_seqs, float scale,
                void *ws, size_t ws_bytes, hswa_stream_t stream);

/* hswa_append_kv followed by hswa_decode in one call, for a decode step of
 * one new token per sequence: k_new, v_new are device [n_seqs][Hkv][d] (row i
 * = sequence i's new token) and d_slots[i] its slot in the layer kind's pool
 * (from hswa_reserve); d_seq_len already counts the new token. On the fast
 * path the CTA that streams the page holding a sequence's last token first
 * writes that token's K and V rows there, so the append costs no launch of
 * its own. Same result as the two calls in a row. */
int hswa_decode_append(const hswa_pool *pool, const hswa_layer *layer, const void *q, const void *k_new,
                       const void *v_new, const int32_t *d_slots, void *o, const int32_t *d_bt,
                       const int32_t *d_seq_len, int n_seqs, float scale, void *ws, size_t ws_bytes,
                       hswa_stream_t stream);

/* Most query tokens per sequence hswa_decode_multi takes. */
#define HSWA_DECODE_MAX_TOKENS 16

/* Bytes of workspace hswa_decode_multi needs for n_seqs sequences of n_tok
 * query tokens each (0 for an n_tok outside [1, HSWA_DECODE_MAX_TOKENS]). */
size_t hswa_decode_multi_workspace_size(const hswa_pool *pool, int n_seqs, int n_tok);

/* Decode of n_tok query tokens per sequence in one pass over the KV pages:
 * the verification step of multi-token prediction or speculative decoding
 * ("MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 5.2 MTP
 * Optimization: 3-layer MTP decode; "Following the Bottleneck: Optimizing
 * MiniMax M3 on AMD Instinct MI355X", EAGLE3 adds a second decode loop:
 * multi-token verification, each flattened query row mapped back to its
 * request and its speculative position). For sequence i < n_seqs with
 * L = d_seq_len[i] keys (all n_tok new tokens already appended), query token
 * w < n_tok sits at position t = L - n_tok + w and attends keys [0, t] for a
 * Full layer and [max(0, t - W + 1), t] for an SWA layer (causal among the
 * new tokens). q, o: device [n_seqs][n_tok][Hq][d] in the pool dtype (row
 * i * n_tok + w). A token with t < 0 gets o = 0. n_tok = 1 is hswa_decode.
 * ws: device workspace of at least hswa_decode_multi_workspace_size bytes.
 * The SWA pages must still hold positions from L - n_tok + 1 - W on: release
 * out-of-window pages before the draft tokens are reserved. Bf16 and FP8
 * pools; every page is streamed once for all n_tok tokens. n_tok outside
 * [1, HSWA_DECODE_MAX_TOKENS] gives HSWA_ERR_INVALID_ARG; n_seqs * n_tok
 * above 65535 (query rows the merge of split pages takes in one launch)
 * gives HSWA_ERR_UNSUPPORTED. */
int hswa_decode_multi(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                      const int32_t *d_bt, const int32_t *d_seq_len, int n_seqs, int n_tok, float scale,
                      void *ws, size_t ws_bytes, hswa_stream_t stream);

/* One chunked-prefill chunk of attention (Sec. 1.1: chunked prefill is
 * close to compute-bound). Sequence i < n_seqs has d_prefix_len[i] cached
 * tokens and n_i = d_q_start[i+1] - d_q_start[i] new tokens whose K/V are
 * already appended; query row r (0 <= r < n_i) sits at position
 * t = prefix + r and attends keys [0, t] (Full) or [max(0, t - W + 1), t]
 * (SWA). q, o: device [total_q][Hq][d] with total_q = d_q_start[n_seqs];
 * d_q_start: device int32 [n_seqs + 1], non-decreasing from 0; max_q_len >=
 * every n_i (sizes the grid). The host passes total_q and max_q_len because
 * it cannot read d_q_start without waiting for the device; rows are never
 * read past total_q. scale must be > 0 (HSWA_ERR_INVALID_ARG otherwise). */
int hswa_prefill_chunk(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                       const int32_t *d_bt, const int32_t *d_prefix_len, const int32_t *d_q_start,
                       int n_seqs, int total_q, int max_q_len, float scale, hswa_stream_t stream);

/* Bytes of workspace hswa_prefill_chunk_ws needs for any chunk of n_seqs
 * sequences with at most max_q_len new tokens each: 0 for bf16 and fp32
 * pools (they need none); for an FP8 pool, room for an fp16 copy of every
 * page such a chunk can read (all of a sequence's table row for a Full
 * layer, ceil((W - 1 + max_q_len) / P) + 1 pages for an SWA layer), a block
 * table onto the copies, a per-sequence offset table and an fp16 copy of
 * n_seqs * max_q_len query rows. An upper bound, for callers that do not
 * know the lengths on the host; hswa_prefill_workspace_size_exact is the
 * smaller figure for a known chunk. */
size_t hswa_prefill_workspace_size(const hswa_pool *pool, const hswa_layer *layer, int n_seqs,
                                   int max_q_len);

/* Bytes of workspace a given chunk needs on an FP8 pool: the same layout as
 * above holding exactly the pages the chunk reads (logical pages 0 ..
 * (prefix + n - 1) / P of each sequence for a Full layer, from
 * (prefix - W + 1) / P for an SWA layer) and its q_start[n_seqs] query
 * rows. prefix_len (host int32 [n_seqs]) and q_start (host int32
 * [n_seqs + 1]) hold the values the device arrays of the call will hold.
 * 0 for bf16 and fp32 pools. On the chunked-prefill workload (8 sequences,
 * prefixes of 8K-64K tokens, 4096 new tokens each, 64 / 8 heads, table rows
 * of 972 pages) the Full layer needs 4,897 page copies: 1.82 GB with the
 * 0.54 GB q copy, against 2.58 GB for the upper bound. */
size_t hswa_prefill_workspace_size_exact(const hswa_pool *pool, const hswa_layer *layer, int n_seqs,
                                         const int32_t *prefix_len, const int32_t *q_start);

/* hswa_prefill_chunk with a workspace, which FP8 pools need ("Baidu AI
 * Cloud: Day-0 support for hybrid-architecture LLMs", Optimization 2 item 2:
 * an FP8 KV cache with one scale per token, head and 128-element tile).
 * Same arguments and result as hswa_prefill_chunk. Over an FP8 pool the
 * pages the chunk reads are first dequantized (E4M3 code x scale, rounded
 * once to fp16, saturating at 65504) and q is converted to fp16 (exact for
 * magnitudes in [2^-14, 65504]) into ws; the tensor-core kernel then
 * attends with fp16 operands. q and o are bf16. ws: device, 256-byte
 * aligned, caller-owned, not read before it is written; it must not be
 * reused until the call's work on stream has finished. The page copies are
 * packed sequence after sequence into whatever ws holds past its tables and
 * q copy: hswa_prefill_workspace_size_exact bytes hold every page of the
 * chunk, hswa_prefill_workspace_size bytes every page of any chunk of those
 * sizes. A ws too small for the tables, the q copy and one page copy is
 * HSWA_ERR_INVALID_ARG; pages past what ws holds are not staged, read as
 * zeros and set HSWA_ERR_BOUNDS (hswa_check). Ignored (may be NULL) for
 * bf16 and fp32 pools. hswa_prefill_chunk on an FP8 pool returns
 * HSWA_ERR_INVALID_ARG (no workspace). */
int hswa_prefill_chunk_ws(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                          const int32_t *d_bt, const int32_t *d_prefix_len, const int32_t *d_q_start,
                          int n_seqs, int total_q, int max_q_len, float scale, void *ws, size_t ws_bytes,
                          hswa_stream_t stream);

/* Transfer by SWA mask (Sec. 2.1, Data Transfer: only in-window data moves;
 * "Tiered KV Cache Offloading in vLLM", hybrid models: sliding-window
 * layers reload only the tokens in their window). For sequence i < n_seqs
 * with L_i = d_seq_len[i], n_i = min(L_i, W) tokens at positions
 * [L_i - n_i, L_i) of one SWA layer are packed into dst as a K block
 * [Hkv][n_i][d] then a V block [Hkv][n_i][d], starting at element
 * 2 * Hkv * d * d_tok_offset[i]; d_tok_offset: device int64 [n_seqs + 1],
 * the prefix sum of n_i. W = layer->window. dst may be device memory or
 * pinned host memory mapped into the device address space. An in-window
 * token without an SWA page sets HSWA_ERR_BOUNDS and is skipped. The
 * caller must not reuse dst until work enqueued after this call on stream
 * has finished. FP8 pools (d = 128, P = 64; dst 8-byte aligned): sequence
 * i starts at byte 2 * Hkv * (d + 4) * d_tok_offset[i] and holds K codes
 * [Hkv][n_i][d], V codes [Hkv][n_i][d] (token rows, not the pages'
 * transposed layout), K scales [Hkv][n_i] and V scales [Hkv][n_i] (fp32). */
int hswa_swa_gather(const hswa_pool *pool, const hswa_layer *layer, const int32_t *d_swa_bt,
                    const int32_t *d_seq_len, const int64_t *d_tok_offset, int n_seqs, void *dst,
                    hswa_stream_t stream);

/* Where each sequence's window starts in the packed buffer of
 * hswa_swa_gather / hswa_swa_scatter (Sec. 2.1, Data Transfer: only the
 * in-window tokens move, so sequence i takes n_i = min(L_i, W) token slots,
 * W = layer->window). Host call, no device work: tok_offset_out (host int64
 * [n_seqs + 1]) receives 0, n_0, n_0 + n_1, ..., the d_tok_offset the
 * transfer calls take once the caller has copied it to the device.
 * seq_len: host int32 [n_seqs], the lengths the transfer will read from
 * d_seq_len; NULL takes the pool's own current lengths of sequences
 * 0..n_seqs-1. packed_bytes_out (may be NULL) receives the size of the
 * packed buffer in bytes: 2 * Hkv * d * element size per token, or
 * 2 * Hkv * (d + 4) on FP8 pools. HSWA_ERR_INVALID_ARG for a non-SWA layer,
 * a negative length or n_seqs outside [0, max_seqs]. */
int hswa_swa_window_offsets(const hswa_pool *pool, const hswa_layer *layer, int n_seqs,
                            const int32_t *seq_len, int64_t *tok_offset_out, size_t *packed_bytes_out);

/* Inverse of hswa_swa_gather: write a packed buffer back into the layer's
 * SWA pool pages named by d_swa_bt (after hswa_swa_restore). */
int hswa_swa_scatter(const hswa_pool *pool, const hswa_layer *layer, const int32_t *d_swa_bt,
                     const int32_t *d_seq_len, const int64_t *d_tok_offset, int n_seqs,
                     const void *src, hswa_stream_t stream);

/* Decode without any device allocation by the caller or the library.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot hand over a workspace: a host program that is only given the
 * pool, q and o pointers by another component that owns all device memory
 * (for instance an engine that has reserved the whole HBM for KV pages), or
 * a latency-critical loop that must not pay for an allocation. It computes
 * exactly what hswa_decode computes, with the same arguments minus the
 * workspace: the split-K scratch lives in a fixed array of
 * HSWA_DECODE_NOALLOC_SCRATCH_BYTES in the library's device image, which
 * every GPU that loads the library keeps until the process exits.
 *
 * Limits: n_seqs <= HSWA_DECODE_NOALLOC_MAX_SEQS, and the scratch the
 * launch needs must fit the array:
 *   round_up(16 * (n_seqs + 1), 256) + 2 * 4160 * n_ctas
 *       <= HSWA_DECODE_NOALLOC_SCRATCH_BYTES,
 * with n_ctas = SM count * resident decode CTAs per SM (at most 4). On a
 * 152-SM GB300 that is 304 CTAs over bf16 pools and 456 over FP8 pools
 * (2 and 3 per SM), 2.8 and 4.06 MB at the largest batch, so every batch
 * fits there; a part with more SMs or more resident CTAs per SM can reject
 * large batches. A batch that does not fit returns HSWA_ERR_INVALID_ARG and
 * launches nothing. The first call on a device looks up the scratch address
 * with that device current; make that first call before any stream capture.
 * All calls on a device share the one scratch array: two calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race
 * on it. Nothing in the scratch has to start at zero; it keeps whatever the
 * last call left there. Calls no cudaMalloc, cudaFree or other allocating
 * routine. */
#define HSWA_DECODE_NOALLOC_SCRATCH_BYTES (4u << 20)
#define HSWA_DECODE_NOALLOC_MAX_SEQS 16384
int hswa_decode_noalloc(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                        const int32_t *d_bt, const int32_t *d_seq_len, int n_seqs, float scale,
                        hswa_stream_t stream);

/* Wait for stream, then read and clear the device error word of the
 * current device: HSWA_OK, HSWA_ERR_BOUNDS or HSWA_ERR_TIMEOUT (or
 * HSWA_ERR_CUDA if the wait itself failed). */
int hswa_check(hswa_stream_t stream);

/* Diagnostic (no counterpart on the pages): launch one block that waits on
 * an mbarrier nothing completes, through the bounded wait every kernel of
 * the library uses. After about a second of GPU time the wait gives up and
 * the device error word reads HSWA_ERR_TIMEOUT (see hswa_check); the context
 * stays usable. Returns the launch status. */
int hswa_selftest_bounded_wait(hswa_stream_t stream);

/* Name of the kernel variant the last device call on this host thread
 * launched (e.g. "decode_mma_bf16_d128"); "" before any launch. */
const char *hswa_last_kernel(void);

/* The CUDA error behind the last HSWA_ERR_CUDA a launch path on this host
 * thread returned ("where: message"), "" if none has been recorded. */
const char *hswa_last_cuda_error(void);

/* Human-readable name of a status code. */
const char *hswa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* HSWA_H */
