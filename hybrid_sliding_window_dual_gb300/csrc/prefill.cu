// Chunked-prefill attention over the dual KV pool.
//
// "MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 1.1: in chunked
// prefill the attention is close to compute-bound; SWA layers attend only to
// the last W tokens, so their cost per query is O(W) instead of O(N).
#include "common.cuh"
#include "internal.h"
#include "kernels.h"

using namespace hswa;

extern "C" int hswa_prefill_chunk(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                                  const int32_t *d_bt, const int32_t *d_prefix_len, const int32_t *d_q_start,
                                  int n_seqs, int max_q_len, float scale, hswa_stream_t stream) {
    if (!pool || !layer || n_seqs < 0 || n_seqs > pool->cfg.max_seqs || max_q_len < 0 ||
        (layer->kind != HSWA_KIND_FULL && layer->kind != HSWA_KIND_SWA) ||
        (layer->kind == HSWA_KIND_SWA && layer->window <= 0))
        return HSWA_ERR_INVALID_ARG;
    if (n_seqs == 0 || max_q_len == 0) return HSWA_OK;
    if (!q || !o || !d_bt || !d_prefix_len || !d_q_start || !layer->k_pool || !layer->v_pool)
        return HSWA_ERR_INVALID_ARG;
    return launch_attention_generic(pool, layer, q, o, d_bt, nullptr, d_prefix_len, d_q_start, max_q_len, n_seqs,
                                    scale, 1, reinterpret_cast<cudaStream_t>(stream));
}
