// Launchers shared between the CUDA translation units of libhswa.
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace hswa {

// CUDA-core attention for any dtype / head_dim (<= 256) / head ratio / page
// size. mode 0: decode, n_rows = sequences x n_tok (row i is query token
// i mod n_tok of sequence i / n_tok, at position L - n_tok + i mod n_tok);
// mode 1: prefill, n_rows = max rows per sequence (row r of sequence s is q
// row q_start[s] + r at position prefix[s] + r).
int launch_attention_generic(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                             const int32_t *bt, const int32_t *seq_len, const int32_t *prefix,
                             const int32_t *q_start, int32_t n_rows, int32_t n_seqs, float scale, int mode,
                             cudaStream_t st, int32_t n_tok = 1);

}  // namespace hswa
