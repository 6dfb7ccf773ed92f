/*
 * CPU oracle for paged Full / sliding-window GQA attention (float64).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain definition that the
 * CUDA library is checked against. Only tests/, __graft_entry__.smoke() and
 * bench.py's cpu_baseline / reference leg may load it. It shares no code,
 * header or constant with the CUDA library.
 *
 * What it computes ("MiMo-V2.5 Series Inference Full-Link Optimization",
 * Sec. 1.1 Computational Complexity Analysis and Sec. 2.1 KVCache Dual Pool):
 *
 *   For a query of sequence s at token position t and query head h, with
 *   kv head g = floor(h * Hkv / Hq) and key set
 *       J = {0, ..., t}                       Full-Attention layer
 *       J = {max(0, t - W + 1), ..., t}       SWA layer (W attended keys,
 *                                             the query's own token included)
 *   the output is
 *       o = sum_{j in J} softmax_j(scale * <q, k_j>) * v_j
 *   where k_j and v_j are read through the block table: physical page
 *   bt[s][j / P], row j mod P, inside a pool laid out [page][Hkv][P][d].
 *
 * The softmax is the two-pass, max-subtracted form, done in double from the
 * exact values of the fp32 or bf16 inputs.  The loops below follow the
 * definition one query at a time; the only parallelism is OpenMP over
 * (query, head), which does not change any result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes of the inputs: 0 = IEEE fp32, 1 = bf16 (upper half of fp32) */
static double elem(const void *base, int64_t idx, int dtype)
{
    if (dtype == 0)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Attention for n_queries query tokens.
 *   q        [n_queries][Hq][d]  (dtype)
 *   k_pool   [num_pages][Hkv][P][d] (dtype), v_pool likewise
 *   q_seq[i] block-table row of query i; q_pos[i] its position t
 *   window   W for an SWA layer, 0 for a Full layer
 *   o        [n_queries][Hq][d]  float64 (written)
 * Returns 0, or -1 when a block-table entry needed by a query is outside
 * [0, num_pages) (a released or never-reserved page), or -2 on bad sizes.
 */
int hswa_oracle_attention(int64_t n_queries, const int32_t *q_seq,
                          const int64_t *q_pos, int n_q_heads, int n_kv_heads,
                          int head_dim, int page_size, int window,
                          double scale, int dtype, const void *q,
                          const void *k_pool, const void *v_pool,
                          int64_t num_pages, const int32_t *block_table,
                          int64_t bt_stride, double *o)
{
    if (n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
        n_q_heads % n_kv_heads != 0 || window < 0)
        return -2;
    int bad = 0;
    const int64_t total = n_queries * n_q_heads;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t qi = 0; qi < total; ++qi) {
        const int64_t i = qi / n_q_heads;
        const int h = (int)(qi % n_q_heads);
        const int g = (int)(((int64_t)h * n_kv_heads) / n_q_heads);
        const int64_t t = q_pos[i];
        const int32_t *bt = block_table + (int64_t)q_seq[i] * bt_stride;
        const int64_t lo = (window > 0 && t - window + 1 > 0) ? t - window + 1 : 0;
        const int64_t n_keys = t - lo + 1;
        double *out = o + qi * head_dim;

        double *score = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
        int64_t *row = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_keys > 0 ? n_keys : 1));
        int my_bad = 0;

        /* pass 1: scaled scores and their maximum */
        double m = -INFINITY;
        for (int64_t j = lo; j <= t; ++j) {
            const int32_t page = bt[j / page_size];
            if (page < 0 || page >= num_pages) {
                my_bad = 1;
                break;
            }
            /* element offset of row (page, g, j mod P, 0) in the pool */
            const int64_t r = (((int64_t)page * n_kv_heads + g) * page_size +
                               j % page_size) * head_dim;
            double dot = 0.0;
            for (int c = 0; c < head_dim; ++c)
                dot += elem(q, qi * head_dim + c, dtype) * elem(k_pool, r + c, dtype);
            score[j - lo] = scale * dot;
            row[j - lo] = r;
            if (score[j - lo] > m)
                m = score[j - lo];
        }

        for (int c = 0; c < head_dim; ++c)
            out[c] = 0.0;
        if (my_bad) {
#pragma omp atomic write
            bad = 1;
        } else if (n_keys > 0) {
            /* pass 2: weights exp(s - m), their sum, and the weighted values */
            double z = 0.0;
            for (int64_t j = 0; j < n_keys; ++j) {
                const double w = exp(score[j] - m);
                z += w;
                for (int c = 0; c < head_dim; ++c)
                    out[c] += w * elem(v_pool, row[j] + c, dtype);
            }
            for (int c = 0; c < head_dim; ++c)
                out[c] /= z;
        }
        free(score);
        free(row);
    }
    return bad ? -1 : 0;
}

/* Value of an E4M3 code (OCP 8-bit float: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, subnormals, S.1111.111 = NaN). */
static double e4m3_value(uint8_t c)
{
    const int e = (c >> 3) & 0xF, m = c & 0x7;
    if ((c & 0x7F) == 0x7F)
        return NAN;
    const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (c & 0x80) ? -mag : mag;
}

/*
 * The same attention over an FP8 KV cache ("Baidu AI Cloud: Day-0 support
 * for hybrid-architecture LLMs", Optimization 2 item 2: FP8 per token, per
 * head, per 128-element tile). Keys and values are the exact dequantized
 * values code * scale:
 *   k_codes [num_pages][Hkv][P][d]   E4M3, k_scale [num_pages][Hkv][P][d/128]
 *   v_codes [num_pages][Hkv][d][P]   E4M3 (each page stored transposed),
 *   v_scale [num_pages][Hkv][P][d/128]
 * q is fp32 (dtype 0) or bf16 (dtype 1). Returns as hswa_oracle_attention.
 */
int hswa_oracle_attention_fp8(int64_t n_queries, const int32_t *q_seq, const int64_t *q_pos,
                              int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                              int window, double scale, int q_dtype, const void *q,
                              const uint8_t *k_codes, const float *k_scale,
                              const uint8_t *v_codes, const float *v_scale, int64_t num_pages,
                              const int32_t *block_table, int64_t bt_stride, double *o)
{
    if (n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim % 128 != 0 ||
        page_size <= 0 || n_q_heads % n_kv_heads != 0 || window < 0)
        return -2;
    const int tiles = head_dim / 128;
    int bad = 0;
    const int64_t total = n_queries * n_q_heads;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t qi = 0; qi < total; ++qi) {
        const int64_t i = qi / n_q_heads;
        const int h = (int)(qi % n_q_heads);
        const int g = (int)(((int64_t)h * n_kv_heads) / n_q_heads);
        const int64_t t = q_pos[i];
        const int32_t *bt = block_table + (int64_t)q_seq[i] * bt_stride;
        const int64_t lo = (window > 0 && t - window + 1 > 0) ? t - window + 1 : 0;
        const int64_t n_keys = t - lo + 1;
        double *out = o + qi * head_dim;
        double *score = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
        int64_t *blk = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_keys > 0 ? n_keys : 1));
        int my_bad = 0;

        double m = -INFINITY;
        for (int64_t j = lo; j <= t; ++j) {
            const int32_t page = bt[j / page_size];
            if (page < 0 || page >= num_pages) {
                my_bad = 1;
                break;
            }
            const int64_t b = (int64_t)page * n_kv_heads + g;  /* (page, kv head) block */
            const int64_t row = j % page_size;
            double dot = 0.0;
            for (int c = 0; c < head_dim; ++c) {
                const double kv = e4m3_value(k_codes[(b * page_size + row) * head_dim + c]) *
                                  (double)k_scale[(b * page_size + row) * tiles + c / 128];
                dot += elem(q, qi * head_dim + c, q_dtype) * kv;
            }
            score[j - lo] = scale * dot;
            blk[j - lo] = b * page_size + row;  /* (block, row) index */
            if (score[j - lo] > m)
                m = score[j - lo];
        }
        for (int c = 0; c < head_dim; ++c)
            out[c] = 0.0;
        if (my_bad) {
#pragma omp atomic write
            bad = 1;
        } else if (n_keys > 0) {
            double z = 0.0;
            for (int64_t jj = 0; jj < n_keys; ++jj) {
                const double w = exp(score[jj] - m);
                const int64_t b = blk[jj] / page_size, row = blk[jj] % page_size;
                z += w;
                for (int c = 0; c < head_dim; ++c)
                    out[c] += w * e4m3_value(v_codes[(b * head_dim + c) * page_size + row]) *
                              (double)v_scale[(b * page_size + row) * tiles + c / 128];
            }
            for (int c = 0; c < head_dim; ++c)
                out[c] /= z;
        }
        free(score);
        free(blk);
    }
    return bad ? -1 : 0;
}

/* Number of OpenMP threads the attention loop runs on. */
int hswa_oracle_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
