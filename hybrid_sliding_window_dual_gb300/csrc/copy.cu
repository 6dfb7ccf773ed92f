// Copy kernels of the dual KV pool: slot-mapped KV append and the
// in-window SWA gather / scatter.
//
// "MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 2.1 (KVCache
// Dual Pool): Full layers keep every token in the Full pool, SWA layers keep
// the window in the SWA pool; cross-tier transfer moves only SWA-mask data.
// "Tiered KV Cache Offloading in vLLM", hybrid models: sliding-window layers
// reload only the tokens inside their window.
//
// All three kernels are HBM- (or host-link-) bound 16-byte copies: a warp
// moves whole 16-byte chunks of a token's K or V row, so a row of
// d * sizeof(dtype) bytes is read and written with full 32-byte sectors.
#include <algorithm>

#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace hswa {
namespace {

using chunk_t = uint4;  // 16 bytes

// k_new / v_new [T][Hkv][row] -> pool [page][Hkv][P][row], row = d * esize
__global__ void append_kv_kernel(const chunk_t *__restrict__ k, const chunk_t *__restrict__ v, chunk_t *kp,
                                 chunk_t *vp, const int32_t *__restrict__ slots, int64_t n_tokens, int32_t hkv,
                                 int32_t page, int32_t chunks_per_row, int64_t pool_slots, int *err) {
    const int64_t per_tok = (int64_t)hkv * chunks_per_row;
    const int64_t total = n_tokens * per_tok;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_tok;
        const int64_t r = i - t * per_tok;  // g * chunks_per_row + c
        const int32_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            set_error(err, HSWA_ERR_BOUNDS);
            continue;
        }
        const int64_t g = r / chunks_per_row, c = r - g * chunks_per_row;
        const int64_t dst = (((int64_t)(slot / page) * hkv + g) * page + slot % page) * chunks_per_row + c;
        kp[dst] = k[i];
        vp[dst] = v[i];
    }
}

// One CTA strip per sequence (blockIdx.y). Packed order per sequence:
// [K | V][Hkv][n_s tokens][row chunks].
template <bool kGather>
__global__ void swa_xfer_kernel(chunk_t *kp, chunk_t *vp, chunk_t *packed, const int32_t *__restrict__ swa_bt,
                                const int32_t *__restrict__ seq_len, const int64_t *__restrict__ tok_offset,
                                int32_t bt_stride, int32_t hkv, int32_t page, int32_t window,
                                int32_t chunks_per_row, int32_t num_pages, int *err) {
    const int32_t s = blockIdx.y;
    const int32_t L = seq_len[s];
    const int64_t n = (int64_t)(L < window ? L : window);
    if (n <= 0) return;
    const int64_t per_kind = (int64_t)hkv * n * chunks_per_row;
    chunk_t *seq_base = packed + tok_offset[s] * 2 * hkv * chunks_per_row;
    const int32_t *btrow = swa_bt + (int64_t)s * bt_stride;
    for (int64_t f = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; f < 2 * per_kind;
         f += (int64_t)gridDim.x * blockDim.x) {
        const int64_t which = f / per_kind;
        int64_t r = f - which * per_kind;
        const int64_t g = r / (n * chunks_per_row);
        r -= g * n * chunks_per_row;
        const int64_t i = r / chunks_per_row, c = r - i * chunks_per_row;
        const int64_t t = L - n + i;  // token position
        const int64_t lp = t / page;
        const int32_t pg = lp < bt_stride ? btrow[lp] : -1;
        if (pg < 0 || pg >= num_pages) {
            set_error(err, HSWA_ERR_BOUNDS);
            continue;
        }
        chunk_t *pool = which ? vp : kp;
        const int64_t at = (((int64_t)pg * hkv + g) * page + t % page) * chunks_per_row + c;
        if (kGather)
            seq_base[f] = pool[at];
        else
            pool[at] = seq_base[f];
    }
}

// FP8 transfer (d = 128, P = 64): one CTA per (kv head, sequence) walks the
// pages of the window. Packed order per sequence (at byte 2 * Hkv * 132 *
// tok_offset): K codes [Hkv][n][128], V codes [Hkv][n][128] (token rows),
// K scales [Hkv][n] and V scales [Hkv][n] (fp32). K rows and scales are
// contiguous runs on both sides; a V page is stored transposed ([128][64]),
// so its window columns go through a shared-memory tile.
template <bool kGather>
__global__ void __launch_bounds__(256) swa_xfer_fp8_kernel(uint8_t *kc, uint8_t *vc, float *ks, float *vs,
                                                           uint8_t *packed, const int32_t *__restrict__ swa_bt,
                                                           const int32_t *__restrict__ seq_len,
                                                           const int64_t *__restrict__ tok_offset, int32_t bt_stride,
                                                           int32_t hkv, int32_t window, int32_t num_pages, int *err) {
    constexpr int kDd = 128, kPg = 64;
    __shared__ __align__(16) uint8_t tile[kDd * kPg];
    const int32_t g = blockIdx.x, s = blockIdx.y;
    const int32_t L = seq_len[s];
    const int32_t n = L < window ? L : window;
    if (n <= 0) return;
    const int32_t t_lo = L - n;
    uint8_t *base = packed + tok_offset[s] * 2 * hkv * (kDd + 4);
    uint8_t *pk = base + (int64_t)g * n * kDd;
    uint8_t *pv = base + ((int64_t)hkv + g) * n * kDd;
    float *pks = reinterpret_cast<float *>(base + 2 * (int64_t)hkv * n * kDd) + (int64_t)g * n;
    float *pvs = pks + (int64_t)hkv * n;
    const int32_t *btrow = swa_bt + (int64_t)s * bt_stride;
    for (int32_t lp = t_lo / kPg; lp <= (L - 1) / kPg; ++lp) {
        const int32_t pg = lp < bt_stride ? btrow[lp] : -1;
        if (pg < 0 || pg >= num_pages) {
            if (threadIdx.x == 0) set_error(err, HSWA_ERR_BOUNDS);
            continue;
        }
        const int32_t r0 = max(t_lo, lp * kPg) - lp * kPg, r1 = min(L, (lp + 1) * kPg) - lp * kPg;
        const int32_t nr = r1 - r0, i0 = lp * kPg + r0 - t_lo;  // window tokens on the page, first one's index
        const int64_t blk = (int64_t)pg * hkv + g;                // (page, kv head) block
        // K rows and both scale runs: 8-byte words (every run starts on an 8-byte boundary)
        uint2 *kpool = reinterpret_cast<uint2 *>(kc + (blk * kPg + r0) * kDd);
        uint2 *kpack = reinterpret_cast<uint2 *>(pk + (int64_t)i0 * kDd);
        for (int32_t w = threadIdx.x; w < nr * kDd / 8; w += blockDim.x) {
            if (kGather)
                kpack[w] = kpool[w];
            else
                kpool[w] = kpack[w];
        }
        for (int32_t k = threadIdx.x; k < nr; k += blockDim.x) {
            if (kGather) {
                pks[i0 + k] = ks[blk * kPg + r0 + k];
                pvs[i0 + k] = vs[blk * kPg + r0 + k];
            } else {
                ks[blk * kPg + r0 + k] = pks[i0 + k];
                vs[blk * kPg + r0 + k] = pvs[i0 + k];
            }
        }
        uint8_t *vpage = vc + blk * kDd * kPg;
        if (kGather) {  // the page's [128][64] block, then token rows out of it
            for (int32_t c = threadIdx.x; c < kDd * kPg / 16; c += blockDim.x)
                reinterpret_cast<uint4 *>(tile)[c] = reinterpret_cast<const uint4 *>(vpage)[c];
            __syncthreads();
            for (int32_t w = threadIdx.x; w < nr * kDd / 8; w += blockDim.x) {
                const int32_t k = w / (kDd / 8), d0 = (w % (kDd / 8)) * 8;
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    lo |= (uint32_t)tile[(d0 + e) * kPg + r0 + k] << (8 * e);
                    hi |= (uint32_t)tile[(d0 + 4 + e) * kPg + r0 + k] << (8 * e);
                }
                reinterpret_cast<uint2 *>(pv + (int64_t)(i0 + k) * kDd)[d0 / 8] = make_uint2(lo, hi);
            }
        } else {  // the page's token rows into the tile, then its window columns back
            for (int32_t w = threadIdx.x; w < nr * kDd / 8; w += blockDim.x)
                reinterpret_cast<uint2 *>(tile)[w] = reinterpret_cast<const uint2 *>(pv + (int64_t)i0 * kDd)[w];
            __syncthreads();
            for (int32_t f = threadIdx.x; f < kDd * nr; f += blockDim.x) {
                const int32_t dd = f / nr, k = f % nr;
                vpage[dd * kPg + r0 + k] = tile[k * kDd + dd];
            }
        }
        __syncthreads();  // the tile is reused by the next page
    }
}

// FP8 append: one warp per (token, kv head). Each lane holds 4 of the 128
// elements of the K row and of the V row; the warp's amax gives the tile's
// scale = amax / 448 (1 for an all-zero tile), each element is divided by it
// (correctly rounded) and rounded to the nearest E4M3 code, saturating. K is
// written as a row of the page, V into column `row` of the transposed page.
__global__ void append_kv_fp8_kernel(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                                     uint8_t *kp, uint8_t *vp, float *ks, float *vs,
                                     const int32_t *__restrict__ slots, int64_t n_tokens, int32_t hkv,
                                     int32_t page, int64_t pool_slots, int *err) {
    const int lane = threadIdx.x & 31;
    const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (w >= n_tokens * hkv) return;
    const int64_t t = w / hkv;
    const int32_t g = (int32_t)(w % hkv);
    const int32_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= pool_slots) {
        if (lane == 0) set_error(err, HSWA_ERR_BOUNDS);
        return;
    }
    const int64_t blk = (int64_t)(slot / page) * hkv + g;  // (page, kv head) block
    const int32_t row = slot % page;
    for (int which = 0; which < 2; ++which) {
        const __nv_bfloat16 *src = (which ? v : k) + (t * hkv + g) * 128 + lane * 4;
        float x[4];
        for (int i = 0; i < 4; ++i) x[i] = __bfloat162float(src[i]);
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        uint8_t q[4];
        for (int i = 0; i < 4; ++i)
            q[i] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[i], scale), __NV_SATFINITE, __NV_E4M3);
        if (which == 0) {
            uint8_t *dst = kp + (blk * page + row) * 128 + lane * 4;
            *reinterpret_cast<uint32_t *>(dst) =
                (uint32_t)q[0] | ((uint32_t)q[1] << 8) | ((uint32_t)q[2] << 16) | ((uint32_t)q[3] << 24);
            if (lane == 0) ks[blk * page + row] = scale;
        } else {
            for (int i = 0; i < 4; ++i) vp[(blk * 128 + lane * 4 + i) * page + row] = q[i];
            if (lane == 0) vs[blk * page + row] = scale;
        }
    }
}

int esize(const hswa_config &c) { return c.dtype == HSWA_DTYPE_F32 ? 4 : 2; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

int grid_for(int64_t work, int block) {
    const int64_t g = (work + block - 1) / block;
    return (int)std::max<int64_t>(1, std::min<int64_t>(g, (int64_t)sm_count() * 32));
}

}  // namespace
}  // namespace hswa

using namespace hswa;

extern "C" int hswa_append_kv(const hswa_pool *pool, const hswa_layer *layer, const void *k, const void *v,
                              const int32_t *d_slots, int n_tokens, hswa_stream_t stream) {
    HSWA_NVTX("hswa_append_kv");
    if (!pool || !layer || n_tokens < 0 || (n_tokens > 0 && (!k || !v || !d_slots)) || !layer->k_pool ||
        !layer->v_pool || (layer->kind != HSWA_KIND_FULL && layer->kind != HSWA_KIND_SWA))
        return HSWA_ERR_INVALID_ARG;
    const hswa_config &c = pool->cfg;
    if (c.dtype == HSWA_DTYPE_FP8_E4M3) {
        if (c.head_dim != 128) return HSWA_ERR_UNSUPPORTED;
        if (!layer->k_scale || !layer->v_scale) return HSWA_ERR_INVALID_ARG;
        if (n_tokens == 0) return HSWA_OK;
        const int32_t num_pages = layer->kind == HSWA_KIND_SWA ? c.swa_pages : c.full_pages;
        const int64_t threads = (int64_t)n_tokens * c.n_kv_heads * 32;
        set_last_kernel("append_kv_fp8");
        append_kv_fp8_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
            (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, (uint8_t *)layer->k_pool, (uint8_t *)layer->v_pool,
            layer->k_scale, layer->v_scale, d_slots, n_tokens, c.n_kv_heads, c.page_size,
            (int64_t)num_pages * c.page_size, error_word());
        return cudaGetLastError() == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
    }
    const int64_t row_bytes = (int64_t)c.head_dim * esize(c);
    if (row_bytes % 16 || !aligned16(k) || !aligned16(v) || !aligned16(layer->k_pool) || !aligned16(layer->v_pool))
        return HSWA_ERR_UNSUPPORTED;
    if (n_tokens == 0) return HSWA_OK;
    const int32_t num_pages = layer->kind == HSWA_KIND_SWA ? c.swa_pages : c.full_pages;
    const int32_t cpr = (int32_t)(row_bytes / 16);
    const int64_t work = (int64_t)n_tokens * c.n_kv_heads * cpr;
    set_last_kernel("append_kv");
    append_kv_kernel<<<grid_for(work, 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        (const chunk_t *)k, (const chunk_t *)v, (chunk_t *)layer->k_pool, (chunk_t *)layer->v_pool, d_slots,
        n_tokens, c.n_kv_heads, c.page_size, cpr, (int64_t)num_pages * c.page_size, error_word());
    return cudaGetLastError() == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
}

static int swa_xfer(const hswa_pool *pool, const hswa_layer *layer, const int32_t *d_swa_bt,
                    const int32_t *d_seq_len, const int64_t *d_tok_offset, int n_seqs, void *buf, bool gather,
                    hswa_stream_t stream) {
    if (!pool || !layer || !d_swa_bt || !d_seq_len || !d_tok_offset || !buf || n_seqs < 0 ||
        n_seqs > pool->cfg.max_seqs || layer->kind != HSWA_KIND_SWA || layer->window <= 0 || !layer->k_pool ||
        !layer->v_pool)
        return HSWA_ERR_INVALID_ARG;
    const hswa_config &c = pool->cfg;
    if (c.dtype == HSWA_DTYPE_FP8_E4M3) {
        if (c.head_dim != 128 || c.page_size != 64 || !layer->k_scale || !layer->v_scale || !aligned16(layer->k_pool) ||
            !aligned16(layer->v_pool) || ((uintptr_t)layer->k_scale & 3) || ((uintptr_t)layer->v_scale & 3) ||
            ((uintptr_t)buf & 7))
            return HSWA_ERR_UNSUPPORTED;
        if (n_seqs == 0) return HSWA_OK;
        set_last_kernel(gather ? "swa_gather_fp8" : "swa_scatter_fp8");
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        const dim3 grid(c.n_kv_heads, n_seqs);
        if (gather)
            swa_xfer_fp8_kernel<true><<<grid, 256, 0, st>>>(
                (uint8_t *)layer->k_pool, (uint8_t *)layer->v_pool, layer->k_scale, layer->v_scale, (uint8_t *)buf,
                d_swa_bt, d_seq_len, d_tok_offset, c.max_pages_per_seq, c.n_kv_heads, layer->window, c.swa_pages,
                error_word());
        else
            swa_xfer_fp8_kernel<false><<<grid, 256, 0, st>>>(
                (uint8_t *)layer->k_pool, (uint8_t *)layer->v_pool, layer->k_scale, layer->v_scale, (uint8_t *)buf,
                d_swa_bt, d_seq_len, d_tok_offset, c.max_pages_per_seq, c.n_kv_heads, layer->window, c.swa_pages,
                error_word());
        return cudaGetLastError() == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
    }
    const int64_t row_bytes = (int64_t)c.head_dim * esize(c);
    if (row_bytes % 16 || !aligned16(buf) || !aligned16(layer->k_pool) || !aligned16(layer->v_pool))
        return HSWA_ERR_UNSUPPORTED;
    if (n_seqs == 0) return HSWA_OK;
    const int32_t cpr = (int32_t)(row_bytes / 16);
    const int block = 256;
    const int64_t per_seq_max = 2LL * c.n_kv_heads * layer->window * cpr;
    const int gx = (int)std::min<int64_t>((per_seq_max + block * 4 - 1) / (block * 4), 1024);
    set_last_kernel(gather ? "swa_gather" : "swa_scatter");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    dim3 grid(std::max(gx, 1), n_seqs);
    if (gather)
        swa_xfer_kernel<true><<<grid, block, 0, st>>>((chunk_t *)layer->k_pool, (chunk_t *)layer->v_pool,
                                                      (chunk_t *)buf, d_swa_bt, d_seq_len, d_tok_offset,
                                                      c.max_pages_per_seq, c.n_kv_heads, c.page_size,
                                                      layer->window, cpr, c.swa_pages, error_word());
    else
        swa_xfer_kernel<false><<<grid, block, 0, st>>>((chunk_t *)layer->k_pool, (chunk_t *)layer->v_pool,
                                                       (chunk_t *)buf, d_swa_bt, d_seq_len, d_tok_offset,
                                                       c.max_pages_per_seq, c.n_kv_heads, c.page_size,
                                                       layer->window, cpr, c.swa_pages, error_word());
    return cudaGetLastError() == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
}

extern "C" int hswa_swa_window_offsets(const hswa_pool *pool, const hswa_layer *layer, int n_seqs,
                                       const int32_t *seq_len, int64_t *tok_offset_out, size_t *packed_bytes_out) {
    if (!pool || !layer || !tok_offset_out || n_seqs < 0 || n_seqs > pool->cfg.max_seqs ||
        layer->kind != HSWA_KIND_SWA || layer->window <= 0)
        return HSWA_ERR_INVALID_ARG;
    const hswa_config &c = pool->cfg;
    const int32_t *lens = seq_len ? seq_len : pool->seq_len.data();
    int64_t off = 0;
    tok_offset_out[0] = 0;
    for (int i = 0; i < n_seqs; ++i) {
        if (lens[i] < 0) return HSWA_ERR_INVALID_ARG;
        off += std::min<int64_t>(lens[i], layer->window);
        tok_offset_out[i + 1] = off;
    }
    if (packed_bytes_out) {
        const int64_t per_token = c.dtype == HSWA_DTYPE_FP8_E4M3 ? 2LL * c.n_kv_heads * (c.head_dim + 4)
                                                                 : 2LL * c.n_kv_heads * c.head_dim * esize(c);
        *packed_bytes_out = (size_t)(off * per_token);
    }
    return HSWA_OK;
}

extern "C" int hswa_swa_gather(const hswa_pool *pool, const hswa_layer *layer, const int32_t *d_swa_bt,
                               const int32_t *d_seq_len, const int64_t *d_tok_offset, int n_seqs, void *dst,
                               hswa_stream_t stream) {
    HSWA_NVTX("hswa_swa_gather");
    return swa_xfer(pool, layer, d_swa_bt, d_seq_len, d_tok_offset, n_seqs, dst, true, stream);
}

extern "C" int hswa_swa_scatter(const hswa_pool *pool, const hswa_layer *layer, const int32_t *d_swa_bt,
                                const int32_t *d_seq_len, const int64_t *d_tok_offset, int n_seqs, const void *src,
                                hswa_stream_t stream) {
    HSWA_NVTX("hswa_swa_scatter");
    return swa_xfer(pool, layer, d_swa_bt, d_seq_len, d_tok_offset, n_seqs, const_cast<void *>(src), false,
                    stream);
}
