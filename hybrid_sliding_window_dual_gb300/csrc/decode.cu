// Decode attention over the dual KV pool (one new token per sequence).
//
// "MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 1.2: decode is
// close to memory-bandwidth-bound and its cost follows the KV bytes read;
// Sec. 2.1 / 5.1: Full layers read the O(N) Full pool, SWA layers only the
// O(W) window of the SWA pool.
//
// Fast path (bf16, d = 128, 8 query heads per kv head, page 64):
//   * The work is the list of (sequence, kv head, page) units, sequences in
//     order. Each CTA takes an equal contiguous share of that list
//     (stream-K style), so CTAs stay balanced whatever the length mix. A
//     piece of a (sequence, kv head) segment that a CTA covers alone is
//     written straight to o; a segment cut between CTAs leaves partial
//     (max, sum, unnormalised o) records that decode_combine merges.
//   * Warp 1 (producer) streams one page of one kv head per stage: K and V
//     as two 64x64 tensor-map boxes each (128-byte swizzle), plus the 8 query
//     rows at the first page of a piece, into a 3-stage mbarrier ring.
//   * Warp 0 (consumer) computes S^T = K Q^T (16 keys x 8 heads per
//     mma.m16n8k16, the 8 GQA heads filling N = 8), an online softmax in the
//     log2 domain, transposes P with movmatrix and accumulates
//     O^T += V^T P^T with V^T read by ldmatrix.trans.
// Multi-token decode (n_tok query tokens per sequence at positions
// L - n_tok .. L - 1: the MTP verification step of "MiMo-V2.5 Series
// Inference Full-Link Optimization", Sec. 5.2, and the multi-token
// verification of "Following the Bottleneck: Optimizing MiniMax M3 on AMD
// Instinct MI355X", EAGLE3 section): up to 3 tokens the same kernel with one
// consumer warp per token; 4 to 16 tokens a tcgen05 kernel whose
// (token, head) rows form one M = 128 tile ("tensor-core multi-token" below).
// Generic path (any dtype / head_dim / ratio / page): one warp per
// (sequence, query head) with CUDA-core dot products.
#include <algorithm>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "kernels.h"
#include "tc.cuh"

namespace hswa {
namespace {

constexpr int kD = 128;
constexpr int kG = 8;
constexpr int kP = 64;
constexpr int kStages = 3;
constexpr uint32_t kBoxBytes = 64 * 128;           // 64 rows x 128 bytes
constexpr uint32_t kPageHeadBytes = 2 * kBoxBytes;  // one page of one kv head
constexpr uint32_t kQBytes = kG * kD * 2;

enum : int32_t { kFirst = 1, kLast = 2, kDirect = 4, kSkip = 8 };

struct StageDesc {
    int32_t seq, kvh, lo, hi, flags, slot;
    int32_t key0;  // absolute position of the page's first key
    int32_t len;   // keys of the sequence (its last query sits at len - 1)
};

// kTok query tokens per sequence share every streamed page (one consumer
// warp each): 1 for plain decode, 2 or 3 for multi-token decode.
template <int kTok_>
struct DecodeSmemT {
    static constexpr int kTok = kTok_;
    static constexpr int kStages = kTok_ <= 2 ? ::hswa::kStages : 2;
    static constexpr bool kTcQ = false;  // q rows travel with the first page of a piece
    uint8_t k[kStages][kPageHeadBytes];
    uint8_t v[kStages][kPageHeadBytes];
    uint8_t q[kStages][kTok * kQBytes];
    StageDesc desc[kStages];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int32_t abort;
};

template <int kTok>
constexpr size_t decode_smem_bytes() { return sizeof(DecodeSmemT<kTok>) + 1024; }  // + alignment slack

// FP8 pools: a stage holds one page of one kv head as E4M3 codes, K as
// [64 keys][128 B] (128-byte swizzle) and V transposed as [128 d][64 B]
// (64-byte swizzle), plus the 64 K and 64 V scales of the page.
constexpr uint32_t kK8Bytes = kP * kD;
constexpr uint32_t kV8Bytes = kD * kP;
constexpr uint32_t kScaleBytes = kP * 4;

constexpr int kConsumers8 = 4;  // FP8 consumer warps, one 16-key group of a page each

template <int kTok>
struct DecodeSmem8T {
    static constexpr int kStages = 3;
    static constexpr bool kTcQ = false;
    uint8_t k[kStages][kK8Bytes];
    uint8_t v[kStages][kV8Bytes];
    uint8_t q[kStages][kTok * kQBytes];
    float ks[kStages][kP];
    float vs[kStages][kP];
    // end-of-piece merge of the consumer warps' (max, sum, o) states
    float mo[kConsumers8 - 1][kTok][kG][kD];
    float mm[kConsumers8 - 1][kTok][kG];
    float ml[kConsumers8 - 1][kTok][kG];
    StageDesc desc[kStages];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t merge;
    int32_t abort;
};

template <int kTok>
constexpr size_t decode_smem8_bytes() { return sizeof(DecodeSmem8T<kTok>) + 1024; }

struct Partial {
    float m[kG];
    float l[kG];
    float o[kG][kD];
};

struct DecodeArgs {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *o;
    const int32_t *bt;
    const int32_t *seq_len;
    const int4 *sdesc;    // [n_seqs + 1] {first unit, key lo, key hi, units}; [n].x = total
    __nv_bfloat16 *k_pool, *v_pool;
    const float *k_scale, *v_scale;  // FP8 pools: [pages][Hkv][P] each
    Partial *part;        // [n_ctas][2]
    // optional fused append: new K / V rows [n_seqs][Hkv][d] written at
    // slots[s] before the page that holds them is streamed (null = none)
    const int32_t *slots;
    const __nv_bfloat16 *k_new, *v_new;
    int64_t pool_slots;
    int32_t n_seqs, bt_stride, hkv, hq, window, num_pages;
    int32_t n_tok;  // query tokens per sequence (multi-token decode), 1 otherwise
    float scale_log2;
    int *err;
};

// Row of q / o holding query token w of sequence s.
__device__ __forceinline__ int64_t q_row(const DecodeArgs &a, int32_t s, int32_t w) {
    return (int64_t)s * a.n_tok + w;
}

// Tensor-core multi-token decode: copies of the 8 n_tok query rows in the
// 128-row tile (each copy takes 64 / copies keys of every page).
__host__ __device__ constexpr int tc_copies(int n_tok) { return n_tok <= 4 ? 4 : n_tok <= 8 ? 2 : 1; }

// Keys [lo, hi) that the last n_tok query tokens of a sequence with L keys
// attend together (positions L - n_tok .. L - 1; W keys each for SWA).
__device__ __forceinline__ void key_range(int32_t L, int32_t window, int32_t n_tok, int32_t &lo, int32_t &hi) {
    hi = L;
    lo = (window > 0 && L - n_tok + 1 - window > 0) ? L - n_tok + 1 - window : 0;
}

// Per-sequence descriptors: the first unit of the sequence (prefix sum of
// units(s) = Hkv * pages touched by the key range [lo, hi)), lo, hi, units.
// desc[n].x is the total number of units.
__global__ void decode_plan(const int32_t *__restrict__ seq_len, int32_t n, int32_t hkv, int32_t page,
                            int32_t window, int32_t n_tok, int4 *__restrict__ desc) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int32_t base = 0; base < n; base += blockDim.x) {
        const int32_t i = base + tid;
        int32_t u = 0, lo = 0, hi = 0;
        if (i < n) {
            key_range(seq_len[i], window, n_tok, lo, hi);
            if (hi > lo) u = hkv * ((hi - 1) / page - lo / page + 1);
        }
        int32_t x = u;  // inclusive warp scan
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int32_t t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += y;
            }
            warp_tot[lane] = t;  // inclusive scan of warp totals
        }
        __syncthreads();
        const int32_t excl = carry + (wid > 0 ? warp_tot[wid - 1] : 0) + x - u;
        if (i < n) desc[i] = make_int4(excl, lo, hi, u);
        __syncthreads();
        if (tid == blockDim.x - 1) carry = excl + u;
        __syncthreads();
    }
    if (tid == 0) desc[n] = make_int4(carry, 0, 0, 0);
}

__device__ __forceinline__ int64_t cta_start(int64_t c, int64_t U, int64_t N) { return c * U / N; }

// Largest c with cta_start(c) <= u.
__device__ __forceinline__ int64_t cta_of(int64_t u, int64_t U, int64_t N) { return ((u + 1) * N - 1) / U; }

// Largest s in [0, n) with desc[s].x <= u (first units non-decreasing,
// desc[0].x = 0 <= u). A 32-way search: every lane probes one position, so
// each step is one round of loads for the whole warp.
__device__ int32_t find_seq(const int4 *desc, int32_t n, int64_t u) {
    const int lane = threadIdx.x & 31;
    int32_t lo = 0, hi = n - 1;  // the answer lies in [lo, hi]
    while (hi - lo >= 32) {
        const int32_t step = (hi - lo + 32) / 32;
        const int32_t idx = min(lo + lane * step, hi);
        const unsigned m = __ballot_sync(0xffffffffu, desc[idx].x <= u);
        const int32_t last = 31 - __clz(m);  // lane 0 probes lo, always true
        lo += last * step;
        hi = min(lo + step - 1, hi);
    }
    const int32_t idx = lo + lane;
    const unsigned m = __ballot_sync(0xffffffffu, idx <= hi && desc[idx].x <= u);
    return lo + 31 - __clz(m);
}

// Byte offset of the 16-byte chunk holding (row, d..d+7) in a stage buffer
// loaded as two 64-column boxes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int d) {
    return (uint32_t)((d >> 6) * kBoxBytes + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4));
}

// Streams the pages of units [u0, u1) into the stage ring. With
// Smem::kTcQ the query tile of each piece goes by tensor map tq into the
// q buffer of Smem::kQBufs slots (released by the MMA thread through q_empty) instead of
// travelling in the stage of the piece's first page.
template <bool kFP8, class Smem>
__device__ void decode_producer(Smem &sm, const CUtensorMap *tk, const CUtensorMap *tv, const DecodeArgs &a,
                                int64_t u0, int64_t u1, const CUtensorMap *tq = nullptr) {
    constexpr int kStages = Smem::kStages;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        prefetch_tmap(tk);
        prefetch_tmap(tv);
        if constexpr (Smem::kTcQ) prefetch_tmap(tq);
    }
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_parity[kStages];
    bool issued[kStages];
    for (int i = 0; i < kStages; ++i) issued[i] = false, issued_parity[i] = 0;
    int32_t pc = 0;  // pieces started (kTcQ: q slot pc & 1)
    bool q_issued[2] = {false, false};
    uint32_t q_parity[2] = {0, 0};

    int64_t u = u0;
    int32_t s = 0;
    int4 d = make_int4(0, 0, 0, 0), dn = d;
    if (u0 < u1) {
        s = find_seq(a.sdesc, a.n_seqs, u0);
        d = a.sdesc[s];
        dn = a.sdesc[s + 1];  // prefetched: the next sequence's descriptor
    }
    // block-table entries of the current sequence, 32 pages per batch, one
    // page per lane; reused by the kv heads of the sequence
    int32_t cached_s = -1, cached_batch = -1, mine = -1;
    while (u < u1) {
        while (u >= (int64_t)d.x + d.w) {  // next sequence with units
            ++s;
            d = dn;
            dn = a.sdesc[s + 1];
        }
        const int32_t lo = d.y, hi = d.z;
        const int32_t pf = lo / kP;
        const int32_t npg = d.w / a.hkv;
        const int64_t seg0 = d.x;
        const int32_t g = (int32_t)((u - seg0) / npg);
        const int32_t pi = (int32_t)((u - seg0) % npg);
        const int64_t seg_start = seg0 + (int64_t)g * npg, seg_end = seg_start + npg;
        const int64_t piece_end = seg_end < u1 ? seg_end : u1;
        const int32_t n = (int32_t)(piece_end - u);
        const bool direct = (u == seg_start) && (piece_end == seg_end);
        const int32_t slot = (u == u0) ? 0 : 1;
        const int32_t *btrow = a.bt + (int64_t)s * a.bt_stride;
        for (int32_t j = 0; j < n; ++j) {
            const int32_t p = pi + j;  // page index in the sequence's key range
            if (s != cached_s || (p >> 5) != cached_batch) {
                cached_s = s;
                cached_batch = p >> 5;
                const int32_t q = (p & ~31) + lane;
                mine = (q < npg && pf + q < a.bt_stride) ? btrow[pf + q] : -1;
            }
            const int32_t page = __shfl_sync(0xffffffffu, mine, p & 31);
            if (!kFP8 && a.slots && p == npg - 1) {
                // fused append: the new token (position hi - 1) lies on the
                // last page of the range; write its K and V rows of this kv
                // head (lanes 0-15: K, 16-31: V, 16 bytes each) before the
                // page is streamed
                const int32_t slot = a.slots[s];
                if (slot >= 0 && slot < a.pool_slots) {
                    const int64_t dst = (((int64_t)(slot / kP) * a.hkv + g) * kP + slot % kP) * kD;
                    const int64_t src = ((int64_t)s * a.hkv + g) * kD;
                    const int c = (lane & 15) * 8;
                    const __nv_bfloat16 *from = (lane < 16 ? a.k_new : a.v_new) + src + c;
                    __nv_bfloat16 *to = (lane < 16 ? a.k_pool : a.v_pool) + dst + c;
                    *reinterpret_cast<uint4 *>(to) = *reinterpret_cast<const uint4 *>(from);
                } else if (slot >= a.pool_slots && lane == 0) {
                    set_error(a.err, HSWA_ERR_BOUNDS);
                }
                fence_proxy_async_global();
                __syncwarp();
            }
            bool ok = true;
            if (lane == 0) {
                if constexpr (Smem::kTcQ) {
                    if (j == 0) {
                        // the piece's n_tok x 8 query rows (token, head), once
                        // per copy: copy cp starts at tile row cp * 128 / R
                        const int b = pc % Smem::kQBufs;
                        const uint32_t par = (pc / Smem::kQBufs) & 1;
                        const int copies = tc_copies(a.n_tok);
                        ok = mbar_wait(&sm.q_empty[b], par ^ 1, a.err) && !*(volatile int32_t *)&sm.abort;
                        if (ok) {
                            mbar_arrive_expect_tx(&sm.q_full[b], copies * a.n_tok * kQBytes);
                            for (int cp = 0; cp < copies; ++cp)
                                for (int dh = 0; dh < 2; ++dh)
                                    tma_load_3d(sm.q[b] + dh * Smem::kQHalfBytes + cp * (128 / copies) * 128, tq,
                                                dh * 64, g * kG, (int32_t)q_row(a, s, 0), &sm.q_full[b]);
                            q_issued[b] = true;
                            q_parity[b] = par;
                        }
                        ++pc;
                    }
                }
                ok = ok && mbar_wait(&sm.empty[stage], phase ^ 1, a.err) && !*(volatile int32_t *)&sm.abort;
                if (ok) {
                    const int32_t lp = pf + pi + j;
                    const int32_t key0 = lp * kP;
                    StageDesc &d = sm.desc[stage];
                    d.seq = s;
                    d.kvh = g;
                    d.lo = lo - key0 > 0 ? lo - key0 : 0;
                    d.hi = hi - key0 < kP ? hi - key0 : kP;
                    d.slot = slot;
                    d.key0 = key0;
                    d.len = hi;
                    int32_t flags = (j == 0 ? kFirst : 0) | (j == n - 1 ? kLast : 0) | (direct ? kDirect : 0);
                    const bool valid = page >= 0 && page < a.num_pages;
                    if (!valid) {
                        set_error(a.err, HSWA_ERR_BOUNDS);
                        flags |= kSkip;
                    }
                    d.flags = flags;
                    const uint32_t page_bytes = kFP8 ? kK8Bytes + kV8Bytes + 2 * kScaleBytes : 4 * kBoxBytes;
                    const uint32_t q_bytes = (!Smem::kTcQ && j == 0) ? a.n_tok * kQBytes : 0;
                    const uint32_t bytes = (valid ? page_bytes : 0) + q_bytes;
                    if (bytes) {
                        mbar_arrive_expect_tx(&sm.full[stage], bytes);
                        if (valid) {
                            const int32_t blk = page * a.hkv + g;  // (page, kv head) block
                            if constexpr (kFP8) {
                                tma_load_2d(sm.k[stage], tk, 0, blk * kP, &sm.full[stage]);
                                tma_load_2d(sm.v[stage], tv, 0, blk * kD, &sm.full[stage]);
                                bulk_g2s(sm.ks[stage], a.k_scale + (int64_t)blk * kP, kScaleBytes, &sm.full[stage]);
                                bulk_g2s(sm.vs[stage], a.v_scale + (int64_t)blk * kP, kScaleBytes, &sm.full[stage]);
                            } else {
                                const int32_t row = blk * kP;
                                tma_load_2d(sm.k[stage], tk, 0, row, &sm.full[stage]);
                                tma_load_2d(sm.k[stage] + kBoxBytes, tk, 64, row, &sm.full[stage]);
                                tma_load_2d(sm.v[stage], tv, 0, row, &sm.full[stage]);
                                tma_load_2d(sm.v[stage] + kBoxBytes, tv, 64, row, &sm.full[stage]);
                            }
                        }
                        if constexpr (!Smem::kTcQ) {
                            if (j == 0)  // the 8 query rows of each token of this kv head
                                for (int w = 0; w < a.n_tok; ++w)
                                    bulk_g2s(sm.q[stage] + w * kQBytes,
                                             a.q + (q_row(a, s, w) * a.hq + (int64_t)g * kG) * kD, kQBytes,
                                             &sm.full[stage]);
                        }
                    } else {
                        mbar_arrive(&sm.full[stage]);
                    }
                    issued[stage] = true;
                    issued_parity[stage] = phase;
                } else {
                    sm.abort = 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) goto drain;
            if (++stage == kStages) stage = 0, phase ^= 1;
        }
        u = piece_end;
    }
drain:
    // never leave the CTA with copies still landing in its shared memory
    if (lane == 0) {
        for (int i = 0; i < kStages; ++i)
            if (issued[i]) mbar_wait(&sm.full[i], issued_parity[i], a.err);
        if constexpr (Smem::kTcQ)
            for (int b = 0; b < Smem::kQBufs; ++b)
                if (q_issued[b]) mbar_wait(&sm.q_full[b], q_parity[b], a.err);
    }
}

// One consumer warp: query token w (8 query heads) of the stage's (sequence,
// kv head).
template <int kTok>
__device__ void decode_consumer(DecodeSmemT<kTok> &sm, const DecodeArgs &a, int64_t u0, int64_t u1, int w) {
    constexpr int kStages = DecodeSmemT<kTok>::kStages;
    const int lane = threadIdx.x & 31;
    const int gr = lane >> 2;  // fragment row group
    const int qd = lane & 3;   // fragment column pair
    uint32_t qf[8][2];
    float oacc[8][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int stage = 0;
    uint32_t phase = 0;
    const uint32_t kbase = smem_u32(sm.k[0]), vbase = smem_u32(sm.v[0]);

    for (int64_t u = u0; u < u1; ++u) {
        bool ok = mbar_wait(&sm.full[stage], phase, a.err) && !*(volatile int32_t *)&sm.abort;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) sm.abort = 1;
            return;
        }
        const StageDesc d = sm.desc[stage];
        if (d.flags & kFirst) {
            const uint32_t *qs = reinterpret_cast<const uint32_t *>(sm.q[stage] + w * kQBytes);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qf[ks][0] = qs[(gr * kD + ks * 16 + 2 * qd) >> 1];
                qf[ks][1] = qs[(gr * kD + ks * 16 + 8 + 2 * qd) >> 1];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }
        if (!(d.flags & kSkip)) {
            const uint32_t kb = kbase + stage * kPageHeadBytes, vb = vbase + stage * kPageHeadBytes;
            // S^T = K Q^T : 4 tiles of 16 keys
            float sacc[4][4];
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                sacc[kt][0] = sacc[kt][1] = sacc[kt][2] = sacc[kt][3] = 0.f;
                const int row = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kb + swz(row, ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
                    mma_bf16_16816(sacc[kt], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                }
            }
            // scale to log2 units and mask the keys this token does not see:
            // its position is t = len - n_tok + w; keys (key0 + r) <= t and,
            // for SWA, > t - W, inside the page's part of the range [lo, hi)
            int32_t r_lo = d.lo, r_hi = d.hi;  // one token: the stage's range is its own
            if constexpr (kTok > 1) {
                const int32_t t = d.len - a.n_tok + w;
                r_hi = min(d.hi, t - d.key0 + 1);
                if (a.window > 0) r_lo = max(d.lo, t - a.window + 1 - d.key0);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                const int r0 = kt * 16 + gr, r1 = r0 + 8;
                const bool v0 = r0 >= r_lo && r0 < r_hi, v1 = r1 >= r_lo && r1 < r_hi;
                sacc[kt][0] = v0 ? sacc[kt][0] * a.scale_log2 : -INFINITY;
                sacc[kt][1] = v0 ? sacc[kt][1] * a.scale_log2 : -INFINITY;
                sacc[kt][2] = v1 ? sacc[kt][2] * a.scale_log2 : -INFINITY;
                sacc[kt][3] = v1 ? sacc[kt][3] * a.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(sacc[kt][0], sacc[kt][2]));
                mx1 = fmaxf(mx1, fmaxf(sacc[kt][1], sacc[kt][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            // with several tokens a page can hold no key that a token sees
            // (n = -inf): then nothing is kept and P stays 0
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            float b0 = n0, b1 = n1, al0, al1;
            if constexpr (kTok > 1) {
                b0 = n0 == -INFINITY ? 0.f : n0;
                b1 = n1 == -INFINITY ? 0.f : n1;
                al0 = n0 == -INFINITY ? 1.f : fast_exp2(m0 - n0);
                al1 = n1 == -INFINITY ? 1.f : fast_exp2(m1 - n1);
            } else {  // a stage holds at least one key of the range: n0, n1 finite
                al0 = fast_exp2(m0 - n0);
                al1 = fast_exp2(m1 - n1);
            }
            m0 = n0;
            m1 = n1;
            float ps0 = 0.f, ps1 = 0.f;
            uint32_t pb[4][2];
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                const float p0 = fast_exp2(sacc[kt][0] - b0), p1 = fast_exp2(sacc[kt][1] - b1);
                const float p2 = fast_exp2(sacc[kt][2] - b0), p3 = fast_exp2(sacc[kt][3] - b1);
                const uint32_t x0 = pack_bf16(p0, p1), x1 = pack_bf16(p2, p3);
                // sum what the MMA will see (the bf16-rounded weights)
                const __nv_bfloat162 r0 = *reinterpret_cast<const __nv_bfloat162 *>(&x0);
                const __nv_bfloat162 r1 = *reinterpret_cast<const __nv_bfloat162 *>(&x1);
                ps0 += __low2float(r0) + __low2float(r1);
                ps1 += __high2float(r0) + __high2float(r1);
                pb[kt][0] = movmatrix_t(x0);
                pb[kt][1] = movmatrix_t(x1);
            }
            l0 = l0 * al0 + ps0;
            l1 = l1 * al1 + ps1;
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                oacc[dt][0] *= al0;
                oacc[dt][1] *= al1;
                oacc[dt][2] *= al0;
                oacc[dt][3] *= al1;
            }
            // O^T += V^T P^T
            const int jj = lane >> 3;
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                const int key = kt * 16 + (lane & 7) + (jj >> 1) * 8;
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(vb + swz(key, dt * 16 + (jj & 1) * 8), a0, a1, a2, a3);
                    mma_bf16_16816(oacc[dt], a0, a1, a2, a3, pb[kt][0], pb[kt][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);

        if (d.flags & kLast) {
            float t0 = l0, t1 = l1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                t0 += __shfl_xor_sync(0xffffffffu, t0, off);
                t1 += __shfl_xor_sync(0xffffffffu, t1, off);
            }
            const int h0 = 2 * qd, h1 = 2 * qd + 1;
            if (d.flags & kDirect) {
                const float i0 = t0 > 0.f ? 1.f / t0 : 0.f, i1 = t1 > 0.f ? 1.f / t1 : 0.f;
                __nv_bfloat16 *o0 = a.o + (q_row(a, d.seq, w) * a.hq + (int64_t)d.kvh * kG + h0) * kD;
                __nv_bfloat16 *o1 = o0 + kD;
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    o0[dt * 16 + gr] = __float2bfloat16_rn(oacc[dt][0] * i0);
                    o1[dt * 16 + gr] = __float2bfloat16_rn(oacc[dt][1] * i1);
                    o0[dt * 16 + gr + 8] = __float2bfloat16_rn(oacc[dt][2] * i0);
                    o1[dt * 16 + gr + 8] = __float2bfloat16_rn(oacc[dt][3] * i1);
                }
            } else {
                Partial &p = a.part[((int64_t)blockIdx.x * 2 + d.slot) * a.n_tok + w];
                if (gr == 0) {
                    p.m[h0] = m0;
                    p.m[h1] = m1;
                    p.l[h0] = t0;
                    p.l[h1] = t1;
                }
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    p.o[h0][dt * 16 + gr] = oacc[dt][0];
                    p.o[h1][dt * 16 + gr] = oacc[dt][1];
                    p.o[h0][dt * 16 + gr + 8] = oacc[dt][2];
                    p.o[h1][dt * 16 + gr + 8] = oacc[dt][3];
                }
            }
        }
        if (++stage == kStages) stage = 0, phase ^= 1;
    }
}

// Consumer warps 0 .. kTok - 1, one query token each (warps past n_tok stay
// idle); warp kTok is the producer.
template <int kTok>
__global__ void __launch_bounds__(32 * (kTok + 1)) decode_mma_bf16_d128(const __grid_constant__ CUtensorMap tk,
                                                                      const __grid_constant__ CUtensorMap tv,
                                                                      DecodeArgs a) {
    using Smem = DecodeSmemT<kTok>;
    extern __shared__ uint8_t raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    if (threadIdx.x == 0) {
        for (int i = 0; i < Smem::kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], a.n_tok);  // the active consumer warps
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();  // the plan (and the table update before it) is complete
    pdl_launch_dependents();
    const int64_t U = a.sdesc[a.n_seqs].x, N = gridDim.x;
    if (U == 0) return;
    const int64_t u0 = cta_start(blockIdx.x, U, N), u1 = cta_start(blockIdx.x + 1, U, N);
    const int warp = threadIdx.x >> 5;
    if (warp == kTok)
        decode_producer<false>(sm, &tk, &tv, a, u0, u1);
    else if (warp < a.n_tok)
        decode_consumer<kTok>(sm, a, u0, u1, warp);
}

// ---------------------------------------------------------- FP8 decode
// Key rows of a 16-key group in the order the QK MMA's A rows take them:
// after the movmatrix transpose of S^T, thread (g, q) then holds P for the
// keys 4q..4q+3 that one 32-bit load of an E4M3 row gives the PV MMA. A rows
// 0-7 take keys {0,1,4,5,10,11,14,15} and rows 8-15 the others, so the eight
// rows of each ldmatrix tile differ in (key & 7) and hit eight different
// 16-byte chunks of the 128-byte swizzle. For q >= 2 the first P pair is
// keys 4q+2, 4q+3: the PV side takes the word's upper two codes first there.
__device__ __forceinline__ int key_of_row(int r) {
    const int q = (r & 7) >> 1;
    return 4 * q + (r & 1) + 2 * ((r >> 3) ^ (q >> 1));
}

// 16-byte chunk of (row, byte) in a [rows][128 B] tile with the 128-byte
// swizzle, and in a [rows][64 B] tile with the 64-byte swizzle.
__device__ __forceinline__ uint32_t swz128(int row, int byte) {
    return (uint32_t)(row * 128 + ((((byte >> 4) ^ (row & 7)) & 7) << 4));
}
__device__ __forceinline__ uint32_t swz64(int row, int byte) {
    return (uint32_t)(row * 64 + ((((byte >> 4) ^ (row >> 1)) & 3) << 4));
}

// Four E4M3 codes (bytes b0..b3 of r) as two exact f16 pairs {b0, b1},
// {b2, b3}: the hardware conversion, two instructions per word (every E4M3
// value, subnormals included, is an f16 value).
__device__ __forceinline__ void e4m3x4_f16x2x2_cvt(uint32_t r, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(r));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Bounded arrival + wait on the consumer warps' merge barrier (128 threads):
// a barrier that gives up (HSWA_ERR_TIMEOUT) if a warp never arrives.
template <class Smem>
__device__ __forceinline__ bool merge_sync(Smem &sm, uint32_t &phase, int *err) {
    mbar_arrive(&sm.merge);
    const bool ok = mbar_wait(&sm.merge, phase, err);
    phase ^= 1;
    return ok;
}

// The consumers over FP8 pages, kTok query tokens per pass (1 or 2). Warp w
// takes the 16 keys 16w..16w+15 of every page: S^T = (K codes as f16) Q^T
// with the key rows taken in key_of_row order and d read 4 codes at a time
// (Q's fragments use the same d order), times the per-key K scale; an online
// softmax of its own per token; P times the per-key V scale feeds the f16 PV
// MMA, whose A operand (V^T) comes from the transposed page without any
// transpose. Every converted K and V fragment feeds the MMAs of all kTok
// tokens. At the end of a piece warps 1-3 hand their (max, sum, o) to warp 0
// through shared memory, which merges and writes.
template <int kTok>
__device__ void decode_consumer_fp8(DecodeSmem8T<kTok> &sm, const DecodeArgs &a, int64_t u0, int64_t u1) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int gr = lane >> 2, qd = lane & 3;
    constexpr int kStages = DecodeSmem8T<kTok>::kStages;
    uint32_t qf[kTok][8][2];
    float oacc[kTok][8][4];
    float m0[kTok], m1[kTok], l0[kTok], l1[kTok];
#pragma unroll
    for (int j = 0; j < kTok; ++j) m0[j] = m1[j] = -INFINITY, l0[j] = l1[j] = 0.f;
    int stage = 0;
    uint32_t phase = 0, merge_phase = 0;
    const uint32_t kbase = smem_u32(sm.k[0]), vbase = smem_u32(sm.v[0]);
    const int jj = lane >> 3;
    const int ar = (lane & 7) + 8 * (jj & 1);  // A row this lane addresses in ldmatrix (QK)
    const int c0 = w * 16 + key_of_row(gr), c1 = w * 16 + key_of_row(gr + 8);  // keys of this thread's S rows
    // a V word's code pairs in the order this thread's P pairs take them
    // (key_of_row): as loaded, or its two halves swapped for q >= 2
    const uint32_t vsel = qd >= 2 ? 0x1032u : 0x3210u;

    for (int64_t u = u0; u < u1; ++u) {
        bool ok = mbar_wait(&sm.full[stage], phase, a.err) && !*(volatile int32_t *)&sm.abort;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) sm.abort = 1;
            return;
        }
        const StageDesc d = sm.desc[stage];
        if (d.flags & kFirst) {
#pragma unroll
            for (int j = 0; j < kTok; ++j) {
                const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(sm.q[stage] + j * kQBytes) + gr * kD;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int c = ks * 16 + 4 * qd;
                    qf[j][ks][0] = pack_f16(__bfloat162float(qs[c]), __bfloat162float(qs[c + 1]));
                    qf[j][ks][1] = pack_f16(__bfloat162float(qs[c + 2]), __bfloat162float(qs[c + 3]));
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) oacc[j][i][0] = oacc[j][i][1] = oacc[j][i][2] = oacc[j][i][3] = 0.f;
                m0[j] = m1[j] = -INFINITY;
                l0[j] = l1[j] = 0.f;
            }
        }
        const bool any = !(d.flags & kSkip) && w * 16 + 15 >= d.lo && w * 16 < d.hi;
        if (any) {
            const uint32_t kb = kbase + stage * kK8Bytes, vb = vbase + stage * kV8Bytes;
            float sacc[kTok][4];
#pragma unroll
            for (int j = 0; j < kTok; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
            const int key = w * 16 + key_of_row(ar);
#pragma unroll
            for (int dc = 0; dc < 4; ++dc) {
                uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
                ldsm_x4(kb + swz128(key, dc * 32 + 16 * (jj >> 1)), r0, r1, r2, r3);
                e4m3x4_f16x2x2_cvt(r0, a0, a2);
                e4m3x4_f16x2x2_cvt(r1, a1, a3);
#pragma unroll
                for (int j = 0; j < kTok; ++j) mma_f16_16816(sacc[j], a0, a1, a2, a3, qf[j][2 * dc][0], qf[j][2 * dc][1]);
                e4m3x4_f16x2x2_cvt(r2, a0, a2);
                e4m3x4_f16x2x2_cvt(r3, a1, a3);
#pragma unroll
                for (int j = 0; j < kTok; ++j)
                    mma_f16_16816(sacc[j], a0, a1, a2, a3, qf[j][2 * dc + 1][0], qf[j][2 * dc + 1][1]);
            }
            // K codes entered the MMA as their exact values
            const float s0 = sm.ks[stage][c0] * a.scale_log2;
            const float s1 = sm.ks[stage][c1] * a.scale_log2;
            // V codes enter the MMA as their exact values; P carries the V
            // scale times 2^8 (keeping small weights out of f16's subnormal
            // range), and so does the running sum: O / l stays exact
            const float w0 = sm.vs[stage][c0] * 256.f, w1 = sm.vs[stage][c1] * 256.f;
            uint32_t pb0[kTok], pb1[kTok];
#pragma unroll
            for (int j = 0; j < kTok; ++j) {
                // keys of the page token j sees: its position is
                // t = len - n_tok + j; keys <= t and, for SWA, > t - W
                int32_t lo = d.lo, hi = d.hi;  // one token: the stage's range is its own
                if constexpr (kTok > 1) {
                    const int32_t t = d.len - a.n_tok + j;
                    hi = min(d.hi, t - d.key0 + 1);
                    if (a.window > 0) lo = max(d.lo, t - a.window + 1 - d.key0);
                }
                const bool v0 = c0 >= lo && c0 < hi, v1 = c1 >= lo && c1 < hi;
                sacc[j][0] = v0 ? sacc[j][0] * s0 : -INFINITY;
                sacc[j][1] = v0 ? sacc[j][1] * s0 : -INFINITY;
                sacc[j][2] = v1 ? sacc[j][2] * s1 : -INFINITY;
                sacc[j][3] = v1 ? sacc[j][3] * s1 : -INFINITY;
                float mx0 = fmaxf(sacc[j][0], sacc[j][2]), mx1 = fmaxf(sacc[j][1], sacc[j][3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                // this warp saw at least one valid key in the piece so far
                // (n > -inf), else it keeps nothing and P stays 0
                const float n0 = fmaxf(m0[j], mx0), n1 = fmaxf(m1[j], mx1);
                const float b0 = n0 == -INFINITY ? 0.f : n0, b1 = n1 == -INFINITY ? 0.f : n1;
                const float al0 = n0 == -INFINITY ? 1.f : fast_exp2(m0[j] - n0);
                const float al1 = n1 == -INFINITY ? 1.f : fast_exp2(m1[j] - n1);
                m0[j] = n0;
                m1[j] = n1;
                const float p0 = fast_exp2(sacc[j][0] - b0), p1 = fast_exp2(sacc[j][1] - b1);
                const float p2 = fast_exp2(sacc[j][2] - b0), p3 = fast_exp2(sacc[j][3] - b1);
                l0[j] = l0[j] * al0 + 256.f * (p0 + p2);
                l1[j] = l1[j] * al1 + 256.f * (p1 + p3);
                pb0[j] = movmatrix_t(pack_f16(p0 * w0, p1 * w0));
                pb1[j] = movmatrix_t(pack_f16(p2 * w1, p3 * w1));
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {  // a head's max moved
#pragma unroll
                    for (int dt = 0; dt < 8; ++dt) {
                        oacc[j][dt][0] *= al0;
                        oacc[j][dt][1] *= al1;
                        oacc[j][dt][2] *= al0;
                        oacc[j][dt][3] *= al1;
                    }
                }
            }
            // O^T += V^T P^T: A rows are d (two 16-row tiles per load), 4 key codes per 32-bit word
#pragma unroll
            for (int dp = 0; dp < 4; ++dp) {
                uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
                ldsm_x4(vb + swz64(dp * 32 + jj * 8 + (lane & 7), w * 16), r0, r1, r2, r3);
                e4m3x4_f16x2x2_cvt(__byte_perm(r0, 0u, vsel), a0, a2);
                e4m3x4_f16x2x2_cvt(__byte_perm(r1, 0u, vsel), a1, a3);
#pragma unroll
                for (int j = 0; j < kTok; ++j) mma_f16_16816(oacc[j][2 * dp], a0, a1, a2, a3, pb0[j], pb1[j]);
                e4m3x4_f16x2x2_cvt(__byte_perm(r2, 0u, vsel), a0, a2);
                e4m3x4_f16x2x2_cvt(__byte_perm(r3, 0u, vsel), a1, a3);
#pragma unroll
                for (int j = 0; j < kTok; ++j) mma_f16_16816(oacc[j][2 * dp + 1], a0, a1, a2, a3, pb0[j], pb1[j]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);

        if (d.flags & kLast) {
            const int h0 = 2 * qd, h1 = 2 * qd + 1;
            float t0[kTok], t1[kTok];
#pragma unroll
            for (int j = 0; j < kTok; ++j) {
                t0[j] = l0[j];
                t1[j] = l1[j];
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    t0[j] += __shfl_xor_sync(0xffffffffu, t0[j], off);
                    t1[j] += __shfl_xor_sync(0xffffffffu, t1[j], off);
                }
            }
            if (w > 0) {  // hand this warp's states to warp 0
#pragma unroll
                for (int j = 0; j < kTok; ++j) {
                    if (gr == 0) {
                        sm.mm[w - 1][j][h0] = m0[j];
                        sm.mm[w - 1][j][h1] = m1[j];
                        sm.ml[w - 1][j][h0] = t0[j];
                        sm.ml[w - 1][j][h1] = t1[j];
                    }
#pragma unroll
                    for (int dt = 0; dt < 8; ++dt) {
                        sm.mo[w - 1][j][h0][dt * 16 + gr] = oacc[j][dt][0];
                        sm.mo[w - 1][j][h1][dt * 16 + gr] = oacc[j][dt][1];
                        sm.mo[w - 1][j][h0][dt * 16 + gr + 8] = oacc[j][dt][2];
                        sm.mo[w - 1][j][h1][dt * 16 + gr + 8] = oacc[j][dt][3];
                    }
                }
            }
            ok = merge_sync(sm, merge_phase, a.err);
            if (w == 0 && ok) {
#pragma unroll
                for (int j = 0; j < kTok; ++j) {
                    float M0 = m0[j], M1 = m1[j];
                    for (int i = 0; i < kConsumers8 - 1; ++i) {
                        M0 = fmaxf(M0, sm.mm[i][j][h0]);
                        M1 = fmaxf(M1, sm.mm[i][j][h1]);
                    }
                    const float e0 = M0 == -INFINITY ? 0.f : fast_exp2(m0[j] - M0);
                    const float e1 = M1 == -INFINITY ? 0.f : fast_exp2(m1[j] - M1);
                    float L0 = t0[j] * e0, L1 = t1[j] * e1;
                    float(&acc)[8][4] = oacc[j];  // merged in place: a new piece starts from zero
#pragma unroll
                    for (int dt = 0; dt < 8; ++dt) {
                        acc[dt][0] *= e0;
                        acc[dt][1] *= e1;
                        acc[dt][2] *= e0;
                        acc[dt][3] *= e1;
                    }
                    for (int i = 0; i < kConsumers8 - 1; ++i) {
                        const float f0 = M0 == -INFINITY ? 0.f : fast_exp2(sm.mm[i][j][h0] - M0);
                        const float f1 = M1 == -INFINITY ? 0.f : fast_exp2(sm.mm[i][j][h1] - M1);
                        L0 += f0 * sm.ml[i][j][h0];
                        L1 += f1 * sm.ml[i][j][h1];
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) {
                            acc[dt][0] += f0 * sm.mo[i][j][h0][dt * 16 + gr];
                            acc[dt][1] += f1 * sm.mo[i][j][h1][dt * 16 + gr];
                            acc[dt][2] += f0 * sm.mo[i][j][h0][dt * 16 + gr + 8];
                            acc[dt][3] += f1 * sm.mo[i][j][h1][dt * 16 + gr + 8];
                        }
                    }
                    if (d.flags & kDirect) {
                        const float i0 = L0 > 0.f ? 1.f / L0 : 0.f, i1 = L1 > 0.f ? 1.f / L1 : 0.f;
                        __nv_bfloat16 *o0 = a.o + (q_row(a, d.seq, j) * a.hq + (int64_t)d.kvh * kG + h0) * kD;
                        __nv_bfloat16 *o1 = o0 + kD;
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) {
                            o0[dt * 16 + gr] = __float2bfloat16_rn(acc[dt][0] * i0);
                            o1[dt * 16 + gr] = __float2bfloat16_rn(acc[dt][1] * i1);
                            o0[dt * 16 + gr + 8] = __float2bfloat16_rn(acc[dt][2] * i0);
                            o1[dt * 16 + gr + 8] = __float2bfloat16_rn(acc[dt][3] * i1);
                        }
                    } else {
                        Partial &p = a.part[((int64_t)blockIdx.x * 2 + d.slot) * a.n_tok + j];
                        if (gr == 0) {
                            p.m[h0] = M0;
                            p.m[h1] = M1;
                            p.l[h0] = L0;
                            p.l[h1] = L1;
                        }
#pragma unroll
                        for (int dt = 0; dt < 8; ++dt) {
                            p.o[h0][dt * 16 + gr] = acc[dt][0];
                            p.o[h1][dt * 16 + gr] = acc[dt][1];
                            p.o[h0][dt * 16 + gr + 8] = acc[dt][2];
                            p.o[h1][dt * 16 + gr + 8] = acc[dt][3];
                        }
                    }
                }
            }
            ok = merge_sync(sm, merge_phase, a.err) && ok;  // the merge area is free again
            if (!ok) {
                if (lane == 0) sm.abort = 1;
                return;
            }
        }
        if (++stage == kStages) stage = 0, phase ^= 1;
    }
}

template <int kTok>
__global__ void __launch_bounds__(32 * (kConsumers8 + 1)) decode_mma_fp8_d128(const __grid_constant__ CUtensorMap tk,
                                                                           const __grid_constant__ CUtensorMap tv,
                                                                           DecodeArgs a) {
    using Smem = DecodeSmem8T<kTok>;
    extern __shared__ uint8_t raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    if (threadIdx.x == 0) {
        for (int i = 0; i < Smem::kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kConsumers8);
        }
        mbar_init(&sm.merge, 32 * kConsumers8);
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const int64_t U = a.sdesc[a.n_seqs].x, N = gridDim.x;
    if (U == 0) return;
    const int64_t u0 = cta_start(blockIdx.x, U, N), u1 = cta_start(blockIdx.x + 1, U, N);
    if (threadIdx.x >= 32 * kConsumers8)
        decode_producer<true>(sm, &tk, &tv, a, u0, u1);
    else
        decode_consumer_fp8<kTok>(sm, a, u0, u1);
}

// ------------------------------------------------ tensor-core multi-token
// Multi-token decode on the 5th-generation tensor cores. The n_tok query
// tokens x 8 query heads of a (sequence, kv head) are the rows of one
// M = 128 tile, so every streamed page costs the same two MMA groups:
//   S = Q K^T    8 x tcgen05.mma M128 N64 K16 (the page's 64 keys)
//   O += P V     4 x tcgen05.mma M128 N128 K16, P read from TMEM
// With 8 n_tok <= 128 / R the query rows are repeated R times (R = 4 up to
// 4 tokens, 2 up to 8, else 1): copy c of a row sees only keys
// [c 64 / R, (c + 1) 64 / R) of every page (its P is zero elsewhere) and
// keeps its own running max and sum, so the softmax of a page is spread
// over all four warps instead of one. At the end of a piece the copies of
// a row are merged (weights 2^(m_c - M)) through shared memory.
// TMEM (512 columns): S (up to 4 x 64), P (up to 4 x 32 packed pairs), O
// (128). Page i uses S and P buffer i % kSP; a page is ready to score only
// once PV(i - kSP) is done (below), so the buffers need no other wait.
// Warp 4 streams pages (and each piece's q tile by tensor map). Warp 5
// allocates TMEM and one of its threads issues the QK MMAs, one thread of
// warp 6 the PV MMAs: an MMA takes some 70 cycles to issue and a barrier
// wait after a commit several times that, too much for one thread per page.
// The scores of page i + 1 run on the tensor cores while the softmax of
// page i runs. Warps 0-3: one tile row per thread: mask (only on pages a
// token does not see whole), online softmax in the log2 domain with the
// lazy 2^8 rescale of O, P to TMEM, and the end-of-piece merge and output.
//
// FP8 pools: warps 7-10 convert each E4M3 page into f16 K and V^T tiles
// (every E4M3 value is an f16 value) and the piece's q tile from bf16 to
// f16. With copies (R > 1) q goes into TMEM as f16 pairs (columns 192-255,
// free with 3 S buffers) and the QK MMAs read it from there as their A
// operand, which spares the shared memory the q reads of every page; with
// R = 1, where the softmax bounds the kernel, q stays in shared memory,
// converted in place (measured: TMEM q is 4-8 % faster up to 8 tokens and
// 5-7 % slower at 16). The MMAs run on f16 operands; the softmax multiplies
// the scores by the per-key K scale and P by the per-key V scale.
constexpr int kTcCols = 512;
constexpr uint32_t kTmemP = 256, kTmemO = 384;  // column offsets of P and O (S at 0)
constexpr uint32_t kTmemQ = 192;                // FP8 pools: the q tile, 64 columns of f16 pairs
constexpr float kTcRescaleLog2 = 8.0f;          // rescale O only when the max grows by > 2^8

// bf16 pools: page i is ready to score once its stage has landed, which
// the producer only loads after PV(i - 4) emptied it.
struct DecodeTcSmem {
    static constexpr bool kFP8 = false;
    static constexpr int kStages = 4;
    static constexpr int kSP = kStages;  // S / P buffers
    static constexpr int kQBufs = 2;
    static constexpr bool kTcQ = true;
    static constexpr bool kQTmem = false;  // QK reads q from shared memory
    static constexpr int kThreads = 224;
    static constexpr uint32_t kQHalfBytes = 128 * 128;  // 128 rows x 64 columns of 16-bit values
    uint8_t k[kStages][kPageHeadBytes];                // [d half][64 keys][128 B], 128-byte swizzle
    uint8_t v[kStages][kPageHeadBytes];
    uint8_t q[kQBufs][2 * kQHalfBytes];                // [d half][128 rows][128 B]
    float obuf[kD][32];                                // merge: one 32-row block of O, column-major
    float ep_m[128], ep_l[128];                        // merge: (max, sum) of every tile row
    StageDesc desc[kStages];
    uint64_t full[kStages], empty[kStages];
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[kSP], p_full[kSP];
    uint64_t mma_done[2], ep_bar;
    uint32_t tmem_base;
    int32_t abort;

    __device__ uint64_t *ready(int64_t i) { return &full[i % kStages]; }   // page i can be scored
    __device__ uint64_t *pv_done(int64_t i) { return &empty[i % kStages]; }  // PV(i) has completed
    static __device__ uint32_t par(int64_t i) { return (uint32_t)(i / kStages) & 1; }
    __device__ const StageDesc &page(int64_t i) const { return desc[i % kStages]; }
    __device__ uint64_t *q_ready(int32_t pc) { return &q_full[pc % kQBufs]; }
    __device__ uint32_t k_addr(int64_t i) { return smem_u32(k[i % kStages]); }
    __device__ uint32_t v_addr(int64_t i) { return smem_u32(v[i % kStages]); }
};
static_assert(offsetof(DecodeTcSmem, v) % 1024 == 0 && offsetof(DecodeTcSmem, q) % 1024 == 0,
              "128-byte swizzled tiles need 1024-byte alignment");

// FP8 pools: E4M3 pages land in 4 stages; the converter warps turn page i
// into f16 buffer i % 3 once PV(i - 3) has emptied it, so page i is ready
// to score when its conversion is done.
struct DecodeTc8Smem {
    static constexpr bool kFP8 = true;
    static constexpr int kStages = 4;
    static constexpr int kConv = 3;
    static constexpr int kSP = kConv;
    static constexpr int kQBufs = 1;
    static constexpr bool kTcQ = true;
    static constexpr bool kQTmem = true;  // with copies (R > 1) QK reads q from TMEM column kTmemQ
    static constexpr int kConvThreads = 128;  // converter warps 7 ..
    static constexpr int kThreads = 224 + kConvThreads;
    static constexpr uint32_t kQHalfBytes = 128 * 128;
    uint8_t k[kStages][kK8Bytes];   // E4M3 [64 keys][128 B], 128-byte swizzle
    uint8_t v[kStages][kV8Bytes];   // E4M3 V^T [128 d][64 B], 64-byte swizzle
    uint8_t q[kQBufs][2 * kQHalfBytes];
    uint8_t kc[kConv][kPageHeadBytes];  // f16 K [d half][64 keys][128 B], 128-byte swizzle
    uint8_t vc[kConv][kD * 128];        // f16 V^T [128 d][64 keys = 128 B], 128-byte swizzle
    float ks[kStages][kP], vs[kStages][kP];
    float ksc[kConv][kP], vsc[kConv][kP];  // ksc: the K scale times scale log2 e
    float obuf[kD][32];
    float ep_m[128], ep_l[128];
    StageDesc desc[kStages];
    StageDesc descc[kConv];
    uint64_t full[kStages], empty[kStages];
    uint64_t conv_full[kConv], conv_empty[kConv];
    uint64_t q_full[2], q_empty[2], q_conv[2];
    uint64_t s_full[kSP], p_full[kSP];
    uint64_t mma_done[2], ep_bar;
    uint32_t tmem_base;
    int32_t abort;

    __device__ uint64_t *ready(int64_t i) { return &conv_full[i % kConv]; }
    __device__ uint64_t *pv_done(int64_t i) { return &conv_empty[i % kConv]; }
    static __device__ uint32_t par(int64_t i) { return (uint32_t)(i / kConv) & 1; }
    __device__ const StageDesc &page(int64_t i) const { return descc[i % kConv]; }
    __device__ uint64_t *q_ready(int32_t pc) { return &q_conv[pc % kQBufs]; }
    __device__ uint32_t k_addr(int64_t i) { return smem_u32(kc[i % kConv]); }
    __device__ uint32_t v_addr(int64_t i) { return smem_u32(vc[i % kConv]); }
};
static_assert(offsetof(DecodeTc8Smem, ksc) % 16 == 0 && offsetof(DecodeTc8Smem, vsc) % 16 == 0,
              "the softmax reads the scales 4 at a time");
static_assert(DecodeTc8Smem::kSP * 64 <= (int)kTmemQ && kTmemQ + 64 <= kTmemP, "q sits between S and P in TMEM");
static_assert(offsetof(DecodeTc8Smem, q) % 1024 == 0 && offsetof(DecodeTc8Smem, kc) % 1024 == 0 &&
                  offsetof(DecodeTc8Smem, vc) % 1024 == 0,
              "128-byte swizzled tiles need 1024-byte alignment");

template <class Smem>
constexpr size_t decode_tc_smem_bytes() { return sizeof(Smem) + 1024; }

// Two threads issue the MMAs of the CTA's n pages, each in page order and
// each waiting only on its own barriers:
//   warp 5, lane 0: QK(i) into S buffer i % kSP once page i is ready (and,
//     on a piece's first page, its q tile); commits s_full, and q_empty after
//     the last QK of a piece (the q tile, in shared memory or TMEM, is then
//     free for the next piece);
//   warp 6, lane 0: PV(i) once P(i) is in TMEM; commits pv_done(i) (the
//     bf16 stage, or the FP8 pool's f16 buffer: K was read by QK(i) before
//     P(i) existed).
// A commit arrives once every MMA its thread issued before has completed.
// Page i is ready only after PV(i - kSP), and with it the softmax of page
// i - kSP, are done, so S and P buffer i % kSP are free. The s_full and
// p_full barriers are per buffer: each is at most one phase ahead of a
// waiter for the same reason.
template <bool kQT, class Smem>
__device__ bool decode_tc_qk(Smem &sm, const DecodeArgs &a, int64_t n) {
    constexpr int kSP = Smem::kSP, kQB = Smem::kQBufs;
    constexpr uint32_t kIdQK = idesc_16(128, kP, false, Smem::kFP8);
    const uint32_t tb = sm.tmem_base, qb = smem_u32(sm.q[0]);
    int32_t pc = -1;  // piece of the last scored page
    for (int64_t i = 0; i < n; ++i) {
        if (!mbar_wait(sm.ready(i), Smem::par(i), a.err)) return false;
        const int32_t flags = sm.page(i).flags;
        if (flags & kFirst) {
            ++pc;
            if (!mbar_wait(sm.q_ready(pc), (uint32_t)(pc / kQB) & 1, a.err)) return false;
        }
        if (*(volatile int32_t *)&sm.abort) return false;
        tc_fence_after();
        if (!(flags & kSkip)) {
            // descriptors of the tiles' first bytes; a step adds its byte
            // offset / 16 to the address field (shared memory < 2^18 bytes:
            // no carry out of it)
            const uint64_t qd = sdesc(qb + (pc % kQB) * 2 * Smem::kQHalfBytes, 16, 1024);
            const uint64_t kd = sdesc(sm.k_addr(i), 16, 1024);
            const uint32_t ts = tb + 64 * (uint32_t)(i % kSP);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
                if constexpr (kQT)  // d 16 kk .. 16 kk + 15 are columns 8 kk .. 8 kk + 7
                    mma_ts(ts, tb + kTmemQ + 8 * kk, kd + koff, kIdQK, kk > 0);
                else
                    mma_ss(ts, qd + (((kk >> 2) * Smem::kQHalfBytes + (kk & 3) * 32) >> 4), kd + koff, kIdQK, kk > 0);
            }
        }
        mma_commit(&sm.s_full[i % kSP]);
        if (flags & kLast) mma_commit(&sm.q_empty[pc % kQB]);
    }
    return true;
}

template <class Smem>
__device__ bool decode_tc_pv(Smem &sm, const DecodeArgs &a, int64_t n) {
    constexpr int kSP = Smem::kSP;
    // bf16: V as loaded, [keys][d] (d contiguous: MN-major B, d halves 8 KB
    // apart); FP8: the converted V^T, [d][keys] (keys contiguous: K-major)
    constexpr uint32_t kIdPV = idesc_16(128, kD, !Smem::kFP8, Smem::kFP8);
    const uint32_t tb = sm.tmem_base;
    bool fresh = true;  // no PV yet in the current piece: the next one overwrites O
    for (int64_t i = 0; i < n; ++i) {
        const int b = (int)(i % kSP);
        if (!mbar_wait(&sm.p_full[b], (uint32_t)(i / kSP) & 1, a.err) || *(volatile int32_t *)&sm.abort)
            return false;
        const int32_t flags = sm.page(i).flags;
        if (flags & kFirst) fresh = true;
        tc_fence_after();
        if (!(flags & kSkip)) {
            const uint32_t tp = tb + kTmemP + 32 * b, v = sm.v_addr(i);
            const uint64_t vd = Smem::kFP8 ? sdesc(v, 16, 1024) : sdesc(v, kBoxBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 16 keys a step: 32 bytes on (FP8 V^T rows) or 16 rows of 128 B
                mma_ts(tb + kTmemO, tp + kk * 8, vd + (Smem::kFP8 ? kk * (32 >> 4) : kk * (2048 >> 4)), kIdPV,
                       (fresh && kk == 0) ? 0u : 1u);
            fresh = false;
        }
        mma_commit(sm.pv_done(i));
    }
    return true;
}

// Run one issuer role, then make sure every MMA it issued has completed
// before TMEM is freed.
template <bool kQK, bool kQT, class Smem>
__device__ void decode_tc_issue(Smem &sm, const DecodeArgs &a, int64_t n) {
    bool ok = kQK ? decode_tc_qk<kQT>(sm, a, n) : decode_tc_pv(sm, a, n);
    mma_commit(&sm.mma_done[kQK ? 0 : 1]);
    if (!mbar_wait(&sm.mma_done[kQK ? 0 : 1], 0, a.err)) ok = false;
    if (!ok) sm.abort = 1;
}

// S columns [col, col + kN) of this thread's lane.
template <int kN>
__device__ __forceinline__ void tmem_ld_s(uint32_t taddr, uint32_t (&r)[kN]) {
    if constexpr (kN == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
            "%14, %15}, [%16];"
            : HSWA_R8(0), HSWA_R8(8)
            : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" : HSWA_RW8(0), HSWA_RW8(8)::"memory");
    } else {
#pragma unroll
        for (int c = 0; c < kN / 32; ++c) tmem_ld32(taddr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
#pragma unroll
        for (int c = 0; c < kN / 32; ++c) tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
    }
}

// kN packed P columns of this thread's lane.
template <int kN>
__device__ __forceinline__ void tmem_st_p(uint32_t taddr, const uint32_t (&r)[kN]) {
    if constexpr (kN == 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                     HSWA_W8(0)
                     : "memory");
    } else {
#pragma unroll
        for (int c = 0; c < kN / 16; ++c) tmem_st16(taddr + 16 * c, r + 16 * c);
    }
}

// Bounded arrival + wait on the softmax warps' own barrier (128 threads).
template <class Smem>
__device__ __forceinline__ bool ep_sync(Smem &sm, uint32_t &phase, int *err) {
    mbar_arrive(&sm.ep_bar);
    const bool ok = mbar_wait(&sm.ep_bar, phase, err);
    phase ^= 1;
    return ok;
}

template <int kR, class Smem>
__device__ void decode_tc_softmax(Smem &sm, const DecodeArgs &a, int64_t n) {
    constexpr int kSP = Smem::kSP;
    constexpr int kRows = 128 / kR;  // tile rows per copy
    constexpr int kK = kP / kR;      // keys of a page per copy
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = threadIdx.x, c = r / kRows, j = r % kRows;
    const int w = j >> 3, h = j & 7;
    const bool active = (((warp * 32) % kRows) >> 3) < a.n_tok;  // uniform over the warp
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_o = sm.tmem_base + lane_off + kTmemO;
    const uint32_t t_p = sm.tmem_base + lane_off + kTmemP + c * (kK / 2);
    if constexpr (kR > 1) {
        // P outside this copy's keys stays zero; the copy's own columns are
        // rewritten on every page
        uint32_t z[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) z[x] = 0u;
#pragma unroll
        for (int b = 0; b < kSP; ++b) tmem_st32(sm.tmem_base + lane_off + kTmemP + 32 * b, z);
        tmem_wait_st();
    }
    float m_used = -INFINITY, l = 0.f;  // reference max (log2 units) and sum of P
    uint32_t ep_phase = 0;
    bool ok = true;
    for (int64_t i = 0; i < n && ok; ++i) {
        const int b = (int)(i % kSP);  // S / P buffer
        ok = mbar_wait(sm.ready(i), Smem::par(i), a.err) &&
             mbar_wait(&sm.s_full[b], (uint32_t)(i / kSP) & 1, a.err) && !*(volatile int32_t *)&sm.abort;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const StageDesc d = sm.page(i);
        if (d.flags & kFirst) m_used = -INFINITY, l = 0.f;
        if (active) {
            tc_fence_after();
            uint32_t sr[kK];
            tmem_ld_s<kK>(sm.tmem_base + lane_off + 64 * b + c * kK, sr);
            if constexpr (Smem::kFP8) {
                // the K codes entered the MMA as their exact values: a score
                // in log2 units is S times the key's scale times scale log2 e,
                // a product the converter stored per key
                const float4 *ks = reinterpret_cast<const float4 *>(sm.ksc[i % Smem::kConv] + c * kK);
#pragma unroll
                for (int x = 0; x < kK / 4; ++x) {
                    const float4 k4 = ks[x];
                    const float2 lo = __fmul2_rn(make_float2(__uint_as_float(sr[4 * x]), __uint_as_float(sr[4 * x + 1])),
                                                 make_float2(k4.x, k4.y));
                    const float2 hi = __fmul2_rn(
                        make_float2(__uint_as_float(sr[4 * x + 2]), __uint_as_float(sr[4 * x + 3])), make_float2(k4.z, k4.w));
                    sr[4 * x] = __float_as_uint(lo.x), sr[4 * x + 1] = __float_as_uint(lo.y);
                    sr[4 * x + 2] = __float_as_uint(hi.x), sr[4 * x + 3] = __float_as_uint(hi.y);
                }
            }
            // keys of the page this row's token sees, relative to the copy's
            // first key: [lo_c, hi_c) (position t = len - n_tok + w; W keys
            // ending at t for SWA)
            const int32_t t = d.len - a.n_tok + w;
            const int32_t base = d.key0 + c * kK;
            int32_t hi_c = min(d.hi - c * kK, t - base + 1), lo_c = d.lo - c * kK;
            if (a.window > 0) lo_c = max(lo_c, t - a.window + 1 - base);
            if (w >= a.n_tok || (d.flags & kSkip)) hi_c = 0;
            float m0 = -INFINITY, m1 = -INFINITY;
            // most pages are seen whole by every token of the warp
            if (__any_sync(0xffffffffu, lo_c > 0 || hi_c < kK)) {
#pragma unroll
                for (int x = 0; x < kK; ++x)
                    if (x >= hi_c || x < lo_c) sr[x] = __float_as_uint(-INFINITY);
            }
#pragma unroll
            for (int x = 0; x < kK; x += 4) {
                m0 = max3(m0, __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]));
                m1 = max3(m1, __uint_as_float(sr[x + 2]), __uint_as_float(sr[x + 3]));
            }
            const float mx = Smem::kFP8 ? fmaxf(m0, m1) : fmaxf(m0, m1) * a.scale_log2;
            const bool need = mx > m_used + kTcRescaleLog2;
            const bool resc = need && m_used != -INFINITY;
            const float alpha = resc ? fast_exp2(m_used - mx) : 1.f;
            if (need) m_used = mx;
            const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
            const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(neg_m, neg_m);
            float2 sum2 = make_float2(0.f, 0.f);
            uint32_t pk[kK / 2];
#pragma unroll
            for (int x = 0; x < kK / 2; ++x) {
                const float2 sx = make_float2(__uint_as_float(sr[2 * x]), __uint_as_float(sr[2 * x + 1]));
                const float2 y = Smem::kFP8 ? __fadd2_rn(sx, nm2) : __ffma2_rn(sx, sc2, nm2);
                const float2 p = make_float2(fast_exp2(y.x), fast_exp2(y.y));
                sum2 = __fadd2_rn(sum2, p);
                if constexpr (Smem::kFP8) {  // P carries the V scale: V codes enter the MMA as they are
                    const float4 v4 = reinterpret_cast<const float4 *>(sm.vsc[i % Smem::kConv] + c * kK)[x >> 1];
                    const float2 pv = __fmul2_rn(p, (x & 1) ? make_float2(v4.z, v4.w) : make_float2(v4.x, v4.y));
                    pk[x] = pack_f16(pv.x, pv.y);
                } else {
                    pk[x] = pack_bf16(p.x, p.y);
                }
            }
            tmem_st_p<kK / 2>(t_p + 32 * b, pk);  // P buffer i % kSP: free since page i is ready
            if (__any_sync(0xffffffffu, resc)) {  // never on a piece's first page
                // O holds the piece's earlier pages once PV(i - 1) is done
                // (its pv_done barrier's next phase needs P(i - 1 + kSP);
                // PV(i - 1 - kSP) is done since page i - 1 was ready)
                ok = __all_sync(0xffffffffu, mbar_wait(sm.pv_done(i - 1), Smem::par(i - 1), a.err));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t ov[32];
                    tmem_ld32(t_o + 32 * cc, ov);
                    tmem_wait_ld(ov);
#pragma unroll
                    for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * alpha);
                    tmem_st32(t_o + 32 * cc, ov);
                }
            }
            l = l * alpha + (sum2.x + sum2.y);
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&sm.p_full[b]);
        if (!(d.flags & kLast)) continue;
        // ---- end of the piece: O is final once PV(i) is done, the next
        // phase of its pv_done barrier (PV(i - kSP) is done since page i was
        // ready; PV(i + kSP) needs P(i + kSP))
        if (active) ok = __all_sync(0xffffffffu, mbar_wait(sm.pv_done(i), Smem::par(i), a.err));
        float M = m_used, L = l, wt = 1.f;
        if constexpr (kR > 1) {
            // merge the copies of each row: weights 2^(m_c - M); copy 0 adds
            // the other copies' weighted rows into its own, 32 rows at a time
            sm.ep_m[r] = m_used;
            sm.ep_l[r] = l;
            ok = ep_sync(sm, ep_phase, a.err) && ok;
            M = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < kR; ++cc) M = fmaxf(M, sm.ep_m[cc * kRows + j]);
            L = 0.f;
#pragma unroll
            for (int cc = 0; cc < kR; ++cc) {
                const float mc = sm.ep_m[cc * kRows + j];
                L += mc == -INFINITY ? 0.f : fast_exp2(mc - M) * sm.ep_l[cc * kRows + j];
            }
            wt = m_used == -INFINITY ? 0.f : fast_exp2(m_used - M);
            tc_fence_after();
#pragma unroll 1
            for (int cc = 1; cc < kR; ++cc) {
#pragma unroll 1
                for (int b = 0; b < kRows / 32; ++b) {
                    if (active && ok && warp == (cc * kRows) / 32 + b) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t ov[32];
                            tmem_ld32(t_o + 32 * q4, ov);
                            tmem_wait_ld(ov);
#pragma unroll
                            for (int x = 0; x < 32; ++x) sm.obuf[32 * q4 + x][lane] = __uint_as_float(ov[x]) * wt;
                        }
                    }
                    ok = ep_sync(sm, ep_phase, a.err) && ok;
                    if (active && ok && warp == b) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t ov[32];
                            tmem_ld32(t_o + 32 * q4, ov);
                            tmem_wait_ld(ov);
                            const float own = cc == 1 ? wt : 1.f;  // copy 0's own weight, applied once
#pragma unroll
                            for (int x = 0; x < 32; ++x)
                                ov[x] = __float_as_uint(__uint_as_float(ov[x]) * own + sm.obuf[32 * q4 + x][lane]);
                            tmem_st32(t_o + 32 * q4, ov);
                        }
                        tmem_wait_st();
                    }
                    ok = ep_sync(sm, ep_phase, a.err) && ok;
                }
            }
            wt = 1.f;
        }
        if (!ok) break;
        if (!active || c != 0) continue;
        tc_fence_after();
        const bool row = w < a.n_tok;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        if (d.flags & kDirect) {
            uint4 *dst = reinterpret_cast<uint4 *>(
                a.o + (q_row(a, d.seq, row ? w : 0) * a.hq + (int64_t)d.kvh * kG + h) * kD);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t ov[32];
                tmem_ld32(t_o + 32 * q4, ov);
                tmem_wait_ld(ov);
                if (row) {
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        // L = 0: no key seen, write zeros (O may be unset)
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = L > 0.f ? __uint_as_float(ov[8 * x + e]) * inv : 0.f;
                        dst[q4 * 4 + x] = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                                     pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
                    }
                }
            }
        } else {
            Partial &p = a.part[((int64_t)blockIdx.x * 2 + d.slot) * a.n_tok + (row ? w : 0)];
            float4 *dst = reinterpret_cast<float4 *>(p.o[h]);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t ov[32];
                tmem_ld32(t_o + 32 * q4, ov);
                tmem_wait_ld(ov);
                if (row) {
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        float f[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) f[e] = L > 0.f ? __uint_as_float(ov[4 * x + e]) : 0.f;
                        dst[q4 * 8 + x] = make_float4(f[0], f[1], f[2], f[3]);
                    }
                }
            }
            if (row) {
                p.m[h] = M;
                p.l[h] = L;
            }
        }
    }
    if (!ok) sm.abort = 1;
}


// Eight bf16 (one 16-byte chunk) to f16 in place, clamped to f16's finite range.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float lo = fminf(fmaxf(__uint_as_float(w[e] << 16), -65504.f), 65504.f);
        const float hi = fminf(fmaxf(__uint_as_float(w[e] & 0xFFFF0000u), -65504.f), 65504.f);
        w[e] = pack_f16(lo, hi);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Sixteen E4M3 codes (one 16-byte chunk) as sixteen exact f16 values.
__device__ __forceinline__ void e4m3x16_to_f16(uint4 c, uint4 &lo, uint4 &hi) {
    e4m3x4_f16x2x2_cvt(c.x, lo.x, lo.y);
    e4m3x4_f16x2x2_cvt(c.y, lo.z, lo.w);
    e4m3x4_f16x2x2_cvt(c.z, hi.x, hi.y);
    e4m3x4_f16x2x2_cvt(c.w, hi.z, hi.w);
}

// Warps 7-10 (FP8 pools): page i's E4M3 stage to f16 buffer i % kConv, once
// PV(i - kConv) has emptied it (the f16 buffer's pv_done barrier, waited for
// on every page, so it is never two phases ahead). K [64 keys][128 B]
// becomes [d half][64 keys][128 B] and V^T [128 d][64 B] becomes
// [128 d][128 B], both with the 128-byte swizzle; the scales and the
// stage's descriptor are copied along.
// On a piece's first page the piece's q tile is converted first: with kQT
// into TMEM, where thread (warp w, lane l) writes tile row 32 (w mod 4) + l,
// the lanes its warp may reach, as 64 columns of f16 pairs (the producer
// loads that q tile only after the last QK of the previous piece, q_empty,
// so the TMEM columns are free by the time it lands); else in place in
// shared memory. Then the stage is released to the producer.
template <bool kQT>
__device__ void decode_tc_convert(DecodeTc8Smem &sm, const DecodeArgs &a, int64_t n) {
    constexpr int kStages = DecodeTc8Smem::kStages, kConv = DecodeTc8Smem::kConv, kQB = DecodeTc8Smem::kQBufs;
    constexpr int kCT = DecodeTc8Smem::kConvThreads, kPer = 512 / kCT;  // 16-byte chunks per thread and tile
    constexpr uint32_t kQH = DecodeTc8Smem::kQHalfBytes;
    const int t = threadIdx.x - 7 * 32;  // 0 .. kCT - 1
    const int quad = (threadIdx.x >> 5) & 3, row = 32 * quad + (threadIdx.x & 31);
    const uint32_t t_q = sm.tmem_base + ((uint32_t)(32 * quad) << 16) + kTmemQ;
    int32_t pc = -1;
    bool ok = true;
    for (int64_t i = 0; i < n && ok; ++i) {
        const int st = (int)(i % kStages), b = (int)(i % kConv);
        ok = mbar_wait(&sm.full[st], (uint32_t)(i / kStages) & 1, a.err) &&
             (i < kConv || mbar_wait(&sm.conv_empty[b], (uint32_t)((i - kConv) / kConv) & 1, a.err)) &&
             !*(volatile int32_t *)&sm.abort;
        const StageDesc d = sm.desc[st];
        if (ok && (d.flags & kFirst)) {
            ++pc;
            ok = mbar_wait(&sm.q_full[pc % kQB], (uint32_t)(pc / kQB) & 1, a.err);
        }
        // the TMEM stores below are warp-wide: the warp goes on or stops as one
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if ((d.flags & kFirst) && !kQT) {  // f16 in place, for QK from shared memory
            uint4 *q = reinterpret_cast<uint4 *>(sm.q[pc % kQB]);
#pragma unroll 4
            for (int x = t; x < 2 * (int)DecodeTc8Smem::kQHalfBytes / 16; x += kCT) q[x] = bf16x8_to_f16x8(q[x]);
            fence_proxy_async_shared();
            mbar_arrive(&sm.q_conv[pc % kQB]);
        } else if (d.flags & kFirst) {  // f16 pairs into TMEM
            const uint8_t *q = sm.q[pc % kQB] + row * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // d half h: columns 32 h .. 32 h + 31
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 f = bf16x8_to_f16x8(*reinterpret_cast<const uint4 *>(q + h * kQH + ((c ^ (row & 7)) << 4)));
                    w[4 * c] = f.x, w[4 * c + 1] = f.y, w[4 * c + 2] = f.z, w[4 * c + 3] = f.w;
                }
                tmem_st32(t_q + 32 * h, w);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.q_conv[pc % kQB]);
        }
        if (!(d.flags & kSkip)) {
            const uint8_t *k8 = sm.k[st], *v8 = sm.v[st];
            uint8_t *kc = sm.kc[b], *vc = sm.vc[b];
            // all eight loads first: the stores below could alias them as far
            // as the compiler can tell, and would otherwise serialise them
            uint4 kin[kPer], vin[kPer];
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int x = t + kCT * e;
                const int r = x >> 3, c8 = x & 7;    // K: row r (key), chunk c8 (d 16 c8 .. 16 c8 + 15)
                const int dd = x >> 2, c4 = x & 3;   // V^T: row dd (d), chunk c4 (keys 16 c4 .. 16 c4 + 15)
                kin[e] = *reinterpret_cast<const uint4 *>(k8 + r * 128 + ((c8 ^ (r & 7)) << 4));
                vin[e] = *reinterpret_cast<const uint4 *>(v8 + dd * 64 + ((c4 ^ ((dd >> 1) & 3)) << 4));
            }
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int x = t + kCT * e;
                const int r = x >> 3, c8 = x & 7, dd = x >> 2, c4 = x & 3;
                uint4 lo, hi;
                // K: chunks j0 and j0 + 1 of the row in d half c8 / 4. The eight
                // threads of a quarter warp share the row; the four in the
                // second d half (8 KB on: the same banks) store the upper chunk
                // first, so each store instruction meets 8 distinct chunks
                const bool sw = (c8 & 4) != 0;
                const uint4 kq = sw ? make_uint4(kin[e].z, kin[e].w, kin[e].x, kin[e].y) : kin[e];
                e4m3x16_to_f16(kq, lo, hi);
                uint8_t *krow = kc + (c8 >> 2) * kBoxBytes + r * 128;
                const int j0 = 2 * (c8 & 3) + (sw ? 1 : 0), j1 = j0 ^ 1;
                *reinterpret_cast<uint4 *>(krow + ((j0 ^ (r & 7)) << 4)) = lo;
                *reinterpret_cast<uint4 *>(krow + ((j1 ^ (r & 7)) << 4)) = hi;
                e4m3x16_to_f16(vin[e], lo, hi);
                uint8_t *vrow = vc + dd * 128;
                *reinterpret_cast<uint4 *>(vrow + (((2 * c4) ^ (dd & 7)) << 4)) = lo;
                *reinterpret_cast<uint4 *>(vrow + (((2 * c4 + 1) ^ (dd & 7)) << 4)) = hi;
            }
        }
        if (t < kP)
            sm.ksc[b][t] = sm.ks[st][t] * a.scale_log2;
        else if (t < 2 * kP)
            sm.vsc[b][t - kP] = sm.vs[st][t - kP];
        if (t == 0) sm.descc[b] = d;
        fence_proxy_async_shared();  // the f16 tiles are read by the tensor cores
        mbar_arrive(&sm.conv_full[b]);
        mbar_arrive(&sm.empty[st]);
    }
    if (!ok) sm.abort = 1;
}

template <int kR, class Smem>
__global__ void __launch_bounds__(Smem::kThreads, 1)
    decode_tc_d128(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, DecodeArgs a) {
    extern __shared__ uint8_t raw[];
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < Smem::kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            // bf16: the PV thread's commit; FP8: the 128 converter threads
            mbar_init(&sm.empty[i], Smem::kFP8 ? Smem::kThreads - 224 : 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.q_full[b], 1);
            mbar_init(&sm.q_empty[b], 1);
        }
        for (int b = 0; b < Smem::kSP; ++b) {
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_full[b], 128);
        }
        if constexpr (Smem::kFP8) {
            for (int b = 0; b < Smem::kConv; ++b) {
                mbar_init(&sm.conv_full[b], Smem::kThreads - 224);
                mbar_init(&sm.conv_empty[b], 1);
            }
            for (int b = 0; b < 2; ++b) mbar_init(&sm.q_conv[b], Smem::kThreads - 224);
        }
        mbar_init(&sm.mma_done[0], 1);
        mbar_init(&sm.mma_done[1], 1);
        mbar_init(&sm.ep_bar, 128);
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 5) tmem_alloc<kTcCols>(&sm.tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // the plan (and the table update before it) is complete
    pdl_launch_dependents();
    const int64_t U = a.sdesc[a.n_seqs].x, N = gridDim.x;
    const int64_t u0 = cta_start(blockIdx.x, U, N), u1 = cta_start(blockIdx.x + 1, U, N);
    if (warp < 4) {
        decode_tc_softmax<kR>(sm, a, u1 - u0);
    } else if (warp == 4) {
        decode_producer<Smem::kFP8>(sm, &tk, &tv, a, u0, u1, &tq);
    } else if (warp < 7) {
        if ((threadIdx.x & 31) == 0) {
            if (warp == 5)
                decode_tc_issue<true, Smem::kQTmem && (kR > 1)>(sm, a, u1 - u0);
            else
                decode_tc_issue<false, false>(sm, a, u1 - u0);
        }
        __syncwarp();
    } else if constexpr (Smem::kFP8) {
        decode_tc_convert<Smem::kQTmem && (kR > 1)>(sm, a, u1 - u0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_free<kTcCols>(sm.tmem_base);
}

// Merge the partial records of segments split between CTAs; write zeros
// for sequences without keys.
__global__ void __launch_bounds__(256) decode_combine(DecodeArgs a, int32_t n_ctas) {
    const int32_t s = blockIdx.y / a.n_tok, w = blockIdx.y % a.n_tok, g = blockIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t U = a.sdesc[a.n_seqs].x, N = n_ctas;
    const int4 d = a.sdesc[s];
    const int32_t units = d.w;
    const int h = threadIdx.x >> 5, d0 = (threadIdx.x & 31) * 4;
    __nv_bfloat16 *out = a.o + (q_row(a, s, w) * a.hq + (int64_t)g * kG + h) * kD + d0;
    if (units == 0) {
        for (int i = 0; i < 4; ++i) out[i] = __float2bfloat16_rn(0.f);
        return;
    }
    const int32_t npg = units / a.hkv;
    const int64_t lo = d.x + (int64_t)g * npg, hi = lo + npg;  // [lo, hi)
    const int64_t c_lo = cta_of(lo, U, N), c_hi = cta_of(hi - 1, U, N);
    if (c_lo == c_hi) return;
    float M = -INFINITY;
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        if (cta_start(c, U, N) == cta_start(c + 1, U, N)) continue;
        const int slot = (c == c_lo && cta_start(c, U, N) < lo) ? 1 : 0;
        M = fmaxf(M, a.part[(c * 2 + slot) * a.n_tok + w].m[h]);
    }
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        if (cta_start(c, U, N) == cta_start(c + 1, U, N)) continue;
        const int slot = (c == c_lo && cta_start(c, U, N) < lo) ? 1 : 0;
        const Partial &p = a.part[(c * 2 + slot) * a.n_tok + w];
        const float wt = p.m[h] == -INFINITY ? 0.f : fast_exp2(p.m[h] - M);
        L += wt * p.l[h];
        for (int i = 0; i < 4; ++i) acc[i] += wt * p.o[h][d0 + i];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int i = 0; i < 4; ++i) out[i] = __float2bfloat16_rn(acc[i] * inv);
}

// ----------------------------------------------------------- generic path
template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

}  // namespace

// One warp per (query row, query head): query position t, keys [lo, t].
// mode 0: decode, n_rows = sequences x n_tok (row i is token i mod n_tok of
//         sequence i / n_tok, t = L - n_tok + i mod n_tok);
// mode 1: prefill, n_rows = max rows per sequence; row r < n_s of sequence s
//         is q row q_start[s] + r at t = prefix[s] + r.
template <typename T, int MAXE>
__global__ void attention_generic(const T *__restrict__ q, T *__restrict__ o, const T *__restrict__ kp,
                                  const T *__restrict__ vp, const int32_t *__restrict__ bt,
                                  const int32_t *__restrict__ seq_len, const int32_t *__restrict__ prefix,
                                  const int32_t *__restrict__ q_start, int32_t n_rows, int32_t n_seqs,
                                  int32_t bt_stride, int32_t hq, int32_t hkv, int32_t d, int32_t page,
                                  int32_t window, int32_t num_pages, float scale, int mode, int32_t n_tok,
                                  int *err) {
    const int lane = threadIdx.x & 31;
    const int64_t wid = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t per_seq = mode == 0 ? hq : (int64_t)n_rows * hq;
    if (wid >= per_seq * (mode == 0 ? n_rows : n_seqs)) return;
    const int32_t h = (int32_t)(wid % hq);
    const int32_t g = (int32_t)((int64_t)h * hkv / hq);
    int32_t s, t, row;
    if (mode == 0) {
        row = (int32_t)(wid / hq);
        s = row / n_tok;
        t = seq_len[s] - n_tok + row % n_tok;
    } else {
        s = (int32_t)(wid / per_seq);
        const int32_t r = (int32_t)((wid / hq) % n_rows);
        if (r >= q_start[s + 1] - q_start[s]) return;
        row = q_start[s] + r;
        t = prefix[s] + r;
    }
    float qv[MAXE], acc[MAXE];
    const int ne = (d + 31) / 32;
    const T *qrow = q + ((int64_t)row * hq + h) * d;
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        qv[e] = (e < ne && c < d) ? to_f(qrow[c]) * scale : 0.f;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int32_t lo = (window > 0 && t - window + 1 > 0) ? t - window + 1 : 0;
    const int32_t *btrow = bt + (int64_t)s * bt_stride;
    for (int32_t j = lo; j <= t; ++j) {
        const int32_t pg = j / page < bt_stride ? btrow[j / page] : -1;
        if (pg < 0 || pg >= num_pages) {
            if (lane == 0) set_error(err, HSWA_ERR_BOUNDS);
            continue;
        }
        const int64_t base = (((int64_t)pg * hkv + g) * page + j % page) * d;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
            const int c = lane + 32 * e;
            if (e < ne && c < d) dot += qv[e] * to_f(kp[base + c]);
        }
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float nm = fmaxf(m, dot);
        const float alpha = expf(m - nm), p = expf(dot - nm);
        l = l * alpha + p;
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
            const int c = lane + 32 * e;
            const float vv = (e < ne && c < d) ? to_f(vp[base + c]) : 0.f;
            acc[e] = acc[e] * alpha + p * vv;
        }
        m = nm;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *orow = o + ((int64_t)row * hq + h) * d;
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
        const int c = lane + 32 * e;
        if (e < ne && c < d) orow[c] = from_f<T>(acc[e] * inv);
    }
}

// Launch the generic kernel for decode (mode 0) or prefill (mode 1).
int launch_attention_generic(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                             const int32_t *bt, const int32_t *seq_len, const int32_t *prefix,
                             const int32_t *q_start, int32_t n_rows, int32_t n_seqs, float scale, int mode,
                             cudaStream_t st, int32_t n_tok) {
    const hswa_config &c = pool->cfg;
    if (c.head_dim > 256 || c.dtype == HSWA_DTYPE_FP8_E4M3) return HSWA_ERR_UNSUPPORTED;
    if (n_rows == 0) return HSWA_OK;
    const int32_t window = layer->kind == HSWA_KIND_SWA ? layer->window : 0;
    const int32_t num_pages = layer->kind == HSWA_KIND_SWA ? c.swa_pages : c.full_pages;
    const int64_t threads = (int64_t)n_rows * (mode == 0 ? 1 : n_seqs) * c.n_q_heads * 32;
    const int block = 256;
    const int64_t grid = (threads + block - 1) / block;
    if (grid > INT32_MAX) return HSWA_ERR_UNSUPPORTED;
    int *err = error_word();
    if (c.dtype == HSWA_DTYPE_F32) {
        set_last_kernel(mode == 0 ? "decode_generic_f32" : "prefill_generic_f32");
        attention_generic<float, 8><<<(int)grid, block, 0, st>>>(
            (const float *)q, (float *)o, (const float *)layer->k_pool, (const float *)layer->v_pool, bt, seq_len,
            prefix, q_start, n_rows, n_seqs, c.max_pages_per_seq, c.n_q_heads, c.n_kv_heads, c.head_dim,
            c.page_size, window, num_pages, scale, mode, n_tok, err);
    } else {
        set_last_kernel(mode == 0 ? "decode_generic_bf16" : "prefill_generic_bf16");
        attention_generic<__nv_bfloat16, 8><<<(int)grid, block, 0, st>>>(
            (const __nv_bfloat16 *)q, (__nv_bfloat16 *)o, (const __nv_bfloat16 *)layer->k_pool,
            (const __nv_bfloat16 *)layer->v_pool, bt, seq_len, prefix, q_start, n_rows, n_seqs,
            c.max_pages_per_seq, c.n_q_heads, c.n_kv_heads, c.head_dim, c.page_size, window, num_pages, scale,
            mode, n_tok, err);
    }
    return cudaGetLastError() == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
}

namespace {

bool decode_fp8_ok(const hswa_pool *pool, const hswa_layer *layer, const void *q, const void *o) {
    const hswa_config &c = pool->cfg;
    return c.dtype == HSWA_DTYPE_FP8_E4M3 && c.head_dim == kD && c.n_q_heads == kG * c.n_kv_heads &&
           c.page_size == kP && layer->k_scale && layer->v_scale && ((uintptr_t)q & 15) == 0 &&
           ((uintptr_t)o & 15) == 0 && ((uintptr_t)layer->k_pool & 15) == 0 && ((uintptr_t)layer->v_pool & 15) == 0 &&
           ((uintptr_t)layer->k_scale & 15) == 0 && ((uintptr_t)layer->v_scale & 15) == 0;
}

template <int kTok>
int decode_fp8_ctas_per_sm() {
    static int cache[kMaxDevices] = {};
    return kernel_setup(decode_mma_fp8_d128<kTok>, decode_smem8_bytes<kTok>(), 32 * (kConsumers8 + 1), cache);
}

// Query tokens per sequence from which an FP8 decode runs on the tensor-core
// kernel (below it, decode_mma_fp8_d128 serves 1 or 2 tokens in one pass).
constexpr int kTcMinTokensFp8 = 3;

bool decode_fast_ok(const hswa_pool *pool, const hswa_layer *layer, const void *q, const void *o) {
    const hswa_config &c = pool->cfg;
    return c.dtype == HSWA_DTYPE_BF16 && c.head_dim == kD && c.n_q_heads == kG * c.n_kv_heads &&
           c.page_size == kP && ((uintptr_t)q & 15) == 0 && ((uintptr_t)o & 15) == 0 &&
           ((uintptr_t)layer->k_pool & 15) == 0 && ((uintptr_t)layer->v_pool & 15) == 0;
}

template <int kTok>
int decode_ctas_per_sm_t() {
    static int cache[kMaxDevices] = {};
    return kernel_setup(decode_mma_bf16_d128<kTok>, decode_smem_bytes<kTok>(), 32 * (kTok + 1), cache);
}

int decode_ctas_per_sm() { return decode_ctas_per_sm_t<1>(); }

template <int kR, class Smem>
int decode_tc_ctas_per_sm_t() {
    static int cache[kMaxDevices] = {};
    return kernel_setup(decode_tc_d128<kR, Smem>, decode_tc_smem_bytes<Smem>(), Smem::kThreads, cache);
}

template <class Smem>
int decode_tc_ctas_per_sm(int n_tok) {
    switch (tc_copies(n_tok)) {
    case 4: return decode_tc_ctas_per_sm_t<4, Smem>();
    case 2: return decode_tc_ctas_per_sm_t<2, Smem>();
    default: return decode_tc_ctas_per_sm_t<1, Smem>();
    }
}

template <class Smem>
cudaError_t launch_decode_tc(int n_tok, int n_ctas, cudaStream_t st, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const DecodeArgs &a) {
    constexpr size_t smem = decode_tc_smem_bytes<Smem>();
    switch (tc_copies(n_tok)) {
    case 4: return launch_pdl(decode_tc_d128<4, Smem>, dim3(n_ctas), dim3(Smem::kThreads), smem, st, tq, tk, tv, a);
    case 2: return launch_pdl(decode_tc_d128<2, Smem>, dim3(n_ctas), dim3(Smem::kThreads), smem, st, tq, tk, tv, a);
    default: return launch_pdl(decode_tc_d128<1, Smem>, dim3(n_ctas), dim3(Smem::kThreads), smem, st, tq, tk, tv, a);
    }
}

// q as [n_seqs * n_tok][Hq][d] for the tensor-core multi-token kernels: one
// box is the n_tok x 8 query rows of a (sequence, kv head), 64 columns wide.
bool make_q_tmap(CUtensorMap *tq, const void *q, const hswa_config &c, int n_seqs, int n_tok) {
    return make_tmap_3d(tq, q, kD, (uint64_t)c.n_q_heads, (uint64_t)n_seqs * n_tok, 64, kG, (uint32_t)n_tok,
                        CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Query tokens per sequence from which the tensor-core kernel serves a
// multi-token decode. Below it the mma.sync kernel (one consumer warp per
// token) streams faster; from 4 tokens on its MMA work per page costs more
// than the tensor-core kernel, whose cost per page hardly depends on n_tok
// (decode batch, Full layer: 3 tokens 6.52 against 6.35 TB/s, 4 tokens 6.28
// against 6.39).
constexpr int kTcMinTokens = 4;

int decode_ctas_per_sm_for(int n_tok) {
    switch (n_tok) {
    case 1: return decode_ctas_per_sm_t<1>();
    case 2: return decode_ctas_per_sm_t<2>();
    default: return decode_ctas_per_sm_t<3>();
    }
}

constexpr int kMaxCtasPerSm = 4;

size_t desc_bytes(int n_seqs) { return ((size_t)(n_seqs + 1) * sizeof(int4) + 255) & ~(size_t)255; }

}  // namespace
}  // namespace hswa

using namespace hswa;

extern "C" size_t hswa_decode_multi_workspace_size(const hswa_pool *pool, int n_seqs, int n_tok) {
    if (!pool || n_seqs < 0 || n_tok < 1 || n_tok > HSWA_DECODE_MAX_TOKENS) return 0;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 192;  // no device visible: size for the largest part
    return desc_bytes(n_seqs) + (size_t)sms * kMaxCtasPerSm * 2 * n_tok * sizeof(Partial);
}

extern "C" size_t hswa_decode_workspace_size(const hswa_pool *pool, int n_seqs) {
    return hswa_decode_multi_workspace_size(pool, n_seqs, 1);
}

namespace hswa {
namespace {

int fill_args(DecodeArgs &a, const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
              const int32_t *d_bt, const int32_t *d_seq_len, int n_seqs, float scale, void *ws) {
    const hswa_config &c = pool->cfg;
    const int32_t num_pages = layer->kind == HSWA_KIND_SWA ? c.swa_pages : c.full_pages;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.bt = d_bt;
    a.seq_len = d_seq_len;
    a.sdesc = static_cast<const int4 *>(ws);
    a.k_pool = static_cast<__nv_bfloat16 *>(layer->k_pool);
    a.v_pool = static_cast<__nv_bfloat16 *>(layer->v_pool);
    a.k_scale = layer->k_scale;
    a.v_scale = layer->v_scale;
    a.part = reinterpret_cast<Partial *>(static_cast<uint8_t *>(ws) + desc_bytes(n_seqs));
    a.slots = nullptr;
    a.k_new = a.v_new = nullptr;
    a.pool_slots = (int64_t)num_pages * kP;
    a.n_seqs = n_seqs;
    a.bt_stride = c.max_pages_per_seq;
    a.hkv = c.n_kv_heads;
    a.hq = c.n_q_heads;
    a.window = layer->kind == HSWA_KIND_SWA ? layer->window : 0;
    a.num_pages = num_pages;
    a.n_tok = 1;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.err = error_word();
    return num_pages;
}

// Decode over an FP8 pool (a fused append quantizes first, as its own
// launch): 1 or 2 query tokens per sequence on decode_mma_fp8_d128, more on
// the tensor-core kernel with the pages turned into f16 in shared memory.
int decode_fp8(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o, const int32_t *d_bt,
               const int32_t *d_seq_len, int n_seqs, int n_tok, float scale, void *ws, size_t ws_bytes,
               const int32_t *slots, const void *k_new, const void *v_new, hswa_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!decode_fp8_ok(pool, layer, q, o)) return HSWA_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms <= 0) return HSWA_ERR_CUDA;
    const bool tc = n_tok >= kTcMinTokensFp8;
    const int per_sm = tc ? decode_tc_ctas_per_sm<DecodeTc8Smem>(n_tok)
                          : n_tok == 1 ? decode_fp8_ctas_per_sm<1>() : decode_fp8_ctas_per_sm<2>();
    if (per_sm <= 0) return HSWA_ERR_CUDA;
    const int n_ctas = sms * std::min(per_sm, kMaxCtasPerSm);
    if (!ws || ((uintptr_t)ws & 255) ||
        ws_bytes < desc_bytes(n_seqs) + (size_t)n_ctas * 2 * n_tok * sizeof(Partial))
        return HSWA_ERR_INVALID_ARG;
    if (slots) {
        const int rc = hswa_append_kv(pool, layer, k_new, v_new, slots, n_seqs, stream);
        if (rc != HSWA_OK) return rc;
    }
    const hswa_config &c = pool->cfg;
    DecodeArgs a;
    const int32_t num_pages = fill_args(a, pool, layer, q, o, d_bt, d_seq_len, n_seqs, scale, ws);
    a.n_tok = n_tok;
    const uint64_t blocks = (uint64_t)num_pages * c.n_kv_heads;
    CUtensorMap tk, tv, tq;
    if (!make_tmap_2d(&tk, layer->k_pool, blocks * kP, kD, kP, kD, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tv, layer->v_pool, blocks * kD, kP, kD, kP, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      CU_TENSOR_MAP_SWIZZLE_64B) ||
        (tc && !make_q_tmap(&tq, q, c, n_seqs, n_tok)))
        return HSWA_ERR_CUDA;
    set_last_kernel(tc ? "decode_tc_fp8_d128" : slots ? "append_kv_fp8+decode_mma_fp8_d128" : "decode_mma_fp8_d128");
    cudaError_t e = launch_pdl(decode_plan, dim3(1), dim3(1024), 0, st, d_seq_len, n_seqs, c.n_kv_heads, kP,
                               a.window, n_tok, static_cast<int4 *>(ws));
    if (e == cudaSuccess) {
        if (tc)
            e = launch_decode_tc<DecodeTc8Smem>(n_tok, n_ctas, st, tq, tk, tv, a);
        else if (n_tok == 1)
            e = launch_pdl(decode_mma_fp8_d128<1>, dim3(n_ctas), dim3(32 * (kConsumers8 + 1)),
                           decode_smem8_bytes<1>(), st, tk, tv, a);
        else
            e = launch_pdl(decode_mma_fp8_d128<2>, dim3(n_ctas), dim3(32 * (kConsumers8 + 1)),
                           decode_smem8_bytes<2>(), st, tk, tv, a);
    }
    if (e == cudaSuccess)
        e = launch_pdl(decode_combine, dim3(c.n_kv_heads, n_seqs * n_tok), dim3(256), 0, st, a, n_ctas);
    return e == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
}

template <int kTok>
cudaError_t launch_decode_kernel(int n_ctas, cudaStream_t st, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const DecodeArgs &a) {
    return launch_pdl(decode_mma_bf16_d128<kTok>, dim3(n_ctas), dim3(32 * (kTok + 1)),
                      decode_smem_bytes<kTok>(), st, tk, tv, a);
}

// Decode of n_tok query tokens per sequence, with an optional fused append
// of one new token (slots / k_new / v_new non-null, n_tok == 1 only).
int decode_impl(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o, const int32_t *d_bt,
                const int32_t *d_seq_len, int n_seqs, int n_tok, float scale, void *ws, size_t ws_bytes,
                const int32_t *slots, const void *k_new, const void *v_new, hswa_stream_t stream) {
    if (!pool || !layer || n_seqs < 0 || n_seqs > pool->cfg.max_seqs || n_tok < 1 ||
        n_tok > HSWA_DECODE_MAX_TOKENS || (slots && n_tok != 1) ||
        (layer->kind != HSWA_KIND_FULL && layer->kind != HSWA_KIND_SWA) ||
        (layer->kind == HSWA_KIND_SWA && layer->window <= 0))
        return HSWA_ERR_INVALID_ARG;
    if (n_seqs == 0) return HSWA_OK;
    if (!q || !o || !d_bt || !d_seq_len || !layer->k_pool || !layer->v_pool) return HSWA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool fused = slots != nullptr;
    if (pool->cfg.dtype == HSWA_DTYPE_FP8_E4M3) {
        if ((int64_t)n_seqs * n_tok > 65535) return HSWA_ERR_UNSUPPORTED;  // rows of the combine grid
        return decode_fp8(pool, layer, q, o, d_bt, d_seq_len, n_seqs, n_tok, scale, ws, ws_bytes, slots, k_new,
                          v_new, stream);
    }
    if (!decode_fast_ok(pool, layer, q, o) ||
        (fused && (((uintptr_t)k_new & 15) || ((uintptr_t)v_new & 15)))) {
        if (fused) {
            const int rc = hswa_append_kv(pool, layer, k_new, v_new, slots, n_seqs, stream);
            if (rc != HSWA_OK) return rc;
        }
        return launch_attention_generic(pool, layer, q, o, d_bt, d_seq_len, nullptr, nullptr, n_seqs * n_tok,
                                        n_seqs, scale, 0, st, n_tok);
    }
    const hswa_config &c = pool->cfg;
    if ((int64_t)n_seqs * n_tok > 65535) return HSWA_ERR_UNSUPPORTED;  // rows of the combine grid
    const int sms = sm_count();
    if (sms <= 0) return HSWA_ERR_CUDA;
    const bool tc = n_tok >= kTcMinTokens;
    const int per_sm = tc ? decode_tc_ctas_per_sm<DecodeTcSmem>(n_tok) : decode_ctas_per_sm_for(n_tok);
    if (per_sm <= 0) return HSWA_ERR_CUDA;
    const int n_ctas = sms * std::min(per_sm, kMaxCtasPerSm);
    if (!ws || ((uintptr_t)ws & 255) ||
        ws_bytes < desc_bytes(n_seqs) + (size_t)n_ctas * 2 * n_tok * sizeof(Partial))
        return HSWA_ERR_INVALID_ARG;
    DecodeArgs a;
    const int32_t num_pages = fill_args(a, pool, layer, q, o, d_bt, d_seq_len, n_seqs, scale, ws);
    a.slots = slots;
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.n_tok = n_tok;
    CUtensorMap tk, tv, tq;
    const uint64_t rows = (uint64_t)num_pages * c.n_kv_heads * kP;
    if (!make_tmap_2d(&tk, layer->k_pool, rows, kD, 64, 64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tv, layer->v_pool, rows, kD, 64, 64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return HSWA_ERR_CUDA;
    if (tc && !make_q_tmap(&tq, q, c, n_seqs, n_tok)) return HSWA_ERR_CUDA;
    set_last_kernel(tc ? "decode_tc_bf16_d128" : fused ? "decode_mma_bf16_d128+append" : "decode_mma_bf16_d128");
    // three launches chained with programmatic dependent launch: each one
    // is scheduled while its predecessor finishes and waits for it on entry
    if (launch_pdl(decode_plan, dim3(1), dim3(1024), 0, st, d_seq_len, n_seqs, c.n_kv_heads, kP, a.window, n_tok,
                   static_cast<int4 *>(ws)) != cudaSuccess)
        return HSWA_ERR_CUDA;
    cudaError_t e;
    if (tc) {
        e = launch_decode_tc<DecodeTcSmem>(n_tok, n_ctas, st, tq, tk, tv, a);
    } else switch (n_tok) {
    case 1: e = launch_decode_kernel<1>(n_ctas, st, tk, tv, a); break;
    case 2: e = launch_decode_kernel<2>(n_ctas, st, tk, tv, a); break;
    default: e = launch_decode_kernel<3>(n_ctas, st, tk, tv, a); break;
    }
    if (e != cudaSuccess ||
        launch_pdl(decode_combine, dim3(c.n_kv_heads, n_seqs * n_tok), dim3(256), 0, st, a, n_ctas) != cudaSuccess)
        return HSWA_ERR_CUDA;
    return HSWA_OK;
}

}  // namespace
}  // namespace hswa

extern "C" int hswa_decode(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                           const int32_t *d_bt, const int32_t *d_seq_len, int n_seqs, float scale, void *ws,
                           size_t ws_bytes, hswa_stream_t stream) {
    HSWA_NVTX("hswa_decode");
    return decode_impl(pool, layer, q, o, d_bt, d_seq_len, n_seqs, 1, scale, ws, ws_bytes, nullptr, nullptr, nullptr,
                       stream);
}

extern "C" int hswa_decode_append(const hswa_pool *pool, const hswa_layer *layer, const void *q, const void *k_new,
                                  const void *v_new, const int32_t *d_slots, void *o, const int32_t *d_bt,
                                  const int32_t *d_seq_len, int n_seqs, float scale, void *ws, size_t ws_bytes,
                                  hswa_stream_t stream) {
    HSWA_NVTX("hswa_decode_append");
    if (!k_new || !v_new || !d_slots) return HSWA_ERR_INVALID_ARG;
    return decode_impl(pool, layer, q, o, d_bt, d_seq_len, n_seqs, 1, scale, ws, ws_bytes, d_slots, k_new, v_new,
                       stream);
}

extern "C" int hswa_decode_multi(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                                 const int32_t *d_bt, const int32_t *d_seq_len, int n_seqs, int n_tok, float scale,
                                 void *ws, size_t ws_bytes, hswa_stream_t stream) {
    HSWA_NVTX("hswa_decode_multi");
    return decode_impl(pool, layer, q, o, d_bt, d_seq_len, n_seqs, n_tok, scale, ws, ws_bytes, nullptr, nullptr,
                       nullptr, stream);
}

// ---------------------------------------------------- no-allocation decode
// The split-K scratch of hswa_decode_noalloc: a fixed array in the device
// image. Host code only ever passes the address cudaGetSymbolAddress gives
// for it on the current device; the host-side symbol is a stand-in, not a
// device address.
static __device__ __align__(256) uint8_t g_decode_scratch[HSWA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mu;
void *g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current), or nullptr.
void *decode_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}
}  // namespace

extern "C" int hswa_decode_noalloc(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                                   const int32_t *d_bt, const int32_t *d_seq_len, int n_seqs, float scale,
                                   hswa_stream_t stream) {
    HSWA_NVTX("hswa_decode_noalloc");
    if (!pool || n_seqs < 0 || n_seqs > HSWA_DECODE_NOALLOC_MAX_SEQS) return HSWA_ERR_INVALID_ARG;
    if (n_seqs > 0 && layer && decode_fast_ok(pool, layer, q, o)) {
        // the exact scratch the fast path will use must fit the fixed array
        const int sms = sm_count();
        const int per_sm = decode_ctas_per_sm();
        if (sms <= 0 || per_sm <= 0) return HSWA_ERR_CUDA;
        const size_t need = desc_bytes(n_seqs) + (size_t)sms * std::min(per_sm, kMaxCtasPerSm) * 2 * sizeof(Partial);
        if (need > HSWA_DECODE_NOALLOC_SCRATCH_BYTES) return HSWA_ERR_INVALID_ARG;
    }
    void *ws = decode_scratch();
    if (!ws) return HSWA_ERR_CUDA;
    return hswa_decode(pool, layer, q, o, d_bt, d_seq_len, n_seqs, scale, ws, HSWA_DECODE_NOALLOC_SCRATCH_BYTES,
                       stream);
}
