// Chunked-prefill attention over the dual KV pool.
//
// "MiMo-V2.5 Series Inference Full-Link Optimization", Sec. 1.1: in chunked
// prefill the attention is close to compute-bound; SWA layers attend only to
// the last W tokens, so their cost per query is O(W) instead of O(N).
//
// Fast path (bf16, d = 128, page 64, an even number of query heads per kv
// head): one CTA per (sequence, block of 128 chunk rows, pair of query heads
// of one kv head), on the 5th-generation tensor cores.
//   * S = Q K^T and O += P V are tcgen05.mma (M = 128 rows, N = 128, K = 16)
//     with fp32 accumulators in tensor memory: S_A, S_B, O_A, O_B take the
//     512 TMEM columns of the SM; P (bf16) is written back over S and read by
//     the PV MMA straight from TMEM.
//   * Warp 8 streams Q (once) and K / V tiles of 128 keys (two pages, two
//     64-column boxes per page, 128-byte swizzle) by TMA into a 4-slot ring.
//   * Warp 9 issues the MMAs (one thread) and commits them to mbarriers.
//   * Warps 0-3 and 4-7 own query head A and B: one thread per query row
//     reads its row of S from TMEM, applies the causal / window mask on the
//     tiles that need it, keeps the running max in the log2 domain and only
//     rescales O (in TMEM) when the max grows by more than 2^8, writes P,
//     and at the end normalises its row of O and stores it.
//   * The KV range of a block is clipped to the tiles its rows can see: all
//     of [0, t] for a Full layer, [t - W + 1, t] for an SWA layer.
// Every wait is bounded; on a timeout the CTA records HSWA_ERR_TIMEOUT,
// drains its copies and MMAs, frees its TMEM and returns.
//
// FP8 pools ("Baidu AI Cloud: Day-0 support for hybrid-architecture LLMs",
// Optimization 2 item 2): a staging pass first writes fp16 copies of the
// pages the chunk reads (code x scale, rounded once: 11 significant bits
// against E4M3's 4, so the copy adds an error far below bf16's) and of q into
// the caller's workspace, with a block table onto the page copies; the same
// tensor-core kernel then runs with fp16 operands (q, K, V and P all fp16).
// The chunk's attention is compute-bound (tens of TFLOP per chunk against a
// few GB moved by the staging), so the pass costs about a percent.
#include <algorithm>

#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "kernels.h"
#include "tc.cuh"

namespace hswa {
namespace {

constexpr int kD = 128;
constexpr int kP = 64;
constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per KV tile (two pages)
constexpr int kSlots = 4;
constexpr uint32_t kTileBytes = kBN * kD * 2;  // 32 KB: one K or V tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 64-column half (128 rows x 128 B)
constexpr uint32_t kBoxBytes = kP * 128;         // one page x 64 columns
constexpr int kThreads = 320;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8

struct PrefillSmem {
    uint8_t q[2][kTileBytes];          // Q_A, Q_B: [d half][128 rows][128 B]
    uint8_t kv[kSlots][kTileBytes];    // K or V tiles: [d half][128 keys][128 B]
    uint64_t q_full;
    uint64_t kv_full[kSlots], kv_empty[kSlots];
    uint64_t s_full[2], p_full[2], o_final[2];
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(offsetof(PrefillSmem, kv) % 1024 == 0, "128-byte swizzled tiles need 1024-byte alignment");
constexpr size_t kPrefillSmemBytes = sizeof(PrefillSmem) + 1024;

struct PrefillArgs {
    const int32_t *bt;
    const int32_t *prefix;
    const int32_t *q_start;
    __nv_bfloat16 *o;
    int32_t n_seqs, bt_stride, hq, hkv, window, num_pages;
    int32_t kv_rows;  // rows of the pool tensor map (OOB row = zero fill)
    float scale_log2;
    int *err;
};

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------------------------- work unit
struct Unit {
    int32_t s, qb, hp, g;
    int32_t n_rows;     // valid rows of this block
    int32_t row0;       // q row of the block's first row
    int32_t p0;         // position of the first row
    int32_t tile_lo;    // first KV tile (128 keys)
    int32_t n_tiles;
    int32_t L;          // keys of the sequence after the chunk
};

__device__ __forceinline__ bool make_unit(const PrefillArgs &a, Unit &u) {
    u.hp = blockIdx.x;
    u.qb = blockIdx.y;
    u.s = blockIdx.z;
    const int32_t g_heads = a.hq / a.hkv;
    u.g = (2 * u.hp) / g_heads;
    const int32_t q0 = a.q_start[u.s], n = a.q_start[u.s + 1] - q0;
    if (u.qb * kBM >= n) return false;
    u.n_rows = min(kBM, n - u.qb * kBM);
    u.row0 = q0 + u.qb * kBM;
    const int32_t pre = a.prefix[u.s];
    u.p0 = pre + u.qb * kBM;
    u.L = pre + n;
    const int32_t t_max = u.p0 + u.n_rows - 1;
    const int32_t key_lo = (a.window > 0 && u.p0 - a.window + 1 > 0) ? u.p0 - a.window + 1 : 0;
    u.tile_lo = key_lo / kBN;
    u.n_tiles = t_max / kBN - u.tile_lo + 1;
    return true;
}

// ------------------------------------------------------------------ roles
__device__ void prefill_producer(PrefillSmem &sm, const CUtensorMap *tq, const CUtensorMap *tk,
                                 const CUtensorMap *tv, const PrefillArgs &a, const Unit &u) {
    prefetch_tmap(tq);
    prefetch_tmap(tk);
    prefetch_tmap(tv);
    mbar_arrive_expect_tx(&sm.q_full, 2 * kTileBytes);
    for (int x = 0; x < 2; ++x)
        for (int dh = 0; dh < 2; ++dh)
            tma_load_3d(sm.q[x] + dh * kHalfBytes, tq, dh * 64, 2 * u.hp + x, u.row0, &sm.q_full);
    const int32_t *btrow = a.bt + (int64_t)u.s * a.bt_stride;
    // pages the block's rows can see; the first tile may start on an older
    // page (released for an SWA layer), which is filled with zeros instead
    const int32_t last_page = (u.L - 1) / kP;
    const int32_t first_page = (a.window > 0 && u.p0 - a.window + 1 > 0 ? u.p0 - a.window + 1 : 0) / kP;
    int issued = 0;
    for (int i = 0; i < 2 * u.n_tiles; ++i) {
        const int slot = i % kSlots;
        if (!mbar_wait(&sm.kv_empty[slot], ((i / kSlots) & 1) ^ 1, a.err) || *(volatile int32_t *)&sm.abort) {
            sm.abort = 1;
            break;
        }
        const CUtensorMap *map = (i & 1) ? tv : tk;
        const int32_t tile = u.tile_lo + (i >> 1);
        mbar_arrive_expect_tx(&sm.kv_full[slot], kTileBytes);
        for (int pg = 0; pg < 2; ++pg) {
            const int32_t lp = tile * 2 + pg;
            int32_t row = a.kv_rows;  // out of range: the copy fills zeros
            if (lp >= first_page && lp <= last_page) {
                const int32_t page = lp < a.bt_stride ? btrow[lp] : -1;
                if (page >= 0 && page < a.num_pages)
                    row = (page * a.hkv + u.g) * kP;
                else
                    set_error(a.err, HSWA_ERR_BOUNDS);
            }
            for (int dh = 0; dh < 2; ++dh)
                tma_load_2d(sm.kv[slot] + dh * kHalfBytes + pg * kBoxBytes, map, dh * 64, row, &sm.kv_full[slot]);
        }
        ++issued;
    }
    // drain: never leave copies landing in shared memory after the CTA ends
    for (int i = max(0, issued - kSlots); i < issued; ++i) mbar_wait(&sm.kv_full[i % kSlots], (i / kSlots) & 1, a.err);
}

// S_x = Q_x K^T over d = 128: 8 steps of K = 16 (32 bytes inside a 128-byte
// swizzle row; the second half of d is the second 16 KB block). qd and kd
// are the descriptors of the tiles' first bytes: a step's descriptor is that
// plus its byte offset / 16 in the address field (no carry: shared-memory
// addresses stay below 2^18).
template <bool kF16>
__device__ __forceinline__ void issue_s(uint32_t t_s, uint64_t qd, uint64_t kd) {
    constexpr uint32_t kIdescQK = idesc_16(kBM, kBN, false, kF16);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off16 = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
        mma_ss(t_s, qd + off16, kd + off16, kIdescQK, kk > 0);
    }
}

// O_x += P_x V over 128 keys: 8 steps of K = 16 keys; P_x (bf16 pairs) sits in
// the first 64 columns of S_x, V is MN-major (d contiguous) with the two
// 64-column halves 16 KB apart.
template <bool kF16>
__device__ __forceinline__ void issue_pv(uint32_t t_o, uint32_t t_p, uint64_t vd, bool first_tile) {
    constexpr uint32_t kIdescPV = idesc_16(kBM, kD, true, kF16);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(t_o, t_p + kk * 8, vd + kk * (2048 >> 4), kIdescPV, (first_tile && kk == 0) ? 0u : 1u);
}

template <bool kF16>
__device__ void prefill_mma(PrefillSmem &sm, const PrefillArgs &a, const Unit &u) {
    const uint32_t tbase = sm.tmem_base;
    const uint32_t ts0 = tbase, ts1 = tbase + 128, to0 = tbase + 256, to1 = tbase + 384;
    const uint64_t qd0 = sdesc(smem_u32(sm.q[0]), 16, 1024), qd1 = sdesc(smem_u32(sm.q[1]), 16, 1024);
    bool ok = mbar_wait(&sm.q_full, 0, a.err);
    tc_fence_after();
    const int n = u.n_tiles;
    if (ok && n > 0) {
        ok = mbar_wait(&sm.kv_full[0], 0, a.err);  // K(0)
        if (ok) {
            tc_fence_after();
            const uint64_t k0 = sdesc(smem_u32(sm.kv[0]), 16, 1024);
            issue_s<kF16>(ts0, qd0, k0);
            mma_commit(&sm.s_full[0]);
            issue_s<kF16>(ts1, qd1, k0);
            mma_commit(&sm.s_full[1]);
            mma_commit(&sm.kv_empty[0]);
        }
        for (int j = 0; ok && j < n; ++j) {
            const int iv = 2 * j + 1, ik = 2 * j + 2;  // ring items V(j), K(j + 1)
            const int sv = iv % kSlots, sk = ik % kSlots;
            ok = mbar_wait(&sm.kv_full[sv], (iv / kSlots) & 1, a.err) && mbar_wait(&sm.p_full[0], j & 1, a.err) &&
                 !*(volatile int32_t *)&sm.abort;
            if (!ok) break;
            tc_fence_after();
            const uint64_t vd = sdesc(smem_u32(sm.kv[sv]), kHalfBytes, 1024);
            issue_pv<kF16>(to0, ts0, vd, j == 0);
            const bool more = j + 1 < n;
            uint64_t kd = 0;
            if (more) {
                ok = mbar_wait(&sm.kv_full[sk], (ik / kSlots) & 1, a.err);
                if (!ok) break;
                tc_fence_after();
                kd = sdesc(smem_u32(sm.kv[sk]), 16, 1024);
                issue_s<kF16>(ts0, qd0, kd);
                mma_commit(&sm.s_full[0]);
            }
            ok = mbar_wait(&sm.p_full[1], j & 1, a.err) && !*(volatile int32_t *)&sm.abort;
            if (!ok) break;
            tc_fence_after();
            issue_pv<kF16>(to1, ts1, vd, j == 0);
            mma_commit(&sm.kv_empty[sv]);
            if (more) {
                issue_s<kF16>(ts1, qd1, kd);
                mma_commit(&sm.s_full[1]);
                mma_commit(&sm.kv_empty[sk]);
            }
        }
    }
    // tracks every MMA issued above: the softmax warps wait on it before
    // reading O and before the TMEM is freed
    mma_commit(&sm.o_final[0]);
    mma_commit(&sm.o_final[1]);
    if (!ok) sm.abort = 1;
}

template <bool kF16>
__device__ void prefill_softmax(PrefillSmem &sm, const PrefillArgs &a, const Unit &u, int x) {
    const int warp = (threadIdx.x >> 5) & 3;
    const int r = warp * 32 + (threadIdx.x & 31);  // query row of this thread
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_s = sm.tmem_base + lane_off + 128 * x;
    const uint32_t t_o = sm.tmem_base + lane_off + 256 + 128 * x;
    const int32_t t = u.p0 + min(r, u.n_rows - 1);  // rows past the chunk repeat the last valid row
    const int32_t t_min = u.p0, t_max = u.p0 + u.n_rows - 1;
    const int32_t W = a.window;
    float m_used = -INFINITY, l = 0.f;  // running max (log2 units) and sum of P
    bool ok = true;
    for (int j = 0; j < u.n_tiles; ++j) {
        ok = mbar_wait(&sm.s_full[x], j & 1, a.err) && !*(volatile int32_t *)&sm.abort;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // S row in four 32-column chunks; each load overlaps the mask and
        // max work of the chunk before it
        uint32_t sr[4][32];
        const int32_t k0 = (u.tile_lo + j) * kBN;
        const bool masked = (k0 + kBN - 1 > t_min) || (W > 0 && k0 < t_max - W + 1);
        const int32_t hi_c = t - k0;                       // keys c <= hi_c
        const int32_t lo_c = W > 0 ? t - W + 1 - k0 : -1;  // keys c >= lo_c
        // one max per chunk, each a chain of 8: short dependency chains for a
        // thread that has few warps beside it to hide them
        float mc[4];
        tmem_ld32(t_s, sr[0]);
        tmem_wait_ld(sr[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c + 1 < 4) tmem_ld32(t_s + 32 * (c + 1), sr[c + 1]);
            // raw scores: the scale (> 0) does not change which keys win the max
            if (masked) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int col = c * 32 + i;
                    if (col > hi_c || col < lo_c) sr[c][i] = __float_as_uint(-INFINITY);
                }
            }
            float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                m0 = max3(m0, __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
                m1 = max3(m1, __uint_as_float(sr[c][i + 2]), __uint_as_float(sr[c][i + 3]));
            }
            mc[c] = fmaxf(m0, m1);
            if (c + 1 < 4) tmem_wait_ld(sr[c + 1]);
        }
        const float mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])) * a.scale_log2;
        // A new reference max only when the row max grows by more than 2^8;
        // then O (nothing before the first PV) and l are rescaled.
        const bool need = mx > m_used + kRescaleLog2;
        const bool resc = need && j > 0 && m_used != -INFINITY;
        const float alpha = resc ? fast_exp2(m_used - mx) : 1.f;
        if (need) m_used = mx;
        const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nm2 = make_float2(neg_m, neg_m);
        float2 sums[4];  // one running sum per chunk (chains of 16, not 64)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float2 &sum2 = sums[c];
            sum2 = make_float2(0.f, 0.f);
            // P = 2^(s * scale - m) two keys at a time (packed f32x2 FMA and
            // add), packed to bf16 pairs in place, then its 16 columns (32
            // keys) written over the start of S
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])),
                                            sc2, nm2);
                const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                sum2 = __fadd2_rn(sum2, p);
                sr[c][i] = kF16 ? pack_f16(p.x, p.y) : pack_bf16(p.x, p.y);
            }
            tmem_st16(t_s + 16 * c, sr[c]);
        }
        // the O rescale comes after the P store (the S registers are free
        // then); TMEM loads and stores are warp-wide, so the whole warp takes
        // this path when any of its rows needs it (the others scale by 1)
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t ov[32];
                tmem_ld32(t_o + 32 * c, ov);
                tmem_wait_ld(ov);
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                tmem_st32(t_o + 32 * c, ov);
            }
        }
        const float2 s01 = __fadd2_rn(sums[0], sums[1]), s23 = __fadd2_rn(sums[2], sums[3]);
        const float2 sum2 = __fadd2_rn(s01, s23);
        l = l * alpha + (sum2.x + sum2.y);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_full[x]);
    }
    // epilogue: wait for the last PV (always: TMEM is freed after this
    // function returns), normalise this row of O and store it
    const bool fin = mbar_wait(&sm.o_final[x], 0, a.err);
    ok = __all_sync(0xffffffffu, ok && fin);
    if (!ok) {
        sm.abort = 1;
        return;
    }
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int h = 2 * u.hp + x;
    uint4 *dst = reinterpret_cast<uint4 *>(a.o + ((int64_t)(u.row0 + r) * a.hq + h) * kD);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(t_o + 32 * c, ov);
        tmem_wait_ld(ov);
        if (r < u.n_rows) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 w;
                w.x = pack_bf16(__uint_as_float(ov[8 * i + 0]) * inv, __uint_as_float(ov[8 * i + 1]) * inv);
                w.y = pack_bf16(__uint_as_float(ov[8 * i + 2]) * inv, __uint_as_float(ov[8 * i + 3]) * inv);
                w.z = pack_bf16(__uint_as_float(ov[8 * i + 4]) * inv, __uint_as_float(ov[8 * i + 5]) * inv);
                w.w = pack_bf16(__uint_as_float(ov[8 * i + 6]) * inv, __uint_as_float(ov[8 * i + 7]) * inv);
                dst[c * 4 + i] = w;
            }
        }
    }
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_bf16_d128(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, PrefillArgs a) {
    Unit u;
    if (!make_unit(a, u)) return;
    extern __shared__ uint8_t raw[];
    PrefillSmem &sm =
        *reinterpret_cast<PrefillSmem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sm.s_full[x], 1);
            mbar_init(&sm.p_full[x], 128);
            mbar_init(&sm.o_final[x], 1);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(&sm.tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp < 8)
        prefill_softmax<kF16>(sm, a, u, warp >> 2);
    else if (warp == 8) {
        if ((threadIdx.x & 31) == 0) prefill_producer(sm, &tq, &tk, &tv, a, u);
        __syncwarp();
    } else {
        if ((threadIdx.x & 31) == 0) prefill_mma<kF16>(sm, a, u);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(sm.tmem_base));
}

bool prefill_fast_ok(const hswa_pool *pool, const hswa_layer *layer, const void *q, const void *o) {
    const hswa_config &c = pool->cfg;
    const int g = c.n_q_heads / c.n_kv_heads;
    return (c.dtype == HSWA_DTYPE_BF16 || c.dtype == HSWA_DTYPE_FP8_E4M3) && c.head_dim == kD && c.page_size == kP &&
           g % 2 == 0 && ((uintptr_t)q & 15) == 0 && ((uintptr_t)o & 15) == 0 &&
           ((uintptr_t)layer->k_pool & 15) == 0 && ((uintptr_t)layer->v_pool & 15) == 0;
}

// ------------------------------------------------------------ FP8 staging
// Pages per sequence the staging copy reserves: a Full layer may read every
// logical page; an SWA layer's chunk of at most max_q_len rows reads keys
// [prefix - W + 1, prefix + n), at most W - 1 + max_q_len keys.
int32_t stage_pages_per_seq(const hswa_config &c, const hswa_layer *layer, int max_q_len) {
    if (layer->kind != HSWA_KIND_SWA) return c.max_pages_per_seq;
    const int64_t keys = (int64_t)layer->window - 1 + max_q_len;
    return (int32_t)std::min<int64_t>(c.max_pages_per_seq, (keys + kP - 1) / kP + 1);
}

constexpr size_t align1k(size_t x) { return (x + 1023) & ~(size_t)1023; }

// Workspace of an FP8 chunk: the staging block table, the fp16 K and V page
// copies, and the fp16 copy of q (n_seqs * max_q_len rows at most).
struct StageLayout {
    int32_t per_seq;
    size_t page_bytes, k_off, v_off, q_off, total;
};

StageLayout stage_layout(const hswa_config &c, const hswa_layer *layer, int n_seqs, int max_q_len) {
    StageLayout l;
    l.per_seq = stage_pages_per_seq(c, layer, max_q_len);
    l.page_bytes = (size_t)c.n_kv_heads * kP * kD * sizeof(__half);
    const size_t pages = (size_t)n_seqs * l.per_seq;
    l.k_off = align1k((size_t)n_seqs * c.max_pages_per_seq * sizeof(int32_t));
    l.v_off = l.k_off + align1k(pages * l.page_bytes);
    l.q_off = l.v_off + align1k(pages * l.page_bytes);
    l.total = l.q_off + align1k((size_t)n_seqs * max_q_len * c.n_q_heads * kD * sizeof(__half));
    return l;
}

struct StageArgs {
    const int32_t *bt, *prefix, *q_start;
    const uint8_t *k_codes, *v_codes;  // [page][Hkv][P][d], V pages [page][Hkv][d][P]
    const float *k_scale, *v_scale;    // [page][Hkv][P] (one 128-element tile per row)
    int32_t *stage_bt;                 // [n_seqs][bt_stride]
    __half *k_out, *v_out;             // [n_seqs * per_seq][Hkv][P][d]
    int32_t n_seqs, bt_stride, hkv, window, num_pages, per_seq;
    int *err;
};

// fp16 of an E4M3 code (exact) times its fp32 scale, rounded once to fp16;
// magnitudes past the fp16 range saturate at 65504.
__device__ __forceinline__ __half2 dequant_f16x2(uint8_t c0, uint8_t c1, float s0, float s1) {
    const float2 f =
        __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(c0 | (c1 << 8)), __NV_E4M3)));
    return __floats2half2_rn(fminf(fmaxf(f.x * s0, -65504.f), 65504.f), fminf(fmaxf(f.y * s1, -65504.f), 65504.f));
}

// One block per (logical page j, sequence s): writes the staging table entry
// of (s, j) and, for a page the chunk reads, its fp16 copy (K rows stay
// rows; each kv head's transposed V block [d][P] becomes [P][d]).
__global__ void __launch_bounds__(256) prefill_stage_fp8(StageArgs a) {
    const int32_t j = blockIdx.x, s = blockIdx.y;
    const int32_t pre = a.prefix[s], n = a.q_start[s + 1] - a.q_start[s];
    const int32_t lo_key = (a.window > 0 && pre - a.window + 1 > 0) ? pre - a.window + 1 : 0;
    const int32_t lo_pg = lo_key / kP, hi_pg = n > 0 ? (pre + n - 1) / kP : -1;
    int32_t page = -1, slot = -1;
    if (j >= lo_pg && j <= hi_pg) {
        page = a.bt[(int64_t)s * a.bt_stride + j];
        if (j - lo_pg >= a.per_seq) {  // the workspace was sized for fewer rows
            if (threadIdx.x == 0) set_error(a.err, HSWA_ERR_BOUNDS);
            page = -1;
        }
        if (page >= 0 && page < a.num_pages) slot = s * a.per_seq + (j - lo_pg);
    }
    if (threadIdx.x == 0) a.stage_bt[(int64_t)s * a.bt_stride + j] = slot;  // -1: the kernel reports it if read
    if (slot < 0) return;
    // K: 16 codes per thread and step
    const uint8_t *kc = a.k_codes + (int64_t)page * a.hkv * kP * kD;
    const float *ks = a.k_scale + (int64_t)page * a.hkv * kP;
    __half *ko = a.k_out + (int64_t)slot * a.hkv * kP * kD;
    const int32_t chunks = a.hkv * kP * kD / 16;
    for (int32_t c = threadIdx.x; c < chunks; c += blockDim.x) {
        const uint4 raw = reinterpret_cast<const uint4 *>(kc)[c];
        const float sc = ks[c / (kD / 16)];  // row (kv head, key) of the chunk
        const uint8_t *b = reinterpret_cast<const uint8_t *>(&raw);
        __align__(16) __half2 out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = dequant_f16x2(b[2 * i], b[2 * i + 1], sc, sc);
        reinterpret_cast<uint4 *>(ko)[2 * c] = reinterpret_cast<const uint4 *>(out)[0];
        reinterpret_cast<uint4 *>(ko)[2 * c + 1] = reinterpret_cast<const uint4 *>(out)[1];
    }
    // V: each kv head's [d][P] code block is transposed to [P][d] through
    // shared memory (row stride 65 bytes keeps the column reads off one bank)
    __shared__ uint8_t tile[kD * 65];
    __shared__ float vsc[kP];
    const uint8_t *vc = a.v_codes + (int64_t)page * a.hkv * kD * kP;
    const float *vs = a.v_scale + (int64_t)page * a.hkv * kP;
    __half *vo = a.v_out + (int64_t)slot * a.hkv * kP * kD;
    for (int32_t h = 0; h < a.hkv; ++h) {
        __syncthreads();
        for (int32_t c = threadIdx.x; c < kD * kP / 16; c += blockDim.x) {
            const uint4 raw = reinterpret_cast<const uint4 *>(vc + (int64_t)h * kD * kP)[c];
            const uint8_t *b = reinterpret_cast<const uint8_t *>(&raw);
            const int32_t d = c / (kP / 16), p0 = (c % (kP / 16)) * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i) tile[d * 65 + p0 + i] = b[i];
        }
        if (threadIdx.x < kP) vsc[threadIdx.x] = vs[h * kP + threadIdx.x];
        __syncthreads();
        for (int32_t c = threadIdx.x; c < kP * kD / 8; c += blockDim.x) {
            const int32_t p = c / (kD / 8), d0 = (c % (kD / 8)) * 8;
            const float sc = vsc[p];
            __align__(16) __half2 out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                out[i] = dequant_f16x2(tile[(d0 + 2 * i) * 65 + p], tile[(d0 + 2 * i + 1) * 65 + p], sc, sc);
            *reinterpret_cast<uint4 *>(vo + ((int64_t)h * kP + p) * kD + d0) = *reinterpret_cast<const uint4 *>(out);
        }
    }
}

// q (bf16) to fp16 for the fp16 MMAs: exact for magnitudes in
// [2^-14, 65504], subnormal below, saturated above. 8 elements per step.
__global__ void __launch_bounds__(256) prefill_q_to_f16(const __nv_bfloat16 *__restrict__ q, __half *__restrict__ q16,
                                                        int64_t n8) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 raw = reinterpret_cast<const uint4 *>(q)[i];
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&raw);
        __align__(16) __half2 out[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(b[k]);
            out[k] = __floats2half2_rn(fminf(fmaxf(f.x, -65504.f), 65504.f), fminf(fmaxf(f.y, -65504.f), 65504.f));
        }
        reinterpret_cast<uint4 *>(q16)[i] = *reinterpret_cast<const uint4 *>(out);
    }
}

// The tensor-core prefill over 16-bit pages k_pool / v_pool (num_pages
// pages) addressed through bt; q, K and V all bf16, or all fp16 (f16).
int launch_prefill_tc(const hswa_config &c, int32_t window, const void *k_pool, const void *v_pool, bool f16,
                      int32_t num_pages, const int32_t *bt, const void *q, void *o, const int32_t *d_prefix_len,
                      const int32_t *d_q_start, int n_seqs, int total_q, int max_q_len, float scale,
                      cudaStream_t st) {
    const uint64_t rows = (uint64_t)num_pages * c.n_kv_heads * kP;
    if (rows >= (1ull << 31)) return HSWA_ERR_UNSUPPORTED;
    const CUtensorMapDataType ty = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_3d(&tq, q, kD, c.n_q_heads, (uint64_t)total_q, 64, 1, kBM, ty, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tk, k_pool, rows, kD, kP, 64, ty, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tv, v_pool, rows, kD, kP, 64, ty, CU_TENSOR_MAP_SWIZZLE_128B))
        return HSWA_ERR_CUDA;
    PrefillArgs a;
    a.bt = bt;
    a.prefix = d_prefix_len;
    a.q_start = d_q_start;
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.n_seqs = n_seqs;
    a.bt_stride = c.max_pages_per_seq;
    a.hq = c.n_q_heads;
    a.hkv = c.n_kv_heads;
    a.window = window;
    a.num_pages = num_pages;
    a.kv_rows = (int32_t)rows;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.err = error_word();
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(prefill_tc_bf16_d128<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrefillSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_tc_bf16_d128<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrefillSmemBytes) != cudaSuccess)
            return HSWA_ERR_CUDA;
        attr = true;
    }
    dim3 grid(c.n_q_heads / 2, (max_q_len + kBM - 1) / kBM, n_seqs);
    if (f16)
        prefill_tc_bf16_d128<true><<<grid, kThreads, kPrefillSmemBytes, st>>>(tq, tk, tv, a);
    else
        prefill_tc_bf16_d128<false><<<grid, kThreads, kPrefillSmemBytes, st>>>(tq, tk, tv, a);
    return cudaGetLastError() == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
}

}  // namespace
}  // namespace hswa

using namespace hswa;

extern "C" size_t hswa_prefill_workspace_size(const hswa_pool *pool, const hswa_layer *layer, int n_seqs,
                                              int max_q_len) {
    if (!pool || !layer || n_seqs < 0 || max_q_len < 0 || pool->cfg.dtype != HSWA_DTYPE_FP8_E4M3) return 0;
    if (layer->kind == HSWA_KIND_SWA && layer->window <= 0) return 0;
    return stage_layout(pool->cfg, layer, n_seqs, max_q_len).total;
}

extern "C" int hswa_prefill_chunk_ws(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                                     const int32_t *d_bt, const int32_t *d_prefix_len, const int32_t *d_q_start,
                                     int n_seqs, int total_q, int max_q_len, float scale, void *ws, size_t ws_bytes,
                                     hswa_stream_t stream) {
    if (!pool || !layer || n_seqs < 0 || n_seqs > pool->cfg.max_seqs || max_q_len < 0 || total_q < 0 ||
        !(scale > 0.f) ||
        (n_seqs > 0 && max_q_len > total_q) ||
        (layer->kind != HSWA_KIND_FULL && layer->kind != HSWA_KIND_SWA) ||
        (layer->kind == HSWA_KIND_SWA && layer->window <= 0))
        return HSWA_ERR_INVALID_ARG;
    if (n_seqs == 0 || max_q_len == 0 || total_q == 0) return HSWA_OK;
    if (!q || !o || !d_bt || !d_prefix_len || !d_q_start || !layer->k_pool || !layer->v_pool)
        return HSWA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const hswa_config &c = pool->cfg;
    const int32_t window = layer->kind == HSWA_KIND_SWA ? layer->window : 0;
    const int32_t num_pages = layer->kind == HSWA_KIND_SWA ? c.swa_pages : c.full_pages;
    if (c.dtype == HSWA_DTYPE_FP8_E4M3) {
        if (!prefill_fast_ok(pool, layer, q, o) || c.head_dim != 128 || !layer->k_scale || !layer->v_scale ||
            ((uintptr_t)layer->k_pool & 15) || ((uintptr_t)layer->v_pool & 15))
            return HSWA_ERR_UNSUPPORTED;
        const StageLayout l = stage_layout(c, layer, n_seqs, max_q_len);
        if (!ws || ((uintptr_t)ws & 255) || ws_bytes < l.total) return HSWA_ERR_INVALID_ARG;
        if ((int64_t)total_q > (int64_t)n_seqs * max_q_len) return HSWA_ERR_INVALID_ARG;
        const int64_t staged_pages = (int64_t)n_seqs * l.per_seq;
        if (staged_pages * c.n_kv_heads * kP >= (1ll << 31)) return HSWA_ERR_UNSUPPORTED;
        StageArgs sa;
        sa.bt = d_bt;
        sa.prefix = d_prefix_len;
        sa.q_start = d_q_start;
        sa.k_codes = static_cast<const uint8_t *>(layer->k_pool);
        sa.v_codes = static_cast<const uint8_t *>(layer->v_pool);
        sa.k_scale = layer->k_scale;
        sa.v_scale = layer->v_scale;
        uint8_t *base = static_cast<uint8_t *>(ws);
        sa.stage_bt = reinterpret_cast<int32_t *>(base);
        sa.k_out = reinterpret_cast<__half *>(base + l.k_off);
        sa.v_out = reinterpret_cast<__half *>(base + l.v_off);
        sa.n_seqs = n_seqs;
        sa.bt_stride = c.max_pages_per_seq;
        sa.hkv = c.n_kv_heads;
        sa.window = window;
        sa.num_pages = num_pages;
        sa.per_seq = l.per_seq;
        sa.err = error_word();
        __half *q16 = reinterpret_cast<__half *>(base + l.q_off);
        const int64_t n8 = (int64_t)total_q * c.n_q_heads * kD / 8;
        set_last_kernel("prefill_stage_fp8+prefill_tc_bf16_d128<f16>");
        prefill_stage_fp8<<<dim3(c.max_pages_per_seq, n_seqs), 256, 0, st>>>(sa);
        prefill_q_to_f16<<<(int)std::min<int64_t>((n8 + 255) / 256, 4096), 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(q), q16, n8);
        if (cudaGetLastError() != cudaSuccess) return HSWA_ERR_CUDA;
        return launch_prefill_tc(c, window, sa.k_out, sa.v_out, true, (int32_t)staged_pages, sa.stage_bt, q16, o,
                                 d_prefix_len, d_q_start, n_seqs, total_q, max_q_len, scale, st);
    }
    if (!prefill_fast_ok(pool, layer, q, o))
        return launch_attention_generic(pool, layer, q, o, d_bt, nullptr, d_prefix_len, d_q_start, max_q_len,
                                        n_seqs, scale, 1, st);
    set_last_kernel("prefill_tc_bf16_d128");
    return launch_prefill_tc(c, window, layer->k_pool, layer->v_pool, false, num_pages, d_bt, q, o, d_prefix_len,
                             d_q_start, n_seqs, total_q, max_q_len, scale, st);
}

extern "C" int hswa_prefill_chunk(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                                  const int32_t *d_bt, const int32_t *d_prefix_len, const int32_t *d_q_start,
                                  int n_seqs, int total_q, int max_q_len, float scale, hswa_stream_t stream) {
    return hswa_prefill_chunk_ws(pool, layer, q, o, d_bt, d_prefix_len, d_q_start, n_seqs, total_q, max_q_len, scale,
                                 nullptr, 0, stream);
}
