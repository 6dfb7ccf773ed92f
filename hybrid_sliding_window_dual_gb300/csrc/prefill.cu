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
//   * Warp 9 issues the MMAs of both heads (one thread, the heads in
//     lockstep over each K / V tile) and commits them to mbarriers.
//   * Warps 0-3 and 4-7 own query head A and B: one thread per query row
//     reads its row of S from TMEM, applies the causal / window mask on the
//     tiles that need it, keeps the running max in the log2 domain and only
//     rescales O (in TMEM) when the max grows by more than 2^8, writes P,
//     and at the end normalises its row of O and stores it.
//   * The KV range of a block is clipped to the tiles its rows can see: all
//     of [0, t] for a Full layer, [t - W + 1, t] for an SWA layer.
// SWA layers with W <= 128 run a persistent window kernel instead
// (prefill_swa_tc_d128, below): 64-key pages, two score buffers per head,
// an MMA issuer per head and the pages of a block reused by its head pairs.
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
constexpr uint32_t kStageBytes = 32 * 128;  // per warp: two buffers of 32 rows x 32 columns of O, bf16

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
    int32_t nqb;      // 128-row blocks per sequence in the grid
    int32_t lpt;      // 1: sequences ranked longest first
    int32_t kv_rows;  // rows of the pool tensor map (OOB row = zero fill)
    float scale_log2;
    int *err;
};

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two fp32 values (bit patterns) times inv2, as a bf16 pair.
__device__ __forceinline__ uint32_t scale_pack_bf16(uint32_t a, uint32_t b, float2 inv2) {
    const float2 y = __fmul2_rn(make_float2(__uint_as_float(a), __uint_as_float(b)), inv2);
    return pack_bf16(y.x, y.y);
}

// O *= alpha for this thread's row (TMEM, warp-wide): the rare lazy
// rescale, kept out of line so the page loop stays small.
__device__ __noinline__ void rescale_o_row(uint32_t t_o, float alpha) {
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

// Out-of-line slow part of a wait: the spin after a first try failed.
__device__ __noinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity, int *err) {
    return mbar_wait(bar, parity, err);
}
__device__ __forceinline__ bool mbar_wait_small(uint64_t *bar, uint32_t parity, int *err) {
    return mbar_try_wait(bar, parity) || mbar_wait_spin(bar, parity, err);
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

// Batches up to this many sequences are scheduled longest first.
constexpr int kLptMaxSeqs = 64;

// The sequence of a given rank when sequences are ordered by their keys
// after the chunk, longest first (ties by index). Warp-wide; n_seqs <= 64.
__device__ __forceinline__ int32_t seq_of_rank(const PrefillArgs &a, int32_t rank) {
    const int lane = threadIdx.x & 31;
    int32_t found = -1;
    for (int i = lane; i < a.n_seqs; i += 32) {
        const int32_t key = a.prefix[i] + a.q_start[i + 1] - a.q_start[i];
        int32_t r = 0;
        for (int j = 0; j < a.n_seqs; ++j) {
            const int32_t kj = a.prefix[j] + a.q_start[j + 1] - a.q_start[j];
            r += (kj > key) || (kj == key && j < i);
        }
        if (r == rank) found = i;
    }
    for (int o = 16; o > 0; o >>= 1) found = max(found, __shfl_xor_sync(0xffffffffu, found, o));
    return found;
}

// The unit of this CTA. The 1-D grid runs through (sequence rank, block,
// head pair) with the head pair fastest, so the pairs of one kv head run
// side by side and share its K / V tiles in L2; sequences come longest
// first and each sequence's blocks last row first, so the hardware hands
// the longest units out first and the short ones fill the tail.
__device__ __forceinline__ bool make_unit(const PrefillArgs &a, Unit &u, int32_t seq) {
    const int32_t n_hp = a.hq / 2;
    int64_t lin = blockIdx.x;
    u.hp = (int32_t)(lin % n_hp);
    lin /= n_hp;
    u.qb = a.nqb - 1 - (int32_t)(lin % a.nqb);
    u.s = seq;
    if (u.s < 0) return false;
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
        if (!mbar_wait_small(&sm.kv_empty[slot], ((i / kSlots) & 1) ^ 1, a.err) || *(volatile int32_t *)&sm.abort) {
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
    for (int i = max(0, issued - kSlots); i < issued; ++i) mbar_wait_small(&sm.kv_full[i % kSlots], (i / kSlots) & 1, a.err);
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
    bool ok = mbar_wait_small(&sm.q_full, 0, a.err);
    tc_fence_after();
    const int n = u.n_tiles;
    if (ok && n > 0) {
        ok = mbar_wait_small(&sm.kv_full[0], 0, a.err);  // K(0)
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
            ok = mbar_wait_small(&sm.kv_full[sv], (iv / kSlots) & 1, a.err) && mbar_wait_small(&sm.p_full[0], j & 1, a.err) &&
                 !*(volatile int32_t *)&sm.abort;
            if (!ok) break;
            tc_fence_after();
            const uint64_t vd = sdesc(smem_u32(sm.kv[sv]), kHalfBytes, 1024);
            issue_pv<kF16>(to0, ts0, vd, j == 0);
            const bool more = j + 1 < n;
            uint64_t kd = 0;
            if (more) {
                ok = mbar_wait_small(&sm.kv_full[sk], (ik / kSlots) & 1, a.err);
                if (!ok) break;
                tc_fence_after();
                kd = sdesc(smem_u32(sm.kv[sk]), 16, 1024);
                issue_s<kF16>(ts0, qd0, kd);
                mma_commit(&sm.s_full[0]);
            }
            ok = mbar_wait_small(&sm.p_full[1], j & 1, a.err) && !*(volatile int32_t *)&sm.abort;
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

// One S tile of one query row (this thread's TMEM lane): mask on the raw
// scores where the tile needs it (keys past t, or before t - W + 1), update
// the running max (log2 units) and sum, write P over the start of S, and
// rescale O in TMEM when the max grows by more than 2^8. TMEM loads and
// stores are warp-wide: every lane of the warp calls this.

template <bool kF16>
__device__ __forceinline__ void softmax_tile(uint32_t t_s, uint32_t t_o, int32_t k0, int32_t t, int32_t t_min,
                                             int32_t t_max, int32_t W, float scale_log2, bool first_tile,
                                             float &m_used, float &l) {
    // S row in four 32-column chunks; each load overlaps the mask and max
    // work of the chunk before it
    uint32_t sr[4][32];
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
    const float mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3])) * scale_log2;
    // A new reference max only when the row max grows by more than 2^8;
    // then O (nothing before the first PV) and l are rescaled.
    const bool need = mx > m_used + kRescaleLog2;
    const bool resc = need && !first_tile && m_used != -INFINITY;
    const float alpha = resc ? fast_exp2(m_used - mx) : 1.f;
    if (need) m_used = mx;
    const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
    const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(neg_m, neg_m);
    float2 sums[4];  // one running sum per chunk (chains of 16, not 64)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float2 &sum2 = sums[c];
        sum2 = make_float2(0.f, 0.f);
        // P = 2^(s * scale - m) two keys at a time (packed f32x2 FMA and
        // add), packed to 16-bit pairs in place, then its 16 columns (32
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
    // then); the whole warp takes this path when any of its rows needs it
    // (the others scale by 1)
    if (__any_sync(0xffffffffu, resc)) rescale_o_row(t_o, alpha);
    const float2 s01 = __fadd2_rn(sums[0], sums[1]), s23 = __fadd2_rn(sums[2], sums[3]);
    const float2 sum2 = __fadd2_rn(s01, s23);
    l = l * alpha + (sum2.x + sum2.y);
    tmem_wait_st();
}

// One 64-key page of a window block's S (SWA layer): this lane's row t sees
// keys [t - W + 1, t] and the warp's rows are t_first..t_last. A 32-key
// chunk that no row of the warp sees is neither loaded into the max nor
// exponentiated (its P is 0), and only a chunk that some row sees in part is
// masked key by key: with blocks on 128-key boundaries a warp sees five of
// the eight chunks of a block's four pages, two of them in part. A page's scores
// can be ready while the PV of the page before still runs, so a rescale of
// O first waits for that PV (phase pv_par of pv_bar). False when that wait
// gave up (the warp agrees).
template <bool kF16>
__device__ __forceinline__ bool softmax_page_band(uint32_t t_s, uint32_t t_o, int32_t k0, int32_t t, int32_t t_first,
                                                  int32_t t_last, int32_t W, float scale_log2, bool first_page,
                                                  float &m_used, float &l, uint64_t *pv_bar, uint32_t pv_par,
                                                  int *err) {
    uint32_t sr[2][32];
    const int32_t c_lo = max(0, (t_first - W + 1 - k0) >> 5), c_hi = min(1, (t_last - k0) >> 5);
    const int32_t lo_c = t - W + 1 - k0;  // keys c of the page with lo_c <= c <= lo_c + W - 1
    float mc[2];
    tmem_ld32(t_s, sr[0]);
    tmem_wait_ld(sr[0]);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        if (c == 0) tmem_ld32(t_s + 32, sr[1]);
        mc[c] = -INFINITY;
        if (c_lo <= c && c <= c_hi) {  // the same for every lane
            const bool full = k0 + 32 * c >= t_last - W + 1 && k0 + 32 * c + 31 <= t_first;
            if (!full) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if ((uint32_t)(c * 32 + i - lo_c) > (uint32_t)(W - 1)) sr[c][i] = __float_as_uint(-INFINITY);
            }
            float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                m0 = max3(m0, __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
                m1 = max3(m1, __uint_as_float(sr[c][i + 2]), __uint_as_float(sr[c][i + 3]));
            }
            mc[c] = fmaxf(m0, m1);
        }
        if (c == 0) tmem_wait_ld(sr[1]);
    }
    const float mx = fmaxf(mc[0], mc[1]) * scale_log2;
    const bool need = mx > m_used + kRescaleLog2;
    const bool resc = need && !first_page && m_used != -INFINITY;
    const float alpha = resc ? fast_exp2(m_used - mx) : 1.f;
    if (need) m_used = mx;
    const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
    const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(neg_m, neg_m);
    float2 sums[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        float2 &sum2 = sums[c];
        sum2 = make_float2(0.f, 0.f);
        if (c_lo <= c && c <= c_hi) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 x = __ffma2_rn(
                    make_float2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), sc2, nm2);
                const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                sum2 = __fadd2_rn(sum2, p);
                sr[c][i] = kF16 ? pack_f16(p.x, p.y) : pack_bf16(p.x, p.y);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) sr[c][i] = 0u;  // no row of the warp sees these keys
        }
        tmem_st16(t_s + 16 * c, sr[c]);
    }
    bool ok = true;
    if (__any_sync(0xffffffffu, resc)) {
        ok = __all_sync(0xffffffffu, mbar_wait_small(pv_bar, pv_par, err));
        tc_fence_after();
        if (ok) rescale_o_row(t_o, alpha);
    }
    const float2 sum2 = __fadd2_rn(sums[0], sums[1]);
    l = l * alpha + (sum2.x + sum2.y);
    tmem_wait_st();
    return ok;
}

// Normalise this thread's row of O (TMEM) by 1 / l and store it as bf16 at
// dst (when valid; the TMEM loads are warp-wide, every lane calls this).
__device__ __noinline__ void store_o_row(uint32_t t_o, float l, __nv_bfloat16 *dst_row, bool valid) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(t_o + 32 * c, ov);
        tmem_wait_ld(ov);
        if (valid) {
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

__device__ __forceinline__ void store_o_row_inl(uint32_t t_o, float l, __nv_bfloat16 *dst_row, bool valid) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(t_o + 32 * c, ov);
        tmem_wait_ld(ov);
        if (valid) {
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

// Normalise this thread's row of O (TMEM) and write the warp's 32 rows in
// four 32-column quarters through two 2 KB shared-memory buffers (64-byte
// swizzle) and TMA stores: a buffer is refilled once the store before the
// last has read it, so the stores overlap the packing of the next quarter
// and the writes reach memory as whole 64-byte row pieces. A warp with rows
// past the block's end stores its valid rows from registers.
__device__ __forceinline__ void store_o_rows_staged(uint32_t t_o, float l, uint8_t *stage, const CUtensorMap *to,
                                                    int32_t head, int32_t row_first, bool full_warp,
                                                    __nv_bfloat16 *dst_row, bool valid) {
    if (!full_warp) {
        store_o_row(t_o, l, dst_row, valid);
        return;
    }
    // 1 / l to within 2 ulp (the row is rounded to bf16 after the multiply)
    const float inv = l > 0.f ? __fdividef(1.f, l) : 0.f;
    const float2 inv2 = make_float2(inv, inv);
    const int lane = threadIdx.x & 31;
    uint32_t ov[2][32];
    auto put = [&](int qt, const uint32_t (&v)[32]) {
        uint8_t *buf = stage + (qt & 1) * (kStageBytes / 2);
        if (lane == 0) bulk_wait_read<1>();  // the buffer's previous store has read it
        __syncwarp();
        uint8_t *row = buf + lane * 64;
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // 16-byte chunk j: columns 8j .. 8j + 7 of the quarter
            uint4 w;
            w.x = scale_pack_bf16(v[8 * j + 0], v[8 * j + 1], inv2);
            w.y = scale_pack_bf16(v[8 * j + 2], v[8 * j + 3], inv2);
            w.z = scale_pack_bf16(v[8 * j + 4], v[8 * j + 5], inv2);
            w.w = scale_pack_bf16(v[8 * j + 6], v[8 * j + 7], inv2);
            *reinterpret_cast<uint4 *>(row + ((j ^ ((lane >> 1) & 3)) << 4)) = w;
        }
        fence_proxy_async_shared();  // the buffer is read by the TMA store
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(to, buf, qt * 32, head, row_first);
            bulk_commit();
        }
    };
    tmem_ld32(t_o, ov[0]);
    tmem_ld32(t_o + 32, ov[1]);
    tmem_wait_ld(ov[0]);
    tmem_wait_ld(ov[1]);
    put(0, ov[0]);
    tmem_ld32(t_o + 64, ov[0]);
    put(1, ov[1]);
    tmem_ld32(t_o + 96, ov[1]);
    tmem_wait_ld(ov[0]);
    tmem_wait_ld(ov[1]);
    put(2, ov[0]);
    put(3, ov[1]);
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
    float m_used = -INFINITY, l = 0.f;  // running max (log2 units) and sum of P
    bool ok = true;
    for (int j = 0; j < u.n_tiles; ++j) {
        ok = mbar_wait_small(&sm.s_full[x], j & 1, a.err) && !*(volatile int32_t *)&sm.abort;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        softmax_tile<kF16>(t_s, t_o, (u.tile_lo + j) * kBN, t, t_min, t_max, a.window, a.scale_log2, j == 0, m_used,
                           l);
        tc_fence_before();
        mbar_arrive(&sm.p_full[x]);
    }
    // epilogue: wait for the last PV (always: TMEM is freed after this
    // function returns), normalise this row of O and store it
    const bool fin = mbar_wait_small(&sm.o_final[x], 0, a.err);
    ok = __all_sync(0xffffffffu, ok && fin);
    if (!ok) {
        sm.abort = 1;
        return;
    }
    tc_fence_after();
    const int h = 2 * u.hp + x;
    store_o_row_inl(t_o, l, a.o + ((int64_t)(u.row0 + r) * a.hq + h) * kD, r < u.n_rows);
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_bf16_d128(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, PrefillArgs a) {
    __shared__ int32_t unit_seq;
    if (threadIdx.x < 32) {
        const int32_t rank = (int32_t)(blockIdx.x / ((int64_t)(a.hq / 2) * a.nqb));
        const int32_t seq = a.lpt ? seq_of_rank(a, rank) : rank;
        if (threadIdx.x == 0) unit_seq = seq;
    }
    __syncthreads();
    Unit u;
    if (!make_unit(a, u, unit_seq)) return;
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

// ------------------------------------------ SWA layers: persistent CTAs
// Sliding-window layers with W <= 128 ("MiMo-V2.5 Series Inference
// Full-Link Optimization", Sec. 1.1: an SWA query attends only to the last W
// tokens). A block of query rows at positions [128 m, 128 m + 128) sees keys
// [128 m - W + 1, 128 m + 127]: the 64-key pages 2m - 2 .. 2m + 1, never
// more (fewer when the block is partial or its first key is past a page
// start). Blocks are cut at these absolute boundaries (a chunk's first and
// last block may be partial) and each CTA is persistent, one per SM, walking
// a contiguous share of the unit list
//     for each sequence, for each kv head g, for each block m,
//         for each pair of query heads of g
// so the head pairs of one block reuse its four K / V pages and the next
// block reuses pages 2m and 2m + 1: a page is loaded into shared memory once
// per CTA that needs it. The scores of a head are computed one page at a
// time into two alternating TMEM buffers, so the QK of the next page runs
// while the softmax works on this one. TMEM, barriers and the ring are set
// up once per CTA; a head's next queries load as soon as its last QK MMA of
// the current unit is done, and O leaves through a per-warp shared-memory
// stage and TMA stores. Warps 0-7 softmax (two heads), warp 8 lane 0 loads
// Q and lane 1 loads K / V, warps 9 and 10 issue head A's and head B's MMAs.

constexpr int kQBufs = 2;
constexpr int kDescs = 4;
constexpr int kSwaThreads = kThreads + 32;  // warp 10: head B's MMA issuer

// What the softmax warps need of a unit (written by the Q loader).
struct SwaDesc {
    int32_t p0, n_rows, row0, lo, hi, hp;
};

constexpr uint32_t kPgBytes = kP * kD * 2;  // one K or V page of one kv head: [d half][64 keys][128 B]
constexpr int kPgSlots = 8;                  // K and V of the last four pages

struct SwaSmem {
    uint8_t q[kQBufs][kTileBytes];     // Q of one head: [d half][128 rows][128 B]
    uint8_t kv[kPgSlots][kPgBytes];    // K or V pages: [d half][64 keys][128 B]
    uint8_t ostage[8][kStageBytes];    // per softmax warp: O rows on their way out
    uint64_t q_full[kQBufs], q_empty[kQBufs];
    uint64_t kv_full[kPgSlots], kv_empty[kPgSlots];
    uint64_t s_full[2][2], p_full[2][2];  // [head][S buffer]
    uint64_t pv_done[2], o_final[2], mma_done[2];
    uint64_t desc_full[kDescs], desc_empty[kDescs];
    SwaDesc desc[kDescs];
    uint32_t tmem_base;
    int32_t abort;
    int32_t start_seq, start_off, n_units;  // this CTA's share of the unit list
};
static_assert(offsetof(SwaSmem, kv) % 1024 == 0, "128-byte swizzled tiles need 1024-byte alignment");
static_assert(offsetof(SwaSmem, ostage) % 1024 == 0, "128-byte swizzled tiles need 1024-byte alignment");
constexpr size_t kSwaSmemBytes = sizeof(SwaSmem) + 1024;
static_assert(kSwaSmemBytes <= 232448, "one CTA per SM must fit");

// Units (blocks x kv heads x head pairs) of sequence s.
__device__ __forceinline__ int32_t swa_seq_units(const PrefillArgs &a, int32_t s, int32_t pairs) {
    const int32_t pre = a.prefix[s], n = a.q_start[s + 1] - a.q_start[s];
    if (n <= 0) return 0;
    return ((pre + n - 1) / kBM - pre / kBM + 1) * a.hkv * pairs;
}

// Warp 0: this CTA's share [c U / G, (c + 1) U / G) of the U units of all
// sequences, as (first sequence, unit within it, count).
__device__ void swa_partition(SwaSmem &sm, const PrefillArgs &a, int32_t pairs) {
    const int lane = threadIdx.x & 31;
    int64_t total = 0;
    for (int32_t base = 0; base < a.n_seqs; base += 32) {
        const int32_t i = base + lane;
        int64_t u = i < a.n_seqs ? swa_seq_units(a, i, pairs) : 0;
        for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
        total += u;
    }
    const int64_t u0 = total * blockIdx.x / gridDim.x, u1 = total * (blockIdx.x + 1) / gridDim.x;
    int64_t before = 0, off = 0;
    int32_t s0 = -1;
    for (int32_t base = 0; base < a.n_seqs && s0 < 0; base += 32) {
        const int32_t i = base + lane;
        const int64_t u = i < a.n_seqs ? swa_seq_units(a, i, pairs) : 0;
        int64_t inc = u;
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        const int64_t excl = before + inc - u;
        const unsigned hit = __ballot_sync(0xffffffffu, u > 0 && excl <= u0 && u0 < excl + u);
        if (hit) {
            const int src = __ffs(hit) - 1;
            s0 = base + src;
            off = __shfl_sync(0xffffffffu, u0 - excl, src);
        }
        before += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
        sm.start_seq = s0;
        sm.start_off = (int32_t)off;
        sm.n_units = (s0 >= 0 && u1 > u0) ? (int32_t)(u1 - u0) : 0;
    }
}

// Walk over the unit list; every role walks it the same way.
struct SwaWalk {
    int32_t s, g, m, hpi, left;
    int32_t pre, n, q0, m_lo, m_hi;

    __device__ void seq(const PrefillArgs &a) {
        q0 = a.q_start[s];
        n = a.q_start[s + 1] - q0;
        pre = a.prefix[s];
        m_lo = pre / kBM;
        m_hi = n > 0 ? (pre + n - 1) / kBM : m_lo - 1;
    }
    __device__ void start(const PrefillArgs &a, const SwaSmem &sm, int32_t pairs) {
        s = sm.start_seq;
        left = sm.n_units;
        seq(a);
        const int32_t nb = m_hi - m_lo + 1, off = sm.start_off;
        g = off / (nb * pairs);
        const int32_t r = off - g * nb * pairs;
        m = m_lo + r / pairs;
        hpi = r % pairs;
    }
    __device__ void next(const PrefillArgs &a, int32_t pairs) {
        if (--left <= 0) return;
        if (++hpi < pairs) return;
        hpi = 0;
        if (++m <= m_hi) return;
        m = m_lo;
        if (++g < a.hkv) return;
        g = 0;
        do {
            if (++s >= a.n_seqs) {  // the share ran past the last unit: stop
                left = 0;
                return;
            }
            seq(a);
        } while (m_hi < m_lo);
        m = m_lo;
    }
};

struct SwaBlock {
    int32_t s, g, hp;              // sequence, kv head, pair of query heads
    int32_t p0, n_rows, row0, L;   // first position, rows, first q row, keys after the chunk
    int32_t lo, hi;                // logical pages of keys the block's rows see
    int32_t first_page, last_page; // logical pages its rows can see
    int64_t tile_base;             // identity of page 0 of (s, g)
};

__device__ __forceinline__ SwaBlock swa_block(const SwaWalk &w, const PrefillArgs &a, int32_t pairs) {
    SwaBlock b;
    b.s = w.s;
    b.g = w.g;
    b.hp = w.g * pairs + w.hpi;
    b.p0 = max(w.pre, w.m * kBM);
    const int32_t p_end = min(w.pre + w.n, (w.m + 1) * kBM);
    b.n_rows = p_end - b.p0;
    b.row0 = w.q0 + (b.p0 - w.pre);
    b.L = w.pre + w.n;
    const int32_t key_lo = max(0, b.p0 - a.window + 1);
    b.lo = key_lo / kP;
    b.hi = (p_end - 1) / kP;
    b.first_page = key_lo / kP;
    b.last_page = (b.L - 1) / kP;
    b.tile_base = ((int64_t)b.s * a.hkv + b.g) << 32;
    return b;
}

// The K / V pages in the ring: the last four placed, K and V of placement p
// being loads 2p and 2p + 1 in slots (2p) % 8 and (2p + 1) % 8. A block
// needs at most four pages (W <= 128: keys [128 m - 127, 128 m + 127]),
// consecutive and later than those of the blocks before it in its (sequence,
// kv head), so the page a placement replaces is never one the block needs.
// The loader and the MMA issuers make the same calls in the same order and
// agree on every load index.
struct PageRing {
    int64_t id0, id1, id2, id3;  // page of placement p sits in entry p % 4 (-1: none)
    int32_t next;                // placements so far

    __device__ void init() {
        id0 = id1 = id2 = id3 = -1;
        next = 0;
    }
    // Load index of page pid's K, or -1 when it is not in the ring.
    __device__ int32_t find(int64_t pid) const {
        const int32_t e = id0 == pid ? 0 : id1 == pid ? 1 : id2 == pid ? 2 : id3 == pid ? 3 : -1;
        return e < 0 ? -1 : 2 * (next - 1 - ((next - 1 - e) & 3));
    }
    __device__ int32_t place(int64_t pid) {
        const int32_t p = next++;
        switch (p & 3) {
            case 0: id0 = pid; break;
            case 1: id1 = pid; break;
            case 2: id2 = pid; break;
            default: id3 = pid; break;
        }
        return 2 * p;
    }
};

__device__ void swa_load_q(SwaSmem &sm, const CUtensorMap *tq, const PrefillArgs &a, int32_t pairs) {
    prefetch_tmap(tq);
    SwaWalk w;
    w.start(a, sm, pairs);
    int32_t issued = 0;
    for (int32_t ub = 0; ub < sm.n_units; ++ub) {
        const SwaBlock b = swa_block(w, a, pairs);
        // the unit's descriptor for the softmax warps; its slot was freed
        // (all 256 softmax threads arrived) when unit ub - 4 was stored
        const int dslot = ub % kDescs;
        bool ok = ub < kDescs || (mbar_wait_small(&sm.desc_empty[dslot], ((ub / kDescs) + 1) & 1, a.err) &&
                                  !*(volatile int32_t *)&sm.abort);
        if (ok) {
            SwaDesc &d = sm.desc[dslot];
            d.p0 = b.p0;
            d.n_rows = b.n_rows;
            d.row0 = b.row0;
            d.lo = b.lo;
            d.hi = b.hi;
            d.hp = b.hp;
            mbar_arrive(&sm.desc_full[dslot]);  // release: the fields are visible to the waiters
        }
        for (int x = 0; x < 2 && ok; ++x) {
            const int32_t qi = 2 * ub + x, slot = qi % kQBufs;
            // the buffer's previous item (qi - kQBufs) has been read by its
            // last QK MMA; parity waits stay at most one phase behind
            // because each item waits for the release of the one before
            if (qi >= kQBufs)
                ok = mbar_wait_small(&sm.q_empty[slot], ((qi / kQBufs) + 1) & 1, a.err) &&
                     !*(volatile int32_t *)&sm.abort;
            if (!ok) break;
            mbar_arrive_expect_tx(&sm.q_full[slot], kTileBytes);
            for (int dh = 0; dh < 2; ++dh)
                tma_load_3d(sm.q[slot] + dh * kHalfBytes, tq, dh * 64, 2 * b.hp + x, b.row0, &sm.q_full[slot]);
            ++issued;
        }
        if (!ok) {
            sm.abort = 1;
            break;
        }
        w.next(a, pairs);
    }
    // drain: never leave copies landing in shared memory after the CTA ends
    for (int32_t i = max(0, issued - kQBufs); i < issued; ++i)
        mbar_wait_small(&sm.q_full[i % kQBufs], (i / kQBufs) & 1, a.err);
}

__device__ void swa_load_kv(SwaSmem &sm, const CUtensorMap *tk, const CUtensorMap *tv, const PrefillArgs &a,
                            int32_t pairs) {
    prefetch_tmap(tk);
    prefetch_tmap(tv);
    SwaWalk w;
    w.start(a, sm, pairs);
    PageRing ring;
    ring.init();
    int32_t issued = 0;
    bool ok = true;
    for (int32_t ub = 0; ok && ub < sm.n_units; ++ub) {
        const SwaBlock b = swa_block(w, a, pairs);
        const int32_t *btrow = a.bt + (int64_t)b.s * a.bt_stride;
        for (int32_t lp = b.lo; ok && lp <= b.hi; ++lp) {
            if (ring.find(b.tile_base + lp) >= 0) continue;  // still in the ring
            const int32_t k = ring.place(b.tile_base + lp);
            // a page outside the block's view (an older window page, maybe
            // released, or past the sequence) fills with zeros
            int32_t row = a.kv_rows;
            if (lp >= b.first_page && lp <= b.last_page) {
                const int32_t page = lp < a.bt_stride ? btrow[lp] : -1;
                if (page >= 0 && page < a.num_pages)
                    row = (page * a.hkv + b.g) * kP;
                else
                    set_error(a.err, HSWA_ERR_BOUNDS);
            }
            for (int kv = 0; kv < 2; ++kv) {
                const int32_t i = k + kv;
                const int slot = i % kPgSlots;
                // the slot's previous load (i - 8) belongs to a page no
                // later block of this CTA needs; both issuers released it
                if (i >= kPgSlots)
                    ok = mbar_wait_small(&sm.kv_empty[slot], ((i / kPgSlots) + 1) & 1, a.err) &&
                         !*(volatile int32_t *)&sm.abort;
                if (!ok) break;
                mbar_arrive_expect_tx(&sm.kv_full[slot], kPgBytes);
                for (int dh = 0; dh < 2; ++dh)
                    tma_load_2d(sm.kv[slot] + dh * kBoxBytes, kv ? tv : tk, dh * 64, row, &sm.kv_full[slot]);
                ++issued;
            }
        }
        w.next(a, pairs);
    }
    if (!ok) sm.abort = 1;
    for (int32_t i = max(0, issued - kPgSlots); i < issued; ++i)
        mbar_wait_small(&sm.kv_full[i % kPgSlots], (i / kPgSlots) & 1, a.err);
}

// S = Q K^T for one 64-key page: 8 steps of K = 16 over d (the Q tile's d
// halves are 16 KB apart, the page's 8 KB).
template <bool kF16>
__device__ __forceinline__ void issue_s_page(uint32_t t_s, uint64_t qd, uint64_t kd) {
    constexpr uint32_t kIdesc = idesc_16(kBM, kP, false, kF16);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ss(t_s, qd + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4),
               kd + (((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4), kIdesc, kk > 0);
}

// O += P V over one 64-key page: 4 steps of K = 16 keys; P (16-bit pairs)
// sits in the first 32 columns of the S buffer, V is MN-major (d
// contiguous) with the page's two 64-column halves 8 KB apart.
template <bool kF16>
__device__ __forceinline__ void issue_pv_page(uint32_t t_o, uint32_t t_p, uint64_t vd, bool first) {
    constexpr uint32_t kIdesc = idesc_16(kBM, kD, true, kF16);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ts(t_o, t_p + kk * 8, vd + kk * (2048 >> 4), kIdesc, (first && kk == 0) ? 0u : 1u);
}

// One MMA issuer per query head (warp 9: head A, warp 10: head B), each
// walking the units in order and waiting only on its own head's barriers.
// A head has two 64-column S buffers, so the scores of page j + 1 are
// computed while the softmax works on page j:
//   QK(0) QK(1) | PV(0) QK(2) | PV(1) QK(3) | PV(2) | PV(3)
// QK(j + 2) reuses page j's buffer once PV(j) has read its P (MMAs of one
// thread run in issue order). A K / V slot is released once both heads'
// last uses of it have completed (kv_empty counts a commit from each
// issuer).
template <bool kF16>
__device__ void swa_mma(SwaSmem &sm, const PrefillArgs &a, int32_t pairs, int x) {
    const uint32_t ts0 = sm.tmem_base + 128 * x, to = sm.tmem_base + 256 + 128 * x;
    const uint64_t qd = sdesc(smem_u32(sm.q[x]), 16, 1024);  // one Q buffer per head
    SwaWalk w;
    w.start(a, sm, pairs);
    PageRing ring;
    ring.init();
    int32_t tcount = 0;  // pages so far: S buffer tcount % 2, phase (tcount / 2) & 1
    bool ok = true;
    auto wait_kv = [&](int32_t i) { return mbar_wait_small(&sm.kv_full[i % kPgSlots], (i / kPgSlots) & 1, a.err); };
    for (int32_t ub = 0; ok && ub < sm.n_units; ++ub) {
        const SwaBlock b = swa_block(w, a, pairs);
        SwaWalk nw = w;
        nw.next(a, pairs);
        // pages the next unit needs stay in the ring after this one
        int64_t keep_lo = 0, keep_hi = -1;
        if (ub + 1 < sm.n_units && nw.left > 0) {
            const SwaBlock nb = swa_block(nw, a, pairs);
            keep_lo = nb.tile_base + nb.lo;
            keep_hi = nb.tile_base + nb.hi;
        }
        const int n = b.hi - b.lo + 1;  // 1 .. 4 pages
        int32_t kidx[4];
        bool fresh[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            kidx[j] = -1;
            fresh[j] = false;
            if (j < n) {
                kidx[j] = ring.find(b.tile_base + b.lo + j);
                fresh[j] = kidx[j] < 0;
                if (fresh[j]) kidx[j] = ring.place(b.tile_base + b.lo + j);
            }
        }
        auto qk = [&](int j) {  // QK of page j into buffer (tcount + j) % 2
            const int32_t ki = kidx[j];
            bool good = !fresh[j] || wait_kv(ki);
            if (good) {
                tc_fence_after();
                issue_s_page<kF16>(ts0 + 64 * ((tcount + j) & 1), qd, sdesc(smem_u32(sm.kv[ki % kPgSlots]), 16, 1024));
                mma_commit(&sm.s_full[x][(tcount + j) & 1]);
                if (j == n - 1) mma_commit(&sm.q_empty[x]);
                const int64_t pid = b.tile_base + b.lo + j;
                if (!(pid >= keep_lo && pid <= keep_hi)) mma_commit(&sm.kv_empty[ki % kPgSlots]);
            }
            return good;
        };
        ok = mbar_wait_small(&sm.q_full[x], ub & 1, a.err) && qk(0) && (n < 2 || qk(1));
        if (!ok) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j >= n) break;
            const int32_t t = tcount + j, vi = kidx[j] + 1;
            ok = (!fresh[j] || wait_kv(vi)) && mbar_wait_small(&sm.p_full[x][t & 1], (t >> 1) & 1, a.err) &&
                 !*(volatile int32_t *)&sm.abort;
            if (!ok) break;
            tc_fence_after();
            issue_pv_page<kF16>(to, ts0 + 64 * (t & 1), sdesc(smem_u32(sm.kv[vi % kPgSlots]), kBoxBytes, 1024),
                                j == 0);
            mma_commit(&sm.pv_done[x]);
            const int64_t pid = b.tile_base + b.lo + j;
            if (!(pid >= keep_lo && pid <= keep_hi)) mma_commit(&sm.kv_empty[vi % kPgSlots]);
            if (j + 2 < n) {
                ok = qk(j + 2);
                if (!ok) break;
            }
            if (j == n - 1) mma_commit(&sm.o_final[x]);  // the head's O is final once this completes
        }
        if (!ok) break;
        tcount += n;
        w = nw;
    }
    if (!ok) sm.abort = 1;
    // every MMA issued above has completed before the TMEM is freed
    mma_commit(&sm.mma_done[x]);
    mbar_wait_small(&sm.mma_done[x], 0, a.err);
}

template <bool kF16>
__device__ void swa_softmax(SwaSmem &sm, const CUtensorMap *to, const PrefillArgs &a, int x) {
    const int warp = (threadIdx.x >> 5) & 3;
    const int r = warp * 32 + (threadIdx.x & 31);  // query row of this thread
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_s = sm.tmem_base + lane_off + 128 * x;  // O of the head sits 256 columns on
    uint8_t *stage = sm.ostage[threadIdx.x >> 5];
    int32_t tcount = 0;
    for (int32_t ub = 0; ub < sm.n_units; ++ub) {
        const int dslot = ub % kDescs;
        bool ok = mbar_wait_small(&sm.desc_full[dslot], (ub / kDescs) & 1, a.err);
        if (!__all_sync(0xffffffffu, ok)) {
            sm.abort = 1;
            break;
        }
        // the slot stays ours until this unit's O is stored, so fields
        // needed only then are read then
        const SwaDesc &d = sm.desc[dslot];
        const int32_t lo = d.lo, hi = d.hi;
        const int32_t last = d.n_rows - 1;  // rows past the block repeat its last row
        const int32_t t = d.p0 + min(r, last);
        const int32_t t_first = d.p0 + min(warp * 32, last), t_last = d.p0 + min(warp * 32 + 31, last);
        float m_used = -INFINITY, l = 0.f;
        for (int32_t pg = lo; pg <= hi; ++pg, ++tcount) {
            // S of this page in buffer tcount % 2: the MMA thread writes
            // that buffer again only after this page's P has been read, so
            // the wait is never two phases behind
            const int buf = tcount & 1;
            ok = mbar_wait_small(&sm.s_full[x][buf], (tcount >> 1) & 1, a.err) && !*(volatile int32_t *)&sm.abort;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            ok = softmax_page_band<kF16>(t_s + 64 * buf, t_s + 256, pg * kP, t, t_first, t_last, a.window,
                                         a.scale_log2, pg == lo, m_used, l, &sm.pv_done[x], (tcount - 1) & 1, a.err);
            if (!ok) break;
            tc_fence_before();
            mbar_arrive(&sm.p_full[x][buf]);
        }
        const bool fin = ok && mbar_wait_small(&sm.o_final[x], ub & 1, a.err);
        if (!__all_sync(0xffffffffu, fin)) {
            sm.abort = 1;
            break;
        }
        tc_fence_after();
        // O is read before this thread reports the next unit's first P, and
        // the first PV of the next unit (which overwrites O) waits for that P
        const int32_t h = 2 * d.hp + x;
        store_o_rows_staged(t_s + 256, l, stage, to, h, d.row0 + warp * 32, warp * 32 + 31 <= last,
                            a.o + ((int64_t)(d.row0 + r) * a.hq + h) * kD, r <= last);
        mbar_arrive(&sm.desc_empty[dslot]);
    }
    // the TMA stores are complete before the CTA ends
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
}

template <bool kF16>
__global__ void __launch_bounds__(kSwaThreads, 1)
    prefill_swa_tc_d128(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                        PrefillArgs a) {
    extern __shared__ uint8_t raw[];
    SwaSmem &sm = *reinterpret_cast<SwaSmem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int32_t pairs = (a.hq / a.hkv) / 2;
    if (warp == 0) swa_partition(sm, a, pairs);
    __syncthreads();
    if (sm.n_units == 0) return;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kQBufs; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
        }
        for (int i = 0; i < kPgSlots; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 2);  // one commit from each head's issuer
        }
        for (int x = 0; x < 2; ++x) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&sm.s_full[x][b], 1);
                mbar_init(&sm.p_full[x][b], 128);
            }
            mbar_init(&sm.pv_done[x], 1);
            mbar_init(&sm.o_final[x], 1);
        }
        mbar_init(&sm.mma_done[0], 1);
        mbar_init(&sm.mma_done[1], 1);
        for (int i = 0; i < kDescs; ++i) {
            mbar_init(&sm.desc_full[i], 1);
            mbar_init(&sm.desc_empty[i], 256);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 9) tmem_alloc<512>(&sm.tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp < 8) {
        swa_softmax<kF16>(sm, &to, a, warp >> 2);
    } else if (warp == 8) {
        const int lane = threadIdx.x & 31;
        if (lane == 0)
            swa_load_q(sm, &tq, a, pairs);
        else if (lane == 1)
            swa_load_kv(sm, &tk, &tv, a, pairs);
        __syncwarp();
    } else {
        if ((threadIdx.x & 31) == 0) swa_mma<kF16>(sm, a, pairs, warp - 9);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_free<512>(sm.tmem_base);
}

bool prefill_fast_ok(const hswa_pool *pool, const hswa_layer *layer, const void *q, const void *o) {
    const hswa_config &c = pool->cfg;
    const int g = c.n_q_heads / c.n_kv_heads;
    return (c.dtype == HSWA_DTYPE_BF16 || c.dtype == HSWA_DTYPE_FP8_E4M3) && c.head_dim == kD && c.page_size == kP &&
           g % 2 == 0 && ((uintptr_t)q & 15) == 0 && ((uintptr_t)o & 15) == 0 &&
           ((uintptr_t)layer->k_pool & 15) == 0 && ((uintptr_t)layer->v_pool & 15) == 0;
}

// ------------------------------------------------------------ FP8 staging
// Pages per sequence the staging copy can need at most: a Full layer may
// read every logical page; an SWA layer's chunk of at most max_q_len rows
// reads keys [prefix - W + 1, prefix + n), at most W - 1 + max_q_len keys.
int32_t stage_pages_per_seq(const hswa_config &c, const hswa_layer *layer, int max_q_len) {
    if (layer->kind != HSWA_KIND_SWA) return c.max_pages_per_seq;
    const int64_t keys = (int64_t)layer->window - 1 + max_q_len;
    return (int32_t)std::min<int64_t>(c.max_pages_per_seq, (keys + kP - 1) / kP + 1);
}

// Logical pages [lo, hi] of a sequence the chunk reads (hi < lo: none):
// keys [0, prefix + n) for a Full layer, [prefix - W + 1, prefix + n) for an
// SWA layer.
__host__ __device__ __forceinline__ void chunk_pages(int32_t pre, int32_t n, int32_t window, int32_t &lo,
                                                     int32_t &hi) {
    const int32_t lo_key = (window > 0 && pre - window + 1 > 0) ? pre - window + 1 : 0;
    lo = lo_key / kP;
    hi = n > 0 ? (pre + n - 1) / kP : lo - 1;
}

constexpr size_t align1k(size_t x) { return (x + 1023) & ~(size_t)1023; }

// Workspace of an FP8 chunk: the staging block table [n_seqs][bt_stride],
// each sequence's first page copy (a prefix sum over the pages the chunk
// reads, [n_seqs + 1]), the fp16 copy of the q rows, then as many fp16 K
// and V page copies as the rest holds ("capacity"), packed: sequence s's
// pages take copies off[s] .. off[s + 1] - 1.
struct StageLayout {
    size_t page_bytes, off_off, q_off, k_off, v_off;
    int64_t cap;
};

StageLayout stage_layout(const hswa_config &c, int n_seqs, int64_t q_rows, size_t ws_bytes) {
    StageLayout l;
    l.page_bytes = (size_t)c.n_kv_heads * kP * kD * sizeof(__half);
    l.off_off = align1k((size_t)n_seqs * c.max_pages_per_seq * sizeof(int32_t));
    l.q_off = l.off_off + align1k((size_t)(n_seqs + 1) * sizeof(int32_t));
    l.k_off = l.q_off + align1k((size_t)q_rows * c.n_q_heads * kD * sizeof(__half));
    l.cap = ws_bytes > l.k_off ? (int64_t)((ws_bytes - l.k_off) / (2 * l.page_bytes)) : 0;
    l.v_off = l.k_off + (size_t)l.cap * l.page_bytes;
    return l;
}

// Bytes of a workspace holding q_rows query rows and `pages` page copies.
size_t stage_bytes(const hswa_config &c, int n_seqs, int64_t q_rows, int64_t pages) {
    const StageLayout l = stage_layout(c, n_seqs, q_rows, 0);
    return l.k_off + 2 * (size_t)pages * l.page_bytes;
}

struct StageArgs {
    const int32_t *bt, *prefix, *q_start;
    const uint8_t *k_codes, *v_codes;  // [page][Hkv][P][d], V pages [page][Hkv][d][P]
    const float *k_scale, *v_scale;    // [page][Hkv][P] (one 128-element tile per row)
    int32_t *stage_bt;                 // [n_seqs][bt_stride]
    int32_t *stage_off;                // [n_seqs + 1]: first copy of each sequence
    __half *k_out, *v_out;             // [cap][Hkv][P][d]
    int32_t n_seqs, bt_stride, hkv, window, num_pages, cap;
    int *err;
};

// One block: stage_off = prefix sum of the pages each sequence's chunk reads.
__global__ void __launch_bounds__(256) prefill_stage_plan(StageArgs a) {
    __shared__ int32_t part[256];
    const int32_t per = (a.n_seqs + 255) / 256, s0 = threadIdx.x * per;
    int32_t sum = 0;
    for (int32_t s = s0; s < min(a.n_seqs, s0 + per); ++s) {
        int32_t lo, hi;
        chunk_pages(a.prefix[s], a.q_start[s + 1] - a.q_start[s], a.window, lo, hi);
        sum += max(0, hi - lo + 1);
    }
    part[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {  // 256 partial sums: a serial scan is short
        int32_t run = 0;
        for (int i = 0; i < 256; ++i) {
            const int32_t v = part[i];
            part[i] = run;
            run += v;
        }
        a.stage_off[a.n_seqs] = run;
    }
    __syncthreads();
    int32_t run = part[threadIdx.x];
    for (int32_t s = s0; s < min(a.n_seqs, s0 + per); ++s) {
        a.stage_off[s] = run;
        int32_t lo, hi;
        chunk_pages(a.prefix[s], a.q_start[s + 1] - a.q_start[s], a.window, lo, hi);
        run += max(0, hi - lo + 1);
    }
}

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
    int32_t lo_pg, hi_pg;
    chunk_pages(a.prefix[s], a.q_start[s + 1] - a.q_start[s], a.window, lo_pg, hi_pg);
    int32_t page = -1, slot = -1;
    if (j >= lo_pg && j <= hi_pg) {
        page = a.bt[(int64_t)s * a.bt_stride + j];
        const int32_t copy = a.stage_off[s] + (j - lo_pg);
        if (copy >= a.cap) {  // the workspace holds fewer copies than the chunk reads
            if (threadIdx.x == 0) set_error(a.err, HSWA_ERR_BOUNDS);
            page = -1;
        }
        if (page >= 0 && page < a.num_pages) slot = copy;
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
        return cuda_fail(cudaErrorInvalidValue, "prefill tensor maps");
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
    // the kernels' shared-memory opt-in, once per device
    static int full_b[kMaxDevices], full_h[kMaxDevices], swa_b[kMaxDevices], swa_h[kMaxDevices];
    if (kernel_setup(prefill_tc_bf16_d128<false>, kPrefillSmemBytes, kThreads, full_b) < 0 ||
        kernel_setup(prefill_tc_bf16_d128<true>, kPrefillSmemBytes, kThreads, full_h) < 0)
        return cuda_fail(cudaGetLastError(), "prefill_tc_bf16_d128 shared memory");
    if (kernel_setup(prefill_swa_tc_d128<false>, kSwaSmemBytes, kSwaThreads, swa_b) < 0 ||
        kernel_setup(prefill_swa_tc_d128<true>, kSwaSmemBytes, kSwaThreads, swa_h) < 0)
        return cuda_fail(cudaGetLastError(), "prefill_swa_tc_d128 shared memory");
    if (window > 0 && window <= kBN) {
        // at most four 64-key pages per block: the persistent window kernel
        const int sms = sm_count();
        if (sms <= 0) return HSWA_ERR_CUDA;
        CUtensorMap to;
        if (!make_tmap_3d(&to, o, kD, c.n_q_heads, (uint64_t)total_q, 32, 1, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          CU_TENSOR_MAP_SWIZZLE_64B))
            return cuda_fail(cudaErrorInvalidValue, "prefill output tensor map");
        const int64_t units = (int64_t)n_seqs * ((max_q_len + kBM - 1) / kBM + 1) * (c.n_q_heads / 2);
        const dim3 grid((unsigned)std::min<int64_t>(sms, units));
        if (f16)
            prefill_swa_tc_d128<true><<<grid, kSwaThreads, kSwaSmemBytes, st>>>(tq, tk, tv, to, a);
        else
            prefill_swa_tc_d128<false><<<grid, kSwaThreads, kSwaSmemBytes, st>>>(tq, tk, tv, to, a);
        const cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? HSWA_OK : cuda_fail(e, "prefill_swa_tc_d128 launch");
    }
    a.nqb = (max_q_len + kBM - 1) / kBM;
    a.lpt = n_seqs <= kLptMaxSeqs;
    const int64_t units = (int64_t)n_seqs * a.nqb * (c.n_q_heads / 2);
    if (units >= (1ll << 31)) return HSWA_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)units);
    if (f16)
        prefill_tc_bf16_d128<true><<<grid, kThreads, kPrefillSmemBytes, st>>>(tq, tk, tv, a);
    else
        prefill_tc_bf16_d128<false><<<grid, kThreads, kPrefillSmemBytes, st>>>(tq, tk, tv, a);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? HSWA_OK : cuda_fail(e, "prefill_tc_bf16_d128 launch");
}

}  // namespace
}  // namespace hswa

using namespace hswa;

extern "C" size_t hswa_prefill_workspace_size(const hswa_pool *pool, const hswa_layer *layer, int n_seqs,
                                              int max_q_len) {
    if (!pool || !layer || n_seqs < 0 || max_q_len < 0 || pool->cfg.dtype != HSWA_DTYPE_FP8_E4M3) return 0;
    if (layer->kind == HSWA_KIND_SWA && layer->window <= 0) return 0;
    return stage_bytes(pool->cfg, n_seqs, (int64_t)n_seqs * max_q_len,
                       (int64_t)n_seqs * stage_pages_per_seq(pool->cfg, layer, max_q_len));
}

extern "C" size_t hswa_prefill_workspace_size_exact(const hswa_pool *pool, const hswa_layer *layer, int n_seqs,
                                                    const int32_t *prefix_len, const int32_t *q_start) {
    if (!pool || !layer || n_seqs < 0 || (n_seqs > 0 && (!prefix_len || !q_start)) ||
        pool->cfg.dtype != HSWA_DTYPE_FP8_E4M3)
        return 0;
    if (layer->kind == HSWA_KIND_SWA && layer->window <= 0) return 0;
    const int32_t window = layer->kind == HSWA_KIND_SWA ? layer->window : 0;
    int64_t pages = 0;
    for (int i = 0; i < n_seqs; ++i) {
        int32_t lo, hi;
        chunk_pages(prefix_len[i], q_start[i + 1] - q_start[i], window, lo, hi);
        pages += std::max(0, hi - lo + 1);
    }
    return stage_bytes(pool->cfg, n_seqs, n_seqs > 0 ? q_start[n_seqs] : 0, pages);
}

extern "C" int hswa_prefill_chunk_ws(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                                     const int32_t *d_bt, const int32_t *d_prefix_len, const int32_t *d_q_start,
                                     int n_seqs, int total_q, int max_q_len, float scale, void *ws, size_t ws_bytes,
                                     hswa_stream_t stream) {
    HSWA_NVTX("hswa_prefill_chunk_ws");
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
        const StageLayout l = stage_layout(c, n_seqs, total_q, ws_bytes);
        if (!ws || ((uintptr_t)ws & 255) || l.cap < 1) return HSWA_ERR_INVALID_ARG;
        if ((int64_t)total_q > (int64_t)n_seqs * max_q_len) return HSWA_ERR_INVALID_ARG;
        const int64_t staged_pages = std::min<int64_t>(l.cap, (int64_t)n_seqs * c.max_pages_per_seq);
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
        sa.stage_off = reinterpret_cast<int32_t *>(base + l.off_off);
        sa.k_out = reinterpret_cast<__half *>(base + l.k_off);
        sa.v_out = reinterpret_cast<__half *>(base + l.k_off + (size_t)staged_pages * l.page_bytes);
        sa.n_seqs = n_seqs;
        sa.bt_stride = c.max_pages_per_seq;
        sa.hkv = c.n_kv_heads;
        sa.window = window;
        sa.num_pages = num_pages;
        sa.cap = (int32_t)staged_pages;
        sa.err = error_word();
        __half *q16 = reinterpret_cast<__half *>(base + l.q_off);
        const int64_t n8 = (int64_t)total_q * c.n_q_heads * kD / 8;
        set_last_kernel(window > 0 && window <= kBN ? "prefill_stage_fp8+prefill_swa_tc_d128<f16>"
                                                     : "prefill_stage_fp8+prefill_tc_bf16_d128<f16>");
        prefill_stage_plan<<<1, 256, 0, st>>>(sa);
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
    set_last_kernel(window > 0 && window <= kBN ? "prefill_swa_tc_d128" : "prefill_tc_bf16_d128");
    return launch_prefill_tc(c, window, layer->k_pool, layer->v_pool, false, num_pages, d_bt, q, o, d_prefix_len,
                             d_q_start, n_seqs, total_q, max_q_len, scale, st);
}

extern "C" int hswa_prefill_chunk(const hswa_pool *pool, const hswa_layer *layer, const void *q, void *o,
                                  const int32_t *d_bt, const int32_t *d_prefix_len, const int32_t *d_q_start,
                                  int n_seqs, int total_q, int max_q_len, float scale, hswa_stream_t stream) {
    return hswa_prefill_chunk_ws(pool, layer, q, o, d_bt, d_prefix_len, d_q_start, n_seqs, total_q, max_q_len, scale,
                                 nullptr, 0, stream);
}
