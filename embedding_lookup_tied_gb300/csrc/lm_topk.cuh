// lm_topk.cuh — state and helpers shared by the streaming GEMV kernels of
// the lm_head (lm_head.cu, gemv_q8.cu): the per-CTA candidate lists of the
// fused top-k (ADR-0008 "Remote Embeddings and lm_head Service", POST
// /v1/logits: top_k {token_id, prob}), the online softmax (max, sum exp)
// and the split of the vocab rows over the CTAs.  Included by CUDA sources
// only; everything is internal to each translation unit.
#pragma once

#include "lhs_internal.cuh"

namespace lhs {
namespace {

constexpr int BM = 128;                   // table rows per block
constexpr int kCandTotal = 2048;             // candidate keys per CTA (all residuals)
constexpr int kBatchChunk = 8;               // residuals per projection pass
constexpr int kBarAll = 15;                  // named barrier: all consumers (groups use 1..8)
constexpr int kMaxConsumerWarps = 16;        // largest consumer group of the top-k state
constexpr int kWarpLists = 8;                // warps with lists of their own (per-warp mode)
constexpr int kWarpListSlots = kCandTotal / kWarpLists;  // 256 keys per warp, all columns
constexpr int kWarpRowsPerRound = 16;        // rows a warp offers between two of its cuts

// ---------------------------------------------------------------------------
// shared top-k state (both GEMV kernels)
// ---------------------------------------------------------------------------
struct TopkShared {
    uint64_t cand[kCandTotal];
    // Column c's radix-select histogram and its scratch keys share bytes:
    // the select has finished with hist[c] (behind a group barrier) before
    // scratch[c] is written, and nothing reads hist[c] after that.
    union {
        uint64_t scratch[kBatchChunk][kMaxK];
        unsigned hist[kBatchChunk][256];
    };
    uint64_t tau[kBatchChunk];
    uint64_t tmin[kBatchChunk];
    float2 ms_warp[kMaxConsumerWarps][kBatchChunk];
    int cnt[kBatchChunk];
    int nsel[kBatchChunk];
    int sel_digit[kBatchChunk];
    int sel_above[kBatchChunk];
    int need_compact;
    int abort_flag;
    // per-warp lists (warp_lists_fit): counts and k-th best keys, warp x column
    int wcnt[kWarpLists][kBatchChunk];
    uint64_t wtau[kWarpLists][kBatchChunk];
};

static_assert(sizeof(uint64_t) * kMaxK == sizeof(unsigned) * 256, "a column's hist and scratch coincide");

__device__ __forceinline__ int ld_volatile(const int *p) { return *reinterpret_cast<const volatile int *>(p); }

struct Group {  // the threads that own one residual column during selection
    int gtid, T, bar_id, col;
};

__device__ __forceinline__ void group_sync(const Group &g) {
    if (g.T == 32) __syncwarp();
    else named_bar_sync(g.bar_id, g.T);
}

// Split `nthreads` consumer threads into pow2(ncols) groups.
__device__ __forceinline__ Group make_group(int tid, int nthreads, int ncols) {
    int p = 1;
    while (p < ncols) p <<= 1;
    Group g;
    g.T = nthreads / p;
    g.col = tid / g.T;
    g.gtid = tid % g.T;
    g.bar_id = 1 + g.col;  // ids 1..4 (only used when T > 32, i.e. p <= 4)
    return g;
}

// Radix select over 8-bit digits of 64-bit keys: find the kk-th largest of
// keys[0..cnt) (keys unique) and return (prefix, mask) such that exactly kk
// keys satisfy (key & mask) >= prefix.  Executed by the T threads of a group.
__device__ __forceinline__ void group_radix_select(const uint64_t *keys, int cnt, int kk, unsigned *hist,
                                   int *sel_digit, int *sel_above, const Group &g,
                                   uint64_t &prefix_out, uint64_t &mask_out) {
    uint64_t prefix = 0, mask = 0;
    int need = kk;
    const int lane = g.gtid & 31;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = g.gtid; i < 256; i += g.T) hist[i] = 0;
        group_sync(g);
        // histogram of the digit, one atomic per distinct digit per warp
        // (keys that share a prefix mostly share the next digit too)
        for (int base = 0; base < cnt; base += g.T) {
            const int i = base + g.gtid;
            uint32_t digit = 0xFFFFFFFFu;
            if (i < cnt) {
                const uint64_t key = keys[i];
                if ((key & mask) == prefix) digit = static_cast<uint32_t>(key >> shift) & 255u;
            }
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, digit);
            if (digit != 0xFFFFFFFFu && __ffs(peers) - 1 == lane)
                atomicAdd(&hist[digit], static_cast<unsigned>(__popc(peers)));
        }
        group_sync(g);
        if (g.gtid < 32) {
            // lane L owns digits 255-8L ... 248-8L (descending)
            unsigned c[8];
            unsigned lsum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = hist[255 - 8 * lane - i];
                lsum += c[i];
            }
            unsigned incl = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            const unsigned excl = incl - lsum;
            if (excl < static_cast<unsigned>(need) && static_cast<unsigned>(need) <= incl) {
                unsigned run = excl;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (run + c[i] >= static_cast<unsigned>(need)) {
                        *sel_digit = 255 - 8 * lane - i;
                        *sel_above = static_cast<int>(run);
                        break;
                    }
                    run += c[i];
                }
            }
        }
        group_sync(g);
        const int d = *sel_digit;
        const int above = *sel_above;
        const int bin = static_cast<int>(hist[d]);
        need -= above;
        prefix |= static_cast<uint64_t>(d) << shift;
        mask |= 0xFFull << shift;
        group_sync(g);  // everyone has read hist / sel_* before they change
        if (bin == need) break;
    }
    prefix_out = prefix;
    mask_out = mask;
}

// Cut keys[0..*cnt) down to its kk best (kk <= kMaxK), in place; *tau
// becomes the kk-th best key.  Group-collective.
// Short lists (n^2 / group size <= kDirectWork compares per thread) are cut
// by ranking every key against all the others (keys are unique: its rank is
// its place), one pass instead of the radix select's digit passes.
constexpr int kDirectWork = 512;

__device__ __forceinline__ void group_compact(uint64_t *keys, int *cnt, uint64_t *tau, int kk, TopkShared &sm,
                              const Group &g) {
    const int n = *cnt;
    if (n <= kk) return;  // uniform across the group
    if (n <= kMaxK * 2 + 128 && n * n <= g.T * kDirectWork) {
        for (int i = g.gtid; i < n; i += g.T) {
            const uint64_t key = keys[i];
            int rank = 0;
#pragma unroll 4
            for (int q = 0; q < n; ++q) rank += keys[q] > key;
            if (rank < kk) sm.scratch[g.col][rank] = key;
        }
        group_sync(g);
        for (int i = g.gtid; i < kk; i += g.T) keys[i] = sm.scratch[g.col][i];
        if (g.gtid == 0) {
            *cnt = kk;
            *tau = sm.scratch[g.col][kk - 1];
        }
        group_sync(g);
        return;
    }
    uint64_t prefix, mask;
    group_radix_select(keys, n, kk, sm.hist[g.col], &sm.sel_digit[g.col], &sm.sel_above[g.col], g,
                       prefix, mask);
    if (g.gtid == 0) {
        sm.nsel[g.col] = 0;
        sm.tmin[g.col] = ~0ull;
    }
    group_sync(g);
    uint64_t kmin = ~0ull;
    for (int i = g.gtid; i < n; i += g.T) {
        const uint64_t key = keys[i];
        if ((key & mask) >= prefix) {
            const int pos = atomicAdd(&sm.nsel[g.col], 1);
            sm.scratch[g.col][pos] = key;
            kmin = key < kmin ? key : kmin;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, kmin, o);
        kmin = other < kmin ? other : kmin;
    }
    if ((g.gtid & 31) == 0 && kmin != ~0ull)
        atomicMin(reinterpret_cast<unsigned long long *>(&sm.tmin[g.col]),
                  static_cast<unsigned long long>(kmin));
    group_sync(g);
    for (int i = g.gtid; i < kk; i += g.T) keys[i] = sm.scratch[g.col][i];
    if (g.gtid == 0) {
        *cnt = kk;
        *tau = sm.tmin[g.col];
    }
    group_sync(g);
}

// Online softmax state (m, s): s = sum exp((v - m) / T) over the values
// seen, m their max.  Of the two rescalings exp((m - m') / T) and
// exp((v - m') / T) one has a zero argument, i.e. is exactly 1, so only the
// other is evaluated.  The common case, a term below the running max, uses
// the hardware exponential (__expf: a few ulp where the terms matter, i.e.
// near the max; the far terms it rounds worse are smaller by e^-|x|), which
// keeps the sum within ~1e-6 of the exact one; the rare new-max rescaling of
// the whole sum uses the accurate expf.
__device__ __forceinline__ void ms_update(float &m, float &s, float v, float invT) {
    const float mn = fmaxf(m, v);
    if (mn == -INFINITY) return;
    if (m >= v) {
        s = s + __expf((v - mn) * invT);
    } else {
        s = s * expf((m - mn) * invT) + 1.0f;
        m = mn;
    }
}
// s * exp((m - M) / T), the sum of a partial (m, s) rescaled to a max M >= m
// (exactly s when m == M, including the empty partial m = M = -inf).
__device__ __forceinline__ float ms_rescaled(float m, float s, float M, float invT) {
    return m == M ? s : (m == -INFINITY ? 0.0f : s * expf((m - M) * invT));
}

__device__ __forceinline__ float2 ms_combine(float2 a, float2 b, float invT) {
    const float mn = fmaxf(a.x, b.x);
    if (mn == -INFINITY) return make_float2(-INFINITY, 0.0f);
    if (a.x >= b.x) return make_float2(a.x, a.y + b.y * expf((b.x - a.x) * invT));
    return make_float2(b.x, b.y + a.y * expf((a.x - b.x) * invT));
}

__device__ __forceinline__ void topk_init(TopkShared &sm, int tid, int nthreads) {
    for (int b = tid; b < kBatchChunk; b += nthreads) {
        sm.cnt[b] = 0;
        sm.tau[b] = 0ull;
    }
    for (int i = tid; i < kWarpLists * kBatchChunk; i += nthreads) {
        sm.wcnt[i / kBatchChunk][i % kBatchChunk] = 0;
        sm.wtau[i / kBatchChunk][i % kBatchChunk] = 0ull;
    }
    if (tid == 0) {
        sm.need_compact = 0;
        sm.abort_flag = 0;
    }
}

// Offer one logit: appended when it beats the column's current k-th best.
__device__ __forceinline__ void topk_offer(TopkShared &sm, int col, int cap, float v, int32_t id) {
    const uint64_t key = topk_key(v, id);
    if (key > sm.tau[col]) {
        const int pos = atomicAdd(&sm.cnt[col], 1);
        sm.cand[col * cap + pos] = key;
    }
}

// After a round that could add up to `round_max` candidates per column:
// cut lists back to k once they hold 2k+64 entries (so the threshold rises
// early and later rounds offer few candidates), and always before they could
// overflow.  The cut runs while the producer keeps the TMA ring full, so it
// costs no HBM time while it is shorter than the ring.  All consumers call.
__device__ __forceinline__ void topk_round_end(TopkShared &sm, int tid, int nthreads, int ncols, int k, int cap,
                               int round_max) {
    named_bar_sync(kBarAll, nthreads);
    if (tid == 0) {
        const int limit = min(cap - round_max, 2 * k + 64);
        int need = 0;
        for (int b = 0; b < ncols; ++b) need |= (sm.cnt[b] > limit);
        sm.need_compact = need;
    }
    named_bar_sync(kBarAll, nthreads);
    if (sm.need_compact) {
        const Group g = make_group(tid, nthreads, ncols);
        if (g.col < ncols) group_compact(sm.cand + g.col * cap, &sm.cnt[g.col], &sm.tau[g.col], k, sm, g);
        named_bar_sync(kBarAll, nthreads);
    }
}

// Final cut to k and write the CTA's partial list and (m, s) per column.
// Each list is written sorted, largest key first, and padded with 0 (below
// every key).  A candidate's place is the number of larger candidates in its
// column (keys are unique), so when the lists are short every candidate is
// ranked directly — one pass, no selection rounds; otherwise a radix select
// first cuts each column to k.
constexpr int kRankWork = 512;  // comparisons per thread for the direct ranking

__device__ __forceinline__ void topk_finish(TopkShared &sm, int tid, int nthreads, int ncols, int k, int cap,
                            int b_off, int batch_total, uint64_t *part_keys, float2 *part_ms,
                            float invT) {
    named_bar_sync(kBarAll, nthreads);
    int work = 0;
    for (int b = 0; b < ncols; ++b) work += sm.cnt[b] * sm.cnt[b];
    if (work > nthreads * kRankWork) {  // uniform: every thread read the same counts
        const Group g = make_group(tid, nthreads, ncols);
        if (g.col < ncols) group_compact(sm.cand + g.col * cap, &sm.cnt[g.col], &sm.tau[g.col], k, sm, g);
        named_bar_sync(kBarAll, nthreads);
    }
    int total = 0;
    for (int b = 0; b < ncols; ++b) total += sm.cnt[b];
    for (int i = tid; i < total; i += nthreads) {
        int b = 0, j = i;
        while (j >= sm.cnt[b]) j -= sm.cnt[b++];
        const int n = sm.cnt[b];
        const uint64_t *src = sm.cand + b * cap;
        const uint64_t key = src[j];
        int rank = 0;
#pragma unroll 4
        for (int q = 0; q < n; ++q) rank += src[q] > key;
        if (rank < k)
            part_keys[(static_cast<size_t>(blockIdx.x) * batch_total + b_off + b) * k + rank] = key;
    }
    for (int i = tid; i < ncols * k; i += nthreads) {
        const int b = i / k, j = i % k;
        if (j >= sm.cnt[b])
            part_keys[(static_cast<size_t>(blockIdx.x) * batch_total + b_off + b) * k + j] = 0ull;
    }
    if (tid < ncols) {
        // the warps' (m, s): max first, then the rescaled sums (independent exps)
        const int nw = nthreads / 32;
        float M = -INFINITY;
        for (int w = 0; w < nw; ++w) M = fmaxf(M, sm.ms_warp[w][tid].x);
        float S = 0.0f;
#pragma unroll 4
        for (int w = 0; w < nw; ++w) S += ms_rescaled(sm.ms_warp[w][tid].x, sm.ms_warp[w][tid].y, M, invT);
        part_ms[static_cast<size_t>(blockIdx.x) * batch_total + b_off + tid] = make_float2(M, S);
    }
}

// ---------------------------------------------------------------------------
// Per-warp candidate lists.  Each of kWarpLists consumer warps keeps its own
// list per residual column in its kWarpListSlots slots of cand (column b at
// b * cap_w, cap_w = kWarpListSlots / pow2(ncols)) and cuts it alone, so the
// stream has no CTA-wide barrier: a warp cuts its list back to k (sorted,
// largest first; the k-th key becomes its threshold) once it could not take
// another kWarpRowsPerRound offers, or holds 2k + 32 keys.  At the end every
// warp sorts what it holds, and the CTA ranks each key among the union of
// the sorted lists by binary search.  Used when a column's list holds k plus
// one round of offers (warp_lists_fit).
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int pow2_at_least(int n) {
    int q = 1;
    while (q < n) q <<= 1;
    return q;
}
__host__ __device__ __forceinline__ int warp_list_cap(int ncols) { return kWarpListSlots / pow2_at_least(ncols); }
__host__ __device__ __forceinline__ bool warp_lists_fit(int ncols, int k) {
    return k >= 1 && k + kWarpRowsPerRound <= warp_list_cap(ncols);
}
__device__ __forceinline__ int warp_list_limit(int ncols, int k) {
    const int a = warp_list_cap(ncols) - kWarpRowsPerRound, b = 2 * k + 32;
    return a < b ? a : b;
}

// Offer one logit to warp w's list for column b (any subset of the warp's
// lanes, one logit each).
__device__ __forceinline__ void wl_offer(TopkShared &sm, int w, int b, int cap_w, float v, int32_t id) {
    const uint64_t key = topk_key(v, id);
    if (key > sm.wtau[w][b]) {
        const int pos = atomicAdd(&sm.wcnt[w][b], 1);
        sm.cand[w * kWarpListSlots + b * cap_w + pos] = key;
    }
}

// Warp w's list of column b cut to its best min(n, k), sorted, largest first
// (keys are unique: a key's rank is its place); the threshold becomes the
// k-th key once the list holds k.  Warp-collective.
__device__ __forceinline__ void wl_cut(TopkShared &sm, int w, int b, int cap_w, int k, int lane) {
    uint64_t *keys = sm.cand + w * kWarpListSlots + b * cap_w;
    uint64_t *tmp = sm.scratch[w];  // per-warp row (the CTA-wide select is not used in this mode)
    const int n = sm.wcnt[w][b];
    for (int i = lane; i < n; i += 32) {
        const uint64_t key = keys[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) rank += keys[j] > key;
        if (rank < k) tmp[rank] = key;
    }
    __syncwarp();
    const int m = n < k ? n : k;
    for (int i = lane; i < m; i += 32) keys[i] = tmp[i];
    __syncwarp();
    if (lane == 0) {
        sm.wcnt[w][b] = m;
        if (m == k) sm.wtau[w][b] = keys[k - 1];
    }
    __syncwarp();
}

// After a round of the warp's offers: cut the lists that could not take
// another round.  Warp-collective; ncols and the counts are uniform after
// the warp barrier.
__device__ __forceinline__ void wl_round_end(TopkShared &sm, int w, int ncols, int k, int lane) {
    __syncwarp();
    const int cap_w = warp_list_cap(ncols), limit = warp_list_limit(ncols, k);
    for (int b = 0; b < ncols; ++b)
        if (sm.wcnt[w][b] > limit) wl_cut(sm, w, b, cap_w, k, lane);
}

// Number of keys greater than `key` in a list sorted largest first.
__device__ __forceinline__ int count_above(const uint64_t *list, int n, uint64_t key) {
    int lo = 0, hi = n;  // list[0, lo) > key, list[hi, n) <= key
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (list[mid] > key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// End of the pass: every warp sorts (and cuts to k) its lists, then the
// CTA writes its partial list per column, sorted and padded with 0, and
// (m, s) from ms_warp, as topk_finish does.  All nthreads consumers call it
// (warps 0 .. kWarpLists-1 own the lists).
__device__ __forceinline__ void wl_finish(TopkShared &sm, int tid, int nthreads, int ncols, int k, int b_off,
                                          int batch_total, uint64_t *part_keys, float2 *part_ms, float invT) {
    const int w = tid >> 5, lane = tid & 31;
    const int cap_w = warp_list_cap(ncols);
    if (w < kWarpLists)
        for (int b = 0; b < ncols; ++b) wl_cut(sm, w, b, cap_w, k, lane);
    named_bar_sync(kBarAll, nthreads);
    // keys: (column b, warp ww, index i) over the columns' lists
    const int per_col = kWarpLists * k;
    for (int e = tid; e < ncols * per_col; e += nthreads) {
        const int b = e / per_col, ww = (e % per_col) / k, i = e % k;
        if (i >= sm.wcnt[ww][b]) continue;
        const uint64_t key = sm.cand[ww * kWarpListSlots + b * cap_w + i];
        int rank = i;
#pragma unroll
        for (int o = 0; o < kWarpLists; ++o)
            if (o != ww) rank += count_above(sm.cand + o * kWarpListSlots + b * cap_w, sm.wcnt[o][b], key);
        if (rank < k) part_keys[(static_cast<size_t>(blockIdx.x) * batch_total + b_off + b) * k + rank] = key;
    }
    for (int e = tid; e < ncols * k; e += nthreads) {
        const int b = e / k, j = e % k;
        int total = 0;
#pragma unroll
        for (int o = 0; o < kWarpLists; ++o) total += sm.wcnt[o][b];
        if (j >= total) part_keys[(static_cast<size_t>(blockIdx.x) * batch_total + b_off + b) * k + j] = 0ull;
    }
    if (tid < ncols) {
        const int nw = nthreads / 32;
        float M = -INFINITY;
        for (int ww = 0; ww < nw; ++ww) M = fmaxf(M, sm.ms_warp[ww][tid].x);
        float S = 0.0f;
#pragma unroll 4
        for (int ww = 0; ww < nw; ++ww) S += ms_rescaled(sm.ms_warp[ww][tid].x, sm.ms_warp[ww][tid].y, M, invT);
        part_ms[static_cast<size_t>(blockIdx.x) * batch_total + b_off + tid] = make_float2(M, S);
    }
}

// Row range of CTA c: 16-row units split evenly.
__device__ __forceinline__ void cta_rows(int64_t V, int G, int c, int64_t &r0, int64_t &r1) {
    const int64_t units = (V + 15) / 16;
    r0 = (units * c / G) * 16;
    r1 = (units * (c + 1) / G) * 16;
    if (r1 > V) r1 = V;
    if (r0 > V) r0 = V;
}

// Blocks of CTA c in the tensor-core GEMV, interleaved over the table: the
// full 128-row blocks c, c + G, c + 2G, ... of the first q = V / (G * BM)
// rounds, then CTA c's even share (16-row units) of the rows after them.
// Every CTA streams the same number of rows give or take 16, drawn from all
// over the table.
__device__ __forceinline__ int tc_blocks(int64_t V, int G, int c) {
    const int64_t q = V / (static_cast<int64_t>(G) * BM);
    int64_t s0, s1;
    cta_rows(V - q * G * BM, G, c, s0, s1);
    return static_cast<int>(q) + (s1 > s0 ? 1 : 0);
}
__device__ __forceinline__ void tc_block(int64_t V, int G, int c, int blk, int64_t &row0, int &rows) {
    const int64_t q = V / (static_cast<int64_t>(G) * BM);
    if (blk < q) {
        row0 = (c + static_cast<int64_t>(blk) * G) * BM;
        rows = BM;
    } else {
        int64_t s0, s1;
        cta_rows(V - q * G * BM, G, c, s0, s1);
        row0 = q * G * BM + s0;
        rows = static_cast<int>(s1 - s0);
    }
}

}  // namespace
}  // namespace lhs
