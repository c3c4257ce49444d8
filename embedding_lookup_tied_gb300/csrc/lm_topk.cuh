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
    // selection-warp mode: the two staging slots of block logits (in the
    // bytes of scratch / hist, unused in that mode) and their barriers
    uint64_t sel_full[2];
    uint64_t sel_empty[2];
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
// exp((v - m') / T) one has a zero argument, i.e. is exactly 1, so one
// exponential of (min(m, v) - m') / T serves both cases, without a branch:
// s' = s + t when v does not raise the max, s' = s t + 1 when it does.  It
// is the hardware exponential (__expf: a few ulp where the terms matter,
// i.e. near the max; the far terms it rounds worse are smaller by e^-|x|),
// which keeps the sum within ~1e-6 of the exact one.
__device__ __forceinline__ void ms_update(float &m, float &s, float v, float invT) {
    const float mn = fmaxf(m, v);
    if (mn == -INFINITY) return;
    const float t = __expf((fminf(m, v) - mn) * invT);
    s = v > m ? fmaf(s, t, 1.0f) : s + t;
    m = mn;
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

__device__ __forceinline__ void topk_write_lists(TopkShared &sm, int tid, int nthreads, int ncols, int k, int cap,
                                                 int b_off, int batch_total, uint64_t *part_keys) {
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
}

__device__ __forceinline__ void topk_finish(TopkShared &sm, int tid, int nthreads, int ncols, int k, int cap,
                            int b_off, int batch_total, uint64_t *part_keys, float2 *part_ms,
                            float invT) {
    topk_write_lists(sm, tid, nthreads, ncols, k, cap, b_off, batch_total, part_keys);
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

__host__ __device__ __forceinline__ int pow2_at_least(int n) {
    int q = 1;
    while (q < n) q <<= 1;
    return q;
}

// Bitonic sort, largest first, of the warp's 32 * KPL keys: lane l holds
// elements l, 32 + l, 64 + l, ...  Partners 32 or more apart sit in the same
// lane; nearer ones in lane l ^ t, exchanged by shuffles.
template <int KPL>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&x)[KPL], int lane) {
    constexpr int N = 32 * KPL;
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int t = size >> 1; t > 0; t >>= 1) {
            if (t >= 32) {
                const int tq = t >> 5;
#pragma unroll
                for (int q = 0; q < KPL; ++q) {
                    const int pq = q ^ tq;
                    if (pq > q) {  // element i = 32 q + l, partner i + t
                        const int i = 32 * q + lane;
                        const bool desc = (i & size) == 0;  // this run sorts largest first
                        const uint64_t a = x[q], c = x[pq];
                        const bool swap = desc ? (a < c) : (a > c);
                        x[q] = swap ? c : a;
                        x[pq] = swap ? a : c;
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < KPL; ++q) {
                    const int i = 32 * q + lane;
                    const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, x[q], t);
                    const bool desc = (i & size) == 0;
                    const bool lower = (lane & t) == 0;  // the smaller index of the pair
                    // the lower index keeps the larger key in a descending run
                    const bool keep_max = desc == lower;
                    x[q] = keep_max ? (o > x[q] ? o : x[q]) : (o < x[q] ? o : x[q]);
                }
            }
        }
    }
}

// keys[0, n) (n <= 32 KPL) sorted largest first in place, the first min(n, k)
// written back.  Warp-collective.
template <int KPL>
__device__ __forceinline__ void warp_sort_cut(uint64_t *keys, int n, int k, int lane) {
    uint64_t x[KPL];
#pragma unroll
    for (int q = 0; q < KPL; ++q) {
        const int i = 32 * q + lane;
        x[q] = i < n ? keys[i] : 0ull;  // 0 is below every key
    }
    warp_sort_desc<KPL>(x, lane);
    __syncwarp();
    const int m = n < k ? n : k;
#pragma unroll
    for (int q = 0; q < KPL; ++q)
        if (32 * q + lane < m) keys[32 * q + lane] = x[q];
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Selection warp.  The consumer warps of a streaming GEMV only stage each
// 128-row block's logits, [column][row] f32, in one of two slots (the bytes
// of scratch / hist) and arrive on the slot's full barrier; one selection
// warp owns every candidate list of the CTA (column b in cand[b * cap ..],
// count and threshold in its registers), takes each staged block, folds it
// into the online softmax (m, s) and its lists, cuts a list back to k with a
// warp radix select once it holds more than the limit, and releases the
// slot.  The streaming warps never wait for each other or run the
// selection; at the end the selection warp writes (m, s) per column and
// the counts, and after a final barrier the consumers write the lists
// (topk_write_lists: they have the CTA-wide lists' layout).
// ---------------------------------------------------------------------------
constexpr int kSelSlots = 2;
constexpr int kSelLimitMax = BM;  // lists never exceed kSelLimitMax + BM = 256 keys
static_assert(sizeof(float) * kSelSlots * kBatchChunk * BM >= sizeof(unsigned) * 256 * kBatchChunk,
              "the staging slots hold a histogram per column for the final cut");
static_assert(sizeof(uint64_t) * kBatchChunk * kMaxK >= sizeof(float) * kSelSlots * kBatchChunk * BM,
              "the staging slots fit in the scratch keys' bytes");

__device__ __forceinline__ float *sel_slot(TopkShared &sm, int blk) {
    return reinterpret_cast<float *>(sm.scratch) + (blk & 1) * (kBatchChunk * BM);
}
// Consumer side: wait until block blk's slot is free (the selection warp has
// taken block blk - 2); false when the wait ran out.
__device__ __forceinline__ bool sel_acquire(TopkShared &sm, int blk) {
    const int n = blk >> 1;
    return n == 0 || mbar_wait(&sm.sel_empty[blk & 1], (n - 1) & 1, kWaitTimeoutNs);
}
// Consumer side: this warp's rows of block blk are staged (every consumer
// warp arrives once per block, rows or not).
__device__ __forceinline__ void sel_publish(TopkShared &sm, int blk, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.sel_full[blk & 1]);
}
__device__ __forceinline__ void sel_init(TopkShared &sm, int consumer_warps) {
    for (int i = 0; i < kSelSlots; ++i) {
        mbar_init(&sm.sel_full[i], consumer_warps);
        mbar_init(&sm.sel_empty[i], 1);
    }
}

constexpr int kBarFinal = 14;  // named barrier: consumers + selection warp, end of a pass
static_assert(sizeof(float2) * kMaxConsumerWarps * kBatchChunk >= sizeof(unsigned) * 256,
              "ms_warp's bytes hold the selection warp's histogram");

// keys[0, n) (unique, k < n <= 256) cut in place to exactly its k largest,
// in their original order, by a radix select over 8-bit digits (hist: 256
// words of shared scratch); returns the k-th largest.  Warp-collective, out
// of line (its registers stay out of the caller's loop).
__device__ __noinline__ uint64_t warp_cut_to_k(uint64_t *keys, int n, int k, unsigned *hist, int *sel_digit,
                                               int *sel_above, int lane) {
    Group g;
    g.gtid = lane;
    g.T = 32;
    g.bar_id = 0;
    g.col = 0;
    uint64_t prefix, mask;
    group_radix_select(keys, n, k, hist, sel_digit, sel_above, g, prefix, mask);
    // stable compaction, chunk by chunk: a survivor's new place is at most
    // its old one, and every lane has read its key before the chunk's writes
    const unsigned lt = (1u << lane) - 1u;
    int out = 0;
    uint64_t kmin = ~0ull;
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const uint64_t key = i < n ? keys[i] : 0ull;
        const bool keep = i < n && (key & mask) >= prefix;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
        __syncwarp();
        if (keep) {
            keys[out + __popc(bal & lt)] = key;
            kmin = key < kmin ? key : kmin;
        }
        out += __popc(bal);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, kmin, o);
        kmin = other < kmin ? other : kmin;
    }
    __syncwarp();
    return kmin;
}

// The selection warp's whole job for one projection pass.  rows_of(blk,
// row0, rows) gives block blk's first vocab row and row count.  Returns
// false when it stopped early (timeout or the consumers' abort).
template <typename RowsOf>
__device__ __forceinline__ bool sel_run(TopkShared &sm, int nblk, RowsOf rows_of, int ncols, int k, float invT,
                                        int b_off, int batch_total, float2 *part_ms, int32_t *err, int lane) {
    const int cap = kCandTotal / pow2_at_least(ncols);
    int limit = cap - BM;
    limit = limit < 2 * k + 64 ? limit : 2 * k + 64;
    limit = limit < kSelLimitMax ? limit : kSelLimitMax;  // >= k for k <= kMaxK
    uint64_t tau[kBatchChunk];
    int cnt[kBatchChunk];
    float ms_m[kBatchChunk], ms_s[kBatchChunk];
#pragma unroll
    for (int b = 0; b < kBatchChunk; ++b) {
        tau[b] = 0ull;
        cnt[b] = 0;
        ms_m[b] = -INFINITY;
        ms_s[b] = 0.0f;
    }
    const unsigned lt = (1u << lane) - 1u;
    bool ok = true;
    for (int blk = 0; blk < nblk && ok; ++blk) {
                if (!mbar_wait(&sm.sel_full[blk & 1], (blk >> 1) & 1, kWaitTimeoutNs)) {
            ok = false;
            break;
        }
        int64_t row0;
        int rows;
        rows_of(blk, row0, rows);
        const float *st = sel_slot(sm, blk);
#pragma unroll
        for (int b = 0; b < kBatchChunk; ++b) {
            if (b >= ncols) break;
#pragma unroll
            for (int q = 0; q < BM / 32; ++q) {
                const int r = lane + 32 * q;
                const bool valid = r < rows;
                const float v = st[b * BM + r];
                if (valid) ms_update(ms_m[b], ms_s[b], v, invT);
                const uint64_t key = topk_key(v, static_cast<int32_t>(row0 + r));
                const bool pass = valid && key > tau[b];
                const unsigned mask = __ballot_sync(0xFFFFFFFFu, pass);
                if (pass) sm.cand[b * cap + cnt[b] + __popc(mask & lt)] = key;
                cnt[b] += __popc(mask);
            }
            if (cnt[b] > limit) {
                __syncwarp();
                tau[b] = warp_cut_to_k(sm.cand + b * cap, cnt[b], k, reinterpret_cast<unsigned *>(sm.ms_warp),
                                       &sm.sel_digit[0], &sm.sel_above[0], lane);
                cnt[b] = k;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sel_empty[blk & 1]);
    }
    if (!ok) {
        if (lane == 0) {
            set_err(err, LHS_ERRBIT_TIMEOUT);
            sm.abort_flag = 1;
        }
        __syncwarp();
        return false;
    }
    // (m, s) per column; the counts for the consumers, who sort the lists
    // after the final barrier (sel_finish)
#pragma unroll
    for (int b = 0; b < kBatchChunk; ++b) {
        if (b >= ncols) break;
        float M = ms_m[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        float S = ms_rescaled(ms_m[b], ms_s[b], M, invT);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
        if (lane == 0) {
            part_ms[static_cast<size_t>(blockIdx.x) * batch_total + b_off + b] = make_float2(M, S);
            sm.cnt[b] = cnt[b];
        }
    }
    return true;
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
