// lm_head.cu — steps 2+3: tied lm_head projection with fused top-k.
//
// ADR-0008 "Remote Embeddings and lm_head Service", POST /v1/logits: the
// projection residual @ lm_head.T over every vocab row, answered as top_k
// {token_id, prob} (or the raw logit vector); Open Question 1: the lm_head
// is the embedding table itself.  HELIX "Columnar Embedding", §5: the
// projection needs all vocab rows, so every call streams the whole table.
//
// Design (one GPU, the table resident in HBM):
//  * The vocab is split into G contiguous row ranges, one per CTA (G = SM
//    count), balanced to 16 rows.  Each CTA streams its rows once.
//  * f16/bf16 tables, hidden % 8 == 0: tensor-core streaming GEMV.  A
//    producer warp drives a ring of TMA tiles (128 table rows x 64 k,
//    128-byte swizzle) plus the matching 16 x 64 operand tile of the
//    residuals; 8 consumer warps run mma.sync m16n8k16 (f32 accumulate), each
//    on 16 vocab rows.  The residuals enter as two 16-bit rows each
//    (hi = rn16(x), lo = rn16(x - hi)), so the product keeps ~16 (bf16) or
//    ~22 (f16) bits of every f32 residual.
//  * Q8_0 tables, hidden % 256 == 0: the tensor-core GEMV of gemv_q8.cu
//    (codes turned into exact f16 in registers, the per-block scale applied
//    in f32 after each block's MMAs).
//  * Other tables (f32, other Q8_0, ragged hidden): CUDA-core GEMV, one warp
//    per row (f32 rows up to 1 KB: a bulk-copy ring of whole rows),
//    residuals in shared memory as f32.
//  * Fused top-k: every logit is offered to a per-CTA candidate list per
//    residual if it beats that list's current k-th best key; lists are cut
//    back to k by a radix select when they fill.  An online (max, sum exp)
//    per residual rides along.  Each CTA writes k candidates and (m, s) per
//    residual; a merge kernel selects the global top-k, sorts it and
//    evaluates the probabilities.  The full logit vector is never written
//    (unless the raw-logits call asks for it, which uses the same kernels
//    and the same summation order).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "lhs_internal.cuh"
#include "lm_topk.cuh"

namespace lhs {
namespace {

// ---------------------------------------------------------------------------
// tile geometry
// ---------------------------------------------------------------------------
constexpr int BK = 64;                    // k per stage: 128 bytes of 16-bit values
// TMA ring depth of the tensor-core GEMV: as deep as shared memory allows
// next to the residual operand (a consumer stall stops the refills; stages
// in flight beyond the bandwidth-delay product absorb it)
constexpr int kStagesRing = 11;       // residual tiles streamed beside the table tiles
constexpr int kStagesResident = 10;   // resident operand: all 16 rows, or the compact
                                      // layout when it is too wide for kStagesCompact
constexpr int kStagesCompact = 12;    // at most 3 residuals: 2 Bc + 1 rows resident
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTcThreads = kConsumers + 32;  // + one producer warp
constexpr int kAStageBytes = BM * BK * 2;    // 16 KB
constexpr int kXStageBytes = 16 * BK * 2;    // 2 KB: 8 hi rows + 8 lo rows
constexpr int kBoxRowsSmall = 16;            // TMA box for the ragged last block
constexpr int kSimtThreads = 256;

// ---------------------------------------------------------------------------
// merge: global top-k of one residual from G partial lists, sorted, + probs.
// Executed by 256 threads synchronised with named barrier `bar_id`.
// ---------------------------------------------------------------------------
constexpr int kMergeHistCand = 1024;  // candidates the histogram merge ranks directly

struct MergeSmemHead {
    uint64_t sel[kMaxK];
    uint64_t tmin;
    unsigned hist[256];
    float2 ms;
    int nsel, sel_digit, sel_above;
    // histogram merge
    uint64_t cand[kMergeHistCand];
    unsigned lo, hi;            // range of the non-empty keys' order keys
    int n, ncand, bin, above;   // non-empty keys; candidates; the k-th's bin; keys above it
    float wmax[8], wsum[8];     // per-warp softmax (max, sum)
};

__device__ void merge_column(const uint64_t *part_keys, const float2 *part_ms, int G, int stride,
                             int len, int batch_total, int b, int k, float invT, int32_t *out_ids,
                             float *out_logits, float *out_probs, MergeSmemHead &h, uint64_t *keys,
                             int tid, int bar_id) {
    const int n = G * len;
    // all loads of a batch are issued before the first store
    constexpr int U = 8;
    for (int base = 0; base < n; base += U * 256) {
        uint64_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * 256 + tid;
            v[u] = i < n ? __ldcg(part_keys + (static_cast<size_t>(i / len) * batch_total + b) * stride + i % len)
                         : 0ull;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * 256 + tid;
            if (i < n) keys[i] = v[u];
        }
    }
    if (tid < 32) {
        float2 acc = make_float2(-INFINITY, 0.0f);
        float2 o[4];
        for (int g0 = 0; g0 < G; g0 += 128) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int gi = g0 + 32 * u + tid;
                o[u] = gi < G ? __ldcg(part_ms + static_cast<size_t>(gi) * batch_total + b)
                              : make_float2(-INFINITY, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) acc = ms_combine(acc, o[u], invT);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float2 other;
            other.x = __shfl_xor_sync(0xFFFFFFFFu, acc.x, o);
            other.y = __shfl_xor_sync(0xFFFFFFFFu, acc.y, o);
            acc = ms_combine(acc, other, invT);
        }
        if (tid == 0) h.ms = acc;
    }
    named_bar_sync(bar_id, 256);
    Group g;
    g.gtid = tid;
    g.T = 256;
    g.bar_id = bar_id;
    g.col = 0;
    uint64_t prefix, mask;
    group_radix_select(keys, n, k, h.hist, &h.sel_digit, &h.sel_above, g, prefix, mask);
    if (tid == 0) h.nsel = 0;
    named_bar_sync(bar_id, 256);
    for (int i = tid; i < n; i += 256) {
        const uint64_t key = keys[i];
        if ((key & mask) >= prefix) h.sel[atomicAdd(&h.nsel, 1)] = key;
    }
    named_bar_sync(bar_id, 256);
    // rank sort (keys unique): position = number of larger keys
    if (tid < k) {
        const uint64_t mine = h.sel[tid];
        int rank = 0;
        for (int j = 0; j < k; ++j) rank += h.sel[j] > mine;
        const size_t o = static_cast<size_t>(b) * k + rank;
        const float v = key_value(mine);
        out_ids[o] = key_id(mine);
        out_logits[o] = v;
        if (out_probs) out_probs[o] = expf((v - h.ms.x) * invT) / h.ms.y;
    }
    named_bar_sync(bar_id, 256);  // h and keys are free for the next column
}

// ---------------------------------------------------------------------------
// merge of sorted lists.  The GEMV kernels write each CTA's list sorted,
// largest key first, padded with 0 (below every key).  Per residual, 256
// threads (a merge block, or the consumers of the GEMV's last CTA):
//  1. the first R entries of every list and the lists' (max, sum) pairs are
//     staged in shared memory, in one round of L2 reads for all residuals;
//  2. a lower bound L of the global k-th key: from the first m = ceil(k/G)
//     entries of every list (G*m >= k keys), the k-th largest logit order
//     key (the upper 32 bits), with the id bits cleared — at least k keys
//     are >= L;
//  3. the candidates: the entries >= L of every list, a prefix of each
//     (lists whose R staged entries are all >= L are read on from L2),
//     gathered in shared memory;
//  4. a candidate's rank among the candidates is its final position: every
//     key above a candidate is >= L, hence a candidate itself.
// A bound of 0 (fewer than k keys in the sampled prefixes: tiny CTAs) or
// more than kMergeCand candidates (the top keys crowded into few lists)
// sends the residual to a one-key-at-a-time extraction from the list heads
// in L2 instead (merge_extract_warp): slower, same result.
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 256;             // >= G
static_assert(kMergeThreads == 256, "one histogram bin per merge thread");
constexpr int kMergeR = 16;                    // most entries staged per list
constexpr int kMergeSet = 2 * kMergeThreads;   // G*m <= G + k - 1 < 512
constexpr int kMergeCand = 1024;

struct MergeWork {
    uint64_t cand[kMergeCand];
    uint32_t set[kMergeSet];
    unsigned hist[256];  // the sampled keys' histogram (zeroed with lo / hi before the merge)
    float ssum[kMergeThreads / 32];
    uint32_t bound;
    uint32_t lo, hi;     // range of the nonzero sampled keys
    int total;
    float2 msf;
};

// Entries of every list the merge stages: enough for the bound (m) and for
// the few entries per list a residual's top-k usually takes (about 2k/G).
__host__ __device__ __forceinline__ int merge_stage_entries(int G, int k) {
    const int m = (k + G - 1) / G;
    int r = 4 + (4 * k + G - 1) / G;
    if (r < m) r = m;
    if (r > kMergeR) r = kMergeR > m ? kMergeR : m;
    return r < k ? r : k;
}

// Slow path: the top-k taken one key at a time from the list heads, read
// from L2 by one warp; lane l follows lists l, l+32, ... (G <= 256).
__device__ void merge_extract_warp(const uint64_t *part_keys, int G, int batch_total, int b, int k,
                                   float invT, float2 ms, int32_t *out_ids, float *out_logits,
                                   float *out_probs, int lane) {
    constexpr int S = kMergeThreads / 32;
    uint64_t head[S];
    int pos[S];
#pragma unroll
    for (int j = 0; j < S; ++j) {
        const int gi = lane + 32 * j;
        head[j] = gi < G ? __ldcg(part_keys + (static_cast<size_t>(gi) * batch_total + b) * k) : 0ull;
        pos[j] = 0;
    }
    for (int r = 0; r < k; ++r) {
        uint64_t best = 0ull;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < S; ++j)
            if (head[j] > best) {
                best = head[j];
                bj = j;
            }
        uint64_t wbest = best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, wbest, o);
            wbest = other > wbest ? other : wbest;
        }
        if (lane == 0) {
            const size_t o = static_cast<size_t>(b) * k + r;
            const float v = key_value(wbest);
            out_ids[o] = key_id(wbest);
            out_logits[o] = v;
            if (out_probs) out_probs[o] = expf((v - ms.x) * invT) / ms.y;
        }
        if (best == wbest && best != 0ull) {  // the one lane whose list held it
            int pb = 0;
#pragma unroll
            for (int j = 0; j < S; ++j) pb = j == bj ? pos[j] : pb;
            const int gi = lane + 32 * bj;
            const int pn = pb + 1;
            const uint64_t nk =
                pn < k ? __ldcg(part_keys + (static_cast<size_t>(gi) * batch_total + b) * k + pn) : 0ull;
#pragma unroll
            for (int j = 0; j < S; ++j)
                if (j == bj) {
                    head[j] = nk;
                    pos[j] = pn;
                }
        }
    }
}

// Step 1 for residual b: lists[G][R] and sms[G].  All loads of a round are
// issued before the first store; list and entry indexes advance by adding
// (no division per load).
__device__ void stage_sorted_lists(const uint64_t *part_keys, const float2 *part_ms, int G, int k, int R,
                                   int batch_total, int b, uint64_t *lists, float2 *sms, int tid,
                                   int nthreads) {
    constexpr int U = 16;
    const int n = G * R;
    float2 mv = tid < G ? __ldcg(part_ms + static_cast<size_t>(tid) * batch_total + b)
                        : make_float2(-INFINITY, 0.0f);
    const int dc = nthreads / R, dr = nthreads % R;
    for (int base = 0; base < n; base += U * nthreads) {
        int c = (base + tid) / R, j = (base + tid) % R;
        uint64_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            v[u] = base + u * nthreads + tid < n
                       ? __ldcg(part_keys + (static_cast<size_t>(c) * batch_total + b) * k + j)
                       : 0ull;
            c += dc;
            j += dr;
            if (j >= R) {
                j -= R;
                ++c;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * nthreads + tid < n) lists[base + u * nthreads + tid] = v[u];
    }
    if (tid < G) sms[tid] = mv;
}

// Steps 2-4 for residual b, by 256 threads synchronised on named barrier
// `bar_id`.  lists: [G][R] staged entries (R >= ceil(k/G)), sms: [G].  The
// phases are short dependent chains, so independent work runs side by side:
// warp 0 takes the max of the G list maxima while all warps rank the sampled
// keys, the G softmax sums are rescaled to that max in parallel, and
// candidates are appended with one shared atomic per warp instead of a
// block-wide scan.
__device__ void merge_column_sorted(const uint64_t *lists, int R, const float2 *sms, int G, int k,
                                    float invT, const uint64_t *part_keys, int batch_total, int b,
                                    int32_t *out_ids, float *out_logits, float *out_probs, MergeWork &w,
                                    int tid, int bar_id) {
    const int lane = tid & 31, warp = tid >> 5;
    const int m = (k + G - 1) / G;
    const int na = G * m;
    const int na4 = (na + 3) & ~3;
    if (tid == 0) {
        w.bound = 0u;
        w.total = 0;
    }
    unsigned vlo = 0xFFFFFFFFu, vhi = 0u;
    for (int i = tid; i < na4; i += kMergeThreads) {
        const int gi = m == 1 ? i : i / m;
        const uint32_t v = i < na ? static_cast<uint32_t>(lists[gi * R + (i - gi * m)] >> 32) : 0u;
        w.set[i] = v;
        if (v != 0u) {
            vlo = min(vlo, v);
            vhi = max(vhi, v);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        vlo = min(vlo, __shfl_xor_sync(0xFFFFFFFFu, vlo, o));
        vhi = max(vhi, __shfl_xor_sync(0xFFFFFFFFu, vhi, o));
    }
    if (lane == 0 && vlo <= vhi) {
        atomicMin(&w.lo, vlo);
        atomicMax(&w.hi, vhi);
    }
    named_bar_sync(bar_id, kMergeThreads);
    // (max, sum) over the lists, max first: the G rescalings are then
    // independent (one exp each, in parallel) instead of a chain of combines
    if (tid < 32) {
        float mx = -INFINITY;
        for (int gi = lane; gi < G; gi += 32) mx = fmaxf(mx, sms[gi].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (lane == 0) w.msf.x = mx;
    }
    // 2. the bound: the lower edge of the bin, in a 256-bin histogram of the
    //    nonzero sampled order keys over their range, that holds the k-th
    //    largest — at least k sampled keys (so at least k keys) are >= it.
    //    Fewer than k nonzero samples leave the bound at 0.
    {
        const uint32_t lo = w.lo, range = w.hi - lo;
        const int sh = w.lo > w.hi ? 0 : (range < 256u ? 0 : 24 - __clz(range));  // (range >> sh) < 256
        for (int i = tid; i < na; i += kMergeThreads) {
            const uint32_t v = w.set[i];
            if (v != 0u) atomicAdd(&w.hist[(v - lo) >> sh], 1u);
        }
        named_bar_sync(bar_id, kMergeThreads);
        if (warp == 0) {  // lane L owns bins 255-8L ... 248-8L, highest first
            unsigned c[8];
            unsigned lsum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = w.hist[255 - 8 * lane - i];
                lsum += c[i];
            }
            unsigned incl = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            const unsigned excl = incl - lsum;
            if (excl < static_cast<unsigned>(k) && static_cast<unsigned>(k) <= incl) {
                unsigned run = excl;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (run + c[i] >= static_cast<unsigned>(k)) {
                        w.bound = lo + (static_cast<uint32_t>(255 - 8 * lane - i) << sh);
                        break;
                    }
                    run += c[i];
                }
            }
        }
    }
    named_bar_sync(bar_id, kMergeThreads);
    {
        // sum of s_i * exp((m_i - M) / T), one term per thread, block-reduced
        const float M = w.msf.x;
        float t = 0.0f;
        if (tid < G) {
            const float2 v = sms[tid];
            t = v.x == M ? v.y : v.y * expf((v.x - M) * invT);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
        if (lane == 0) w.ssum[warp] = t;
    }
    const uint64_t L = static_cast<uint64_t>(w.bound) << 32;
    // 3. each list's prefix >= L (lists that may go on are read on from L2),
    //    appended at a position taken with one shared atomic per warp
    int n = 0;
    const uint64_t *glist = part_keys + (static_cast<size_t>(tid) * batch_total + b) * k;
    if (tid < G && L != 0ull) {
        while (n < R && lists[tid * R + n] >= L) ++n;
        if (n == R) {
            while (n < k) {
                uint64_t v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = n + u < k ? __ldcg(glist + n + u) : 0ull;
                int c = 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) c += (c == u && v[u] >= L) ? 1 : 0;
                n += c;
                if (c < 8) break;
            }
        }
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    int base = 0;
    if (lane == 31 && incl) base = atomicAdd(&w.total, incl);
    const int off = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - n;
    if (L != 0ull) {
        for (int j = 0; j < n && j < R; ++j)
            if (off + j < kMergeCand) w.cand[off + j] = lists[tid * R + j];
        for (int j = R; j < n; ++j)
            if (off + j < kMergeCand) w.cand[off + j] = __ldcg(glist + j);
    }
    named_bar_sync(bar_id, kMergeThreads);
    const int total = w.total;
    const bool slow = L == 0ull || total > kMergeCand;  // uniform
    float ssum = 0.0f;
#pragma unroll
    for (int q = 0; q < kMergeThreads / 32; ++q) ssum += w.ssum[q];
    const float2 ms = make_float2(w.msf.x, ssum);
    if (slow) {
        if (warp == 0)
            merge_extract_warp(part_keys, G, batch_total, b, k, invT, ms, out_ids, out_logits, out_probs,
                               lane);
    } else {
        // 4. rank among the candidates = final position
        for (int i = tid; i < total; i += kMergeThreads) {
            const uint64_t x = w.cand[i];
            int rank = 0;
#pragma unroll 4
            for (int q = 0; q < total; ++q) rank += w.cand[q] > x;
            if (rank < k) {
                const size_t o = static_cast<size_t>(b) * k + rank;
                const float v = key_value(x);
                out_ids[o] = key_id(x);
                out_logits[o] = v;
                if (out_probs) out_probs[o] = expf((v - ms.x) * invT) / ms.y;
            }
        }
    }
    named_bar_sync(bar_id, kMergeThreads);  // w is free for the next residual
}


// ---------------------------------------------------------------------------
// residual operand prep: x[b][k] (f32 or bf16) -> 16 x Kp rows of the
// table's 16-bit type: rows 0..7 = hi, rows 8..15 = lo (zero padded)
// ---------------------------------------------------------------------------
template <bool BF16T, int XDT>
__global__ void __launch_bounds__(256)
    prep_kernel(const void *__restrict__ resid, int Bc, int K, int Kp, uint16_t *__restrict__ xs,
                int32_t *err) {
    pdl_trigger();  // the projection may start streaming the table now
    pdl_wait();     // x may come from the previous kernel; xs may still be read by it
    const int64_t total = static_cast<int64_t>(8) * Kp;
    int bad = 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int b = static_cast<int>(i / Kp);
        const int kk = static_cast<int>(i % Kp);
        float v = 0.0f;
        if (b < Bc && kk < K) {
            const int64_t src = static_cast<int64_t>(b) * K + kk;
            if (XDT == LHS_F32) v = ld_dep(static_cast<const float *>(resid) + src);
            else v = __uint_as_float(static_cast<uint32_t>(ld_dep(static_cast<const unsigned short *>(resid) + src)) << 16);
        }
        uint16_t hi, lo;
        if (BF16T) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v);
            hi = __bfloat16_as_ushort(h);
            lo = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(h)));
        } else {
            if (!(fabsf(v) < 65504.0f)) bad = 1;
            const __half h = __float2half_rn(v);
            hi = __half_as_ushort(h);
            lo = __half_as_ushort(__float2half_rn(v - __half2float(h)));
        }
        xs[static_cast<int64_t>(b) * Kp + kk] = hi;
        xs[static_cast<int64_t>(8 + b) * Kp + kk] = lo;
    }
    if (bad) set_err(err, LHS_ERRBIT_NONFINITE);
}

// ---------------------------------------------------------------------------
// tensor-core streaming GEMV
// ---------------------------------------------------------------------------
struct TcParams {
    int64_t V;
    int K;
    int nk;          // k stages per block (Kp / 64)
    int Bc;          // residuals in this pass (<= 8)
    int b_off;       // first residual of this pass
    int batch_total;
    int k;           // top-k (0 = raw mode)
    float invT;
    float *raw;      // raw mode: [batch_total x V]
    uint64_t *part_keys;
    float2 *part_ms;
    const void *resid;  // XRES: this pass's residuals [Bc x K]
    int resid_f32;      // XRES: residual dtype f32 (else bf16)
    int32_t *err;
};

// Shared memory of the tensor-core GEMV: the table-tile ring of NST stages,
// barriers and top-k state, then (at the next 1 KB boundary) the residual
// operand: a ring of TMA tiles [NST][16 x 64], or — when it fits — the whole
// operand resident, Kpad / 64 tiles of xres_rows(Bc) rows x 128 bytes,
// written by the consumers themselves.  Both use the TMA 128-byte swizzle:
// within a tile, row r's 16-byte chunk c sits at r * 128 + ((c ^ (r & 7)) << 4).
// The mma reads 16 operand rows per tile, the hi rows of the 8 batch slots
// and then their lo rows.  With at most 3 residuals the resident operand
// keeps only the used ones (hi rows 0 .. Bc-1, lo rows Bc .. 2Bc-1) and one
// zero row, 2 Bc, that every unused slot reads: the rows one 8-row ldmatrix
// reads then have distinct residues mod 8, so no bank conflicts.  From 4
// residuals on it keeps all 16 rows (zeros beyond Bc).
template <int NST>
struct TcSmemT {
    uint8_t a[NST][kAStageBytes];
    uint64_t full[NST];
    uint64_t empty[NST];
    TopkShared tk;
};
template <int NST>
__host__ __device__ constexpr size_t tc_x_offset() { return (sizeof(TcSmemT<NST>) + 1023) & ~size_t(1023); }

__host__ __device__ __forceinline__ int xres_rows(int Bc) { return Bc <= 3 ? 2 * Bc + 1 : 16; }
// resident row of operand row r (r < 8: hi row of batch slot r; else the lo
// row of slot r - 8)
__device__ __forceinline__ int xres_row(int r, int Bc) {
    if (Bc > 3) return r;
    const int b = r & 7;
    return b < Bc ? (r < 8 ? b : Bc + b) : 2 * Bc;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <bool BF16T>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    if (BF16T)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// XRES: the residual operand is resident in shared memory, built by the
// consumers from the residuals (what prep_kernel does otherwise), so the pass
// is one launch and the producer never waits for an earlier kernel.
template <bool BF16T, bool RAW, bool XRES, int NST>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a16,
                   const __grid_constant__ CUtensorMap tm_x, const TcParams p) {
    extern __shared__ uint8_t dyn_smem[];
    TcSmemT<NST> &sm = *reinterpret_cast<TcSmemT<NST> *>(smem_align<1024>(dyn_smem));
    uint8_t *xsm = reinterpret_cast<uint8_t *>(&sm) + tc_x_offset<NST>();
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    int q = 1;
    while (q < p.Bc) q <<= 1;
    const int cap = kCandTotal / q;  // candidate slots per residual

    const int nblk = tc_blocks(p.V, gridDim.x, blockIdx.x);

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    if (tid < kConsumers) topk_init(sm.tk, tid, kConsumers);
    __syncthreads();
    pdl_trigger();  // one wave: the merge may take its place now and wait

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            tma_prefetch_map(&tm_a);
            tma_prefetch_map(&tm_a16);
            tma_prefetch_map(&tm_x);
            const uint32_t total = static_cast<uint32_t>(nblk) * p.nk;
            auto block_rows = [&](int blk) {
                int64_t row0;
                int rows;
                tc_block(p.V, gridDim.x, blockIdx.x, blk, row0, rows);
                return rows;
            };
            auto issue_a = [&](uint32_t j) {
                const int blk = j / p.nk, kc = j % p.nk, s = j % NST;
                int64_t row0;
                int rows;
                tc_block(p.V, gridDim.x, blockIdx.x, blk, row0, rows);
                if (rows == BM) {
                    tma_load_2d(sm.a[s], &tm_a, &sm.full[s], kc * BK, static_cast<int32_t>(row0));
                } else {
                    const int n16 = (rows + kBoxRowsSmall - 1) / kBoxRowsSmall;
                    for (int u = 0; u < n16; ++u)
                        tma_load_2d(sm.a[s] + u * kBoxRowsSmall * BK * 2, &tm_a16, &sm.full[s],
                                    kc * BK, static_cast<int32_t>(row0 + u * kBoxRowsSmall));
                }
            };
            auto stage_bytes = [&](uint32_t j) {
                const int rows = block_rows(j / p.nk);
                const int n16 = (rows + kBoxRowsSmall - 1) / kBoxRowsSmall;
                return static_cast<uint32_t>(rows == BM ? kAStageBytes : n16 * kBoxRowsSmall * BK * 2) +
                       (XRES ? 0u : static_cast<uint32_t>(kXStageBytes));
            };
            // The table is never written by an earlier kernel, so the first
            // ring's worth of table tiles is requested before waiting for the
            // residual operand the preceding kernel prepares.
            const uint32_t pre = total < NST ? total : NST;
            for (uint32_t j = 0; j < pre; ++j) {
                mbar_arrive_expect_tx(&sm.full[j], stage_bytes(j));
                issue_a(j);
            }
            if (!XRES) {
                pdl_wait();
                for (uint32_t j = 0; j < pre; ++j)
                    tma_load_2d(xsm + j * kXStageBytes, &tm_x, &sm.full[j], (j % p.nk) * BK, 0);
            }
            uint32_t it = pre;
            for (; it < total; ++it) {
                const int s = it % NST;
                const uint32_t ph = (it / NST) & 1;
                if (!mbar_wait(&sm.empty[s], ph ^ 1, kWaitTimeoutNs)) {
                    // consumers stopped releasing slots; they record their
                    // own timeout and leave together
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    break;
                }
                if (ld_volatile(&sm.tk.abort_flag)) break;
                mbar_arrive_expect_tx(&sm.full[s], stage_bytes(it));
                issue_a(it);
                if (!XRES) tma_load_2d(xsm + s * kXStageBytes, &tm_x, &sm.full[s], (it % p.nk) * BK, 0);
            }
            // drain: every issued stage must land before the CTA exits
            const uint32_t issued = it;
            for (uint32_t j = (issued > NST ? issued - NST : 0); j < issued; ++j) {
                const int s = j % NST;
                if (!mbar_wait(&sm.full[s], (j / NST) & 1, kWaitTimeoutNs)) {
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int g = lane >> 2, t = lane & 3;
    const int a_row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int a_csel = lane >> 4;
    const int x_row = XRES ? xres_row((lane & 7) + ((lane >> 4) << 3), p.Bc) : (lane & 7) + ((lane >> 4) << 3);
    const int x_csel = (lane >> 3) & 1;
    const uint32_t x_tile = XRES ? static_cast<uint32_t>(xres_rows(p.Bc)) * 128u : static_cast<uint32_t>(kXStageBytes);
    float m_st[2] = {-INFINITY, -INFINITY}, s_st[2] = {0.0f, 0.0f};
    if (XRES) {
        // the residuals may come from the previous kernel, and the partial
        // lists written below may still be read by it
        pdl_wait();
        const int Kp = p.nk * BK;
        const bool compact = p.Bc <= 3;
        const int xtile = xres_rows(p.Bc) * 128;
        int bad = 0;
        for (int b = 0; b < (compact ? p.Bc : 8); ++b) {
            const int rh = b, rl = compact ? p.Bc + b : 8 + b;  // resident rows of slot b (hi, lo)
            for (int kk = tid; kk < Kp; kk += kConsumers) {
                float v = 0.0f;
                if (b < p.Bc && kk < p.K) {
                    const int64_t src = static_cast<int64_t>(b) * p.K + kk;
                    if (p.resid_f32) v = ld_dep(static_cast<const float *>(p.resid) + src);
                    else v = __uint_as_float(static_cast<uint32_t>(ld_dep(static_cast<const unsigned short *>(p.resid) + src)) << 16);
                }
                uint16_t hi, lo;
                if (BF16T) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(v);
                    hi = __bfloat16_as_ushort(h);
                    lo = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(h)));
                } else {
                    if (!(fabsf(v) < 65504.0f)) bad = 1;
                    const __half h = __float2half_rn(v);
                    hi = __half_as_ushort(h);
                    lo = __half_as_ushort(__float2half_rn(v - __half2float(h)));
                }
                // rows rh and rl of tile kk / 64
                const int e = kk & (BK - 1);
                uint8_t *tile = xsm + (kk / BK) * xtile;
                *reinterpret_cast<uint16_t *>(tile + rh * 128 + ((((e >> 3) ^ (rh & 7)) << 4) | ((e & 7) * 2))) = hi;
                *reinterpret_cast<uint16_t *>(tile + rl * 128 + ((((e >> 3) ^ (rl & 7)) << 4) | ((e & 7) * 2))) = lo;
            }
        }
        if (compact) {
            // the zero row that the unused batch slots read
            for (int i = tid; i < p.nk * 8; i += kConsumers)
                *reinterpret_cast<uint4 *>(xsm + (i >> 3) * xtile + 2 * p.Bc * 128 + (i & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
        if (bad && p.Bc > 0) set_err(p.err, LHS_ERRBIT_NONFINITE);
        named_bar_sync(kBarAll, kConsumers);
    }
    uint32_t it = 0;
    for (int blk = 0; blk < nblk; ++blk) {
        int64_t row0;
        int rows;
        tc_block(p.V, gridDim.x, blockIdx.x, blk, row0, rows);
        const bool active = warp * 16 < rows;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kc = 0; kc < p.nk; ++kc, ++it) {
            const int s = it % NST;
            const uint32_t ph = (it / NST) & 1;
            if (!ld_volatile(&sm.tk.abort_flag)) {
                if (!mbar_wait(&sm.full[s], ph, kWaitTimeoutNs)) {
                    if (lane == 0) {
                        set_err(p.err, LHS_ERRBIT_TIMEOUT);
                        sm.tk.abort_flag = 1;
                    }
                } else if (active) {
                    const uint32_t abase = smem_u32(sm.a[s]);
                    const uint32_t xbase = smem_u32(xsm) + static_cast<uint32_t>(XRES ? kc : s) * x_tile;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {
                        const int ca = 2 * ks + a_csel;
                        const int cx = 2 * ks + x_csel;
                        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                        ldsm_x4(abase + a_row * 128 + ((ca ^ (a_row & 7)) << 4), a0, a1, a2, a3);
                        ldsm_x4(xbase + x_row * 128 + ((cx ^ (x_row & 7)) << 4), b0, b1, b2, b3);
                        mma16816<BF16T>(acc, a0, a1, a2, a3, b0, b1);  // hi
                        mma16816<BF16T>(acc, a0, a1, a2, a3, b2, b3);  // lo
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
        // epilogue: thread holds rows (g, g+8) x columns (2t, 2t+1)
        if (active && !ld_volatile(&sm.tk.abort_flag)) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int64_t v = row0 + warp * 16 + g + 8 * r;
                if (v < row0 + rows) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int b = 2 * t + c;
                        if (b < p.Bc) {
                            const float val = acc[2 * r + c];
                            if (RAW) {
                                p.raw[static_cast<int64_t>(p.b_off + b) * p.V + v] = val;
                            } else {
                                ms_update(m_st[c], s_st[c], val, p.invT);
                                topk_offer(sm.tk, b, cap, val, static_cast<int32_t>(v));
                            }
                        }
                    }
                }
            }
        }
        if (!RAW) topk_round_end(sm.tk, tid, kConsumers, p.Bc, p.k, cap, BM);
        else named_bar_sync(kBarAll, kConsumers);
        // the flag only changes inside the main loop, before the barrier
        // above, so every consumer reads the same value here
        if (ld_volatile(&sm.tk.abort_flag)) break;
    }
    // the flag only changes inside the main loop: uniform here
    if (RAW || ld_volatile(&sm.tk.abort_flag)) return;
    // per-warp (m, s) for columns 2t, 2t+1 over g (lanes t, t+4, ...): the
    // max first, then every lane's sum rescaled to it at once and added
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        float M = m_st[c];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        float S = ms_rescaled(m_st[c], s_st[c], M, p.invT);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
        if (g == 0 && 2 * t + c < kBatchChunk) sm.tk.ms_warp[warp][2 * t + c] = make_float2(M, S);
    }
    topk_finish(sm.tk, tid, kConsumers, p.Bc, p.k, cap, p.b_off, p.batch_total, p.part_keys,
                p.part_ms, p.invT);
}

// ---------------------------------------------------------------------------
// CUDA-core streaming GEMV (f32 / Q8_0 / ragged-hidden tables)
// ---------------------------------------------------------------------------
struct SimtParams {
    const uint8_t *table;
    int64_t V;
    int K;
    int64_t row_bytes;
    const void *resid;  // first residual of this pass
    int resid_dtype;
    int Bc, b_off, batch_total, k;
    float invT;
    float *raw;
    uint64_t *part_keys;
    float2 *part_ms;
    int32_t *err;
};

template <int DT>
__device__ __forceinline__ float table_elem(const uint8_t *row, int j) {
    if (DT == LHS_F32) return __ldg(reinterpret_cast<const float *>(row) + j);
    if (DT == LHS_F16)
        return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short *>(row) + j)));
    if (DT == LHS_BF16)
        return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(row) + j)) << 16);
    const uint8_t *blk = row + (j >> 5) * 34;
    const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short *>(blk))));
    return __fmul_rn(d, static_cast<float>(static_cast<int8_t>(__ldg(blk + 2 + (j & 31)))));
}

// Dot products of kSimtRows rows with the Bc residuals in shared memory,
// 8 elements per lane step (rows 16-byte aligned, Q8_0 2-byte; K % 8 == 0):
// every row's loads of a step are issued before its multiplies.
constexpr int kSimtRows = 4;

template <int DT>
__device__ __forceinline__ void simt_rows8(const uint8_t *const (&rows)[kSimtRows], int K, const float *xs,
                                           int Bc, int lane, float (&acc)[kSimtRows][kBatchChunk]) {
    const int ng = K >> 3;
    for (int g = lane; g < ng; g += 32) {
        float e[kSimtRows][8];
#pragma unroll
        for (int r = 0; r < kSimtRows; ++r) row_elements8<DT>(rows[r], g, e[r]);
#pragma unroll
        for (int b = 0; b < kBatchChunk; ++b) {
            if (b < Bc) {
                const float4 x0 = *reinterpret_cast<const float4 *>(xs + b * K + 8 * g);
                const float4 x1 = *reinterpret_cast<const float4 *>(xs + b * K + 8 * g + 4);
                const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int r = 0; r < kSimtRows; ++r)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[r][b] = fmaf(e[r][i], xv[i], acc[r][b]);
            }
        }
    }
}

template <int DT, bool RAW, bool VEC>
__global__ void __launch_bounds__(kSimtThreads, 1) gemv_simt_kernel(const SimtParams p) {
    extern __shared__ uint8_t dyn_smem[];
    TopkShared &tk = *reinterpret_cast<TopkShared *>(dyn_smem);
    float *xs = reinterpret_cast<float *>(dyn_smem + ((sizeof(TopkShared) + 15) & ~size_t(15)));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int q = 1;
    while (q < p.Bc) q <<= 1;
    const int cap = kCandTotal / q;
    pdl_trigger();
    pdl_wait();

    for (int64_t i = tid; i < static_cast<int64_t>(p.Bc) * p.K; i += kSimtThreads) {
        float v;
        if (p.resid_dtype == LHS_F32) v = ld_dep(static_cast<const float *>(p.resid) + i);
        else v = __uint_as_float(static_cast<uint32_t>(ld_dep(static_cast<const unsigned short *>(p.resid) + i)) << 16);
        xs[i] = v;
    }
    topk_init(tk, tid, kSimtThreads);
    __syncthreads();

    int64_t r0, r1;
    cta_rows(p.V, gridDim.x, blockIdx.x, r0, r1);
    const int nblk = static_cast<int>((r1 - r0 + BM - 1) / BM);
    float m_st = -INFINITY, s_st = 0.0f;  // lane b < Bc: column b
    for (int blk = 0; blk < nblk; ++blk) {
        const int64_t row0 = r0 + static_cast<int64_t>(blk) * BM;
        for (int rr = 0; rr < 16; rr += kSimtRows) {
            const int64_t v0 = row0 + warp * 16 + rr;
            if (v0 >= r1) break;
            float acc[kSimtRows][kBatchChunk];
#pragma unroll
            for (int r = 0; r < kSimtRows; ++r)
#pragma unroll
                for (int b = 0; b < kBatchChunk; ++b) acc[r][b] = 0.0f;
            if (VEC) {
                // rows past the range read row v0 again; their sums are dropped
                const uint8_t *rows[kSimtRows];
#pragma unroll
                for (int r = 0; r < kSimtRows; ++r) rows[r] = p.table + (v0 + r < r1 ? v0 + r : v0) * p.row_bytes;
                simt_rows8<DT>(rows, p.K, xs, p.Bc, lane, acc);
            } else {
#pragma unroll
                for (int r = 0; r < kSimtRows; ++r) {
                    const uint8_t *row = p.table + (v0 + r < r1 ? v0 + r : v0) * p.row_bytes;
                    for (int j = lane; j < p.K; j += 32) {
                        const float e = table_elem<DT>(row, j);
#pragma unroll
                        for (int b = 0; b < kBatchChunk; ++b)
                            if (b < p.Bc) acc[r][b] = fmaf(e, xs[b * p.K + j], acc[r][b]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kSimtRows; ++r) {
                const int64_t v = v0 + r;
#pragma unroll
                for (int b = 0; b < kBatchChunk; ++b) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[r][b] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][b], o);
                }
                float mine = 0.0f;
#pragma unroll
                for (int b = 0; b < kBatchChunk; ++b)
                    if (lane == b) mine = acc[r][b];
                if (v < r1 && lane < p.Bc) {
                    if (RAW) {
                        p.raw[static_cast<int64_t>(p.b_off + lane) * p.V + v] = mine;
                    } else {
                        ms_update(m_st, s_st, mine, p.invT);
                        topk_offer(tk, lane, cap, mine, static_cast<int32_t>(v));
                    }
                }
            }
        }
        if (!RAW) topk_round_end(tk, tid, kSimtThreads, p.Bc, p.k, cap, BM);
    }
    if (RAW) return;
    if (lane < kBatchChunk) tk.ms_warp[warp][lane] = make_float2(m_st, s_st);
    topk_finish(tk, tid, kSimtThreads, p.Bc, p.k, cap, p.b_off, p.batch_total, p.part_keys,
                p.part_ms, p.invT);
}

// ---------------------------------------------------------------------------
// Bulk-stream CUDA-core GEMV (f32 tables, rows a multiple of 16
// bytes and at most kBulkRowBytesMax): a producer warp copies 32 whole rows
// per stage — one contiguous cp.async.bulk — into a 4-stage ring (one top-k
// round of 128 rows in flight); each of 16 consumer warps multiplies two
// rows of each stage (w and w + 16) side by side, 8 elements per lane step,
// with the residuals in shared memory.  The same per-CTA top-k lists as the
// other GEMVs.
// ---------------------------------------------------------------------------
constexpr int kBulkRows = 32;                // rows per stage: 4 per consumer warp
constexpr int kBulkStages = BM / kBulkRows;  // 4: one top-k round of 128 rows in flight
constexpr int kBulkWarps = 16;               // consumer warps
constexpr int kBulkConsumers = kBulkWarps * 32;
constexpr int kBulkThreads = kBulkConsumers + 32;  // + the producer warp
constexpr int kBulkRowsPerWarp = kBulkRows / kBulkWarps;
constexpr int kBulkRowBytesMax = 1024;  // ring: 4 x 32 rows <= 128 KB

// Elements 8g .. 8g+7 of an f32 row held in shared memory.
template <int DT>
__device__ __forceinline__ void smem_row8(const uint8_t *row, int g, float (&v)[8]) {
    static_assert(DT == LHS_F32, "the bulk-stream GEMV serves f32 tables");
    const float4 a = *reinterpret_cast<const float4 *>(row + 32 * g);
    const float4 b = *reinterpret_cast<const float4 *>(row + 32 * g + 16);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

struct BulkParams {
    const uint8_t *table;
    int64_t V;
    int K;
    int64_t row_bytes;
    const void *resid;
    int resid_dtype;
    int Bc, b_off, batch_total, k;
    float invT;
    float *raw;
    uint64_t *part_keys;
    float2 *part_ms;
    int32_t *err;
};

// Shared memory: [ring kBulkStages x 16 rows][full, empty][TopkShared][xs Bc x K f32]
__host__ __device__ __forceinline__ size_t bulk_ring_bytes(int64_t row_bytes) {
    return static_cast<size_t>(kBulkStages) * kBulkRows * static_cast<size_t>(row_bytes);
}
__host__ __device__ __forceinline__ size_t bulk_tk_offset(int64_t row_bytes) {
    return ((bulk_ring_bytes(row_bytes) + 2 * kBulkStages * 8) + 127) & ~size_t(127);
}
__host__ __device__ __forceinline__ size_t bulk_xs_offset(int64_t row_bytes) {
    return (bulk_tk_offset(row_bytes) + sizeof(TopkShared) + 15) & ~size_t(15);
}

// BC: residual columns the loops are unrolled for (p.Bc <= BC).
template <int DT, bool RAW, int BC>
__global__ void __launch_bounds__(kBulkThreads, 1) gemv_bulk_kernel(const BulkParams p) {
    extern __shared__ uint8_t dyn_smem[];
    uint8_t *base = smem_align<128>(dyn_smem);
    uint8_t *ring = base;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + bulk_ring_bytes(p.row_bytes));
    uint64_t *empty = full + kBulkStages;
    TopkShared &tk = *reinterpret_cast<TopkShared *>(base + bulk_tk_offset(p.row_bytes));
    float *xs = reinterpret_cast<float *>(base + bulk_xs_offset(p.row_bytes));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int q = 1;
    while (q < p.Bc) q <<= 1;
    const int cap = kCandTotal / q;
    const size_t stage_bytes = static_cast<size_t>(kBulkRows) * p.row_bytes;

    int64_t r0, r1;
    cta_rows(p.V, gridDim.x, blockIdx.x, r0, r1);
    const uint32_t total = static_cast<uint32_t>((r1 - r0 + kBulkRows - 1) / kBulkRows);

    if (tid == 0) {
        for (int s = 0; s < kBulkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkWarps);
        }
        fence_mbar_init();
    }
    if (tid < kBulkConsumers) topk_init(tk, tid, kBulkConsumers);
    __syncthreads();
    pdl_trigger();

    if (warp == kBulkWarps) {
        // ---------------- producer: the table only, never written by an earlier kernel
        if (lane == 0) {
            auto issue = [&](uint32_t j) {
                const int s = j % kBulkStages;
                const int64_t row0 = r0 + static_cast<int64_t>(j) * kBulkRows;
                const int64_t nrows = (r1 - row0) < kBulkRows ? (r1 - row0) : kBulkRows;
                const uint32_t bytes = static_cast<uint32_t>(nrows * p.row_bytes);
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_load(ring + s * stage_bytes, p.table + row0 * p.row_bytes, bytes, &full[s]);
            };
            const uint32_t pre = total < kBulkStages ? total : kBulkStages;
            for (uint32_t j = 0; j < pre; ++j) issue(j);
            uint32_t it = pre;
            for (; it < total; ++it) {
                const int s = it % kBulkStages;
                if (!mbar_wait(&empty[s], ((it / kBulkStages) & 1) ^ 1, kWaitTimeoutNs)) {
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    break;
                }
                if (ld_volatile(&tk.abort_flag)) break;
                issue(it);
            }
            // drain: every issued copy must land before the CTA exits
            for (uint32_t j = (it > kBulkStages ? it - kBulkStages : 0); j < it; ++j)
                if (!mbar_wait(&full[j % kBulkStages], (j / kBulkStages) & 1, kWaitTimeoutNs)) {
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    break;
                }
        }
        return;
    }

    // ---------------- consumers
    pdl_wait();  // residuals may come from the previous kernel; partial lists may still be read by it
    for (int64_t i = tid; i < static_cast<int64_t>(p.Bc) * p.K; i += kBulkConsumers) {
        float v;
        if (p.resid_dtype == LHS_F32) v = ld_dep(static_cast<const float *>(p.resid) + i);
        else v = __uint_as_float(static_cast<uint32_t>(ld_dep(static_cast<const unsigned short *>(p.resid) + i)) << 16);
        xs[i] = v;
    }
    named_bar_sync(kBarAll, kBulkConsumers);
    float m_st = -INFINITY, s_st = 0.0f;  // lane b < Bc: column b
    const int ng = p.K >> 3;
    for (uint32_t it = 0; it < total; ++it) {
        const int s = it % kBulkStages;
        const int64_t row0 = r0 + static_cast<int64_t>(it) * kBulkRows;
        const int nrows = static_cast<int>((r1 - row0) < kBulkRows ? (r1 - row0) : kBulkRows);
        if (!ld_volatile(&tk.abort_flag)) {
            if (!mbar_wait(&full[s], (it / kBulkStages) & 1, kWaitTimeoutNs)) {
                if (lane == 0) {
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    tk.abort_flag = 1;
                }
            } else {
                // rows warp + 16h of the stage, side by side; two accumulation
                // chains per row and column (even / odd elements)
                constexpr int RW = kBulkRowsPerWarp;
                int nr = 0;  // warp-uniform
#pragma unroll
                for (int h = 0; h < RW; ++h) nr += warp + kBulkWarps * h < nrows;
                if (nr > 0) {
                    const uint8_t *rows[RW];
#pragma unroll
                    for (int h = 0; h < RW; ++h)
                        rows[h] = ring + s * stage_bytes + (h < nr ? warp + kBulkWarps * h : warp) * p.row_bytes;
                    float c0[RW][BC], c1[RW][BC];
#pragma unroll
                    for (int h = 0; h < RW; ++h)
#pragma unroll
                        for (int b = 0; b < BC; ++b) c0[h][b] = c1[h][b] = 0.0f;
                    for (int g = lane; g < ng; g += 32) {
                        float e[RW][8];
#pragma unroll
                        for (int h = 0; h < RW; ++h) smem_row8<DT>(rows[h], g, e[h]);
#pragma unroll
                        for (int b = 0; b < BC; ++b) {
                            if (BC == 1 || b < p.Bc) {
                                const float4 x0 = *reinterpret_cast<const float4 *>(xs + b * p.K + 8 * g);
                                const float4 x1 = *reinterpret_cast<const float4 *>(xs + b * p.K + 8 * g + 4);
                                const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                                for (int i = 0; i < 8; i += 2)
#pragma unroll
                                    for (int h = 0; h < RW; ++h) {
                                        c0[h][b] = fmaf(e[h][i], xv[i], c0[h][b]);
                                        c1[h][b] = fmaf(e[h][i + 1], xv[i + 1], c1[h][b]);
                                    }
                            }
                        }
                    }
#pragma unroll
                    for (int h = 0; h < RW; ++h) {
                        if (h < nr) {
                            float acc[BC];
#pragma unroll
                            for (int b = 0; b < BC; ++b) acc[b] = c0[h][b] + c1[h][b];
#pragma unroll
                            for (int b = 0; b < BC; ++b)
#pragma unroll
                                for (int o = 16; o > 0; o >>= 1) acc[b] += __shfl_xor_sync(0xFFFFFFFFu, acc[b], o);
                            float mine = 0.0f;
#pragma unroll
                            for (int b = 0; b < BC; ++b)
                                if (lane == b) mine = acc[b];
                            const int64_t v = row0 + warp + kBulkWarps * h;
                            if (lane < p.Bc) {
                                if (RAW) {
                                    p.raw[static_cast<int64_t>(p.b_off + lane) * p.V + v] = mine;
                                } else {
                                    ms_update(m_st, s_st, mine, p.invT);
                                    topk_offer(tk, lane, cap, mine, static_cast<int32_t>(v));
                                }
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if ((it % kBulkStages) == kBulkStages - 1 || it + 1 == total) {
            if (!RAW) topk_round_end(tk, tid, kBulkConsumers, p.Bc, p.k, cap, BM);
            else named_bar_sync(kBarAll, kBulkConsumers);
            // the flag only changes inside the loop, before the barrier above
            if (ld_volatile(&tk.abort_flag)) break;
        }
    }
    if (RAW || ld_volatile(&tk.abort_flag)) return;
    if (lane < kBatchChunk) tk.ms_warp[warp][lane] = make_float2(m_st, s_st);
    topk_finish(tk, tid, kBulkConsumers, p.Bc, p.k, cap, p.b_off, p.batch_total, p.part_keys, p.part_ms, p.invT);
}

// ---------------------------------------------------------------------------
// merge: global top-k per residual from G partial lists, sorted, + probs
// ---------------------------------------------------------------------------

// Top-k of G unsorted lists (a list of `len` keys every `stride`, padded
// with 0: no real key is 0) for residual b, by 256 threads, with a few
// histogram passes instead of a digit-by-digit radix select:
//  A. each warp reads whole lists (no division per load) and appends their
//     non-empty keys to shared memory, tracking the range [lo, hi] of the
//     keys' upper 32 bits (the logit's order key);
//  B. a histogram of (order key - base) >> sh over 256 bins, sh the smallest
//     shift that fits the window in 256 bins (first window: [lo, hi]);
//  C. the bin holding the k-th largest key: the keys in it and in the bins
//     above it (at least k) are the candidates; no other key can be in the
//     top-k.  While they are more than kMergeRankDirect, B and C repeat on
//     that bin alone (256 sub-bins of it), down to single order keys;
//  D. a candidate's rank among the candidates is its final position.
// Fewer than k non-empty keys, or more than kMergeHistCand candidates that
// share one order key (tied logits), take the radix select instead.
constexpr int kMergeRankDirect = 256;

__device__ void merge_column_hist(const uint64_t *part_keys, const float2 *part_ms, int G, int stride,
                                  int len, int batch_total, int b, int k, float invT, int32_t *out_ids,
                                  float *out_logits, float *out_probs, MergeSmemHead &h, uint64_t *keys,
                                  int tid) {
    constexpr int W = 8, U = 8;
    const int lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        h.n = 0;
        h.ncand = 0;
        h.lo = 0xFFFFFFFFu;
        h.hi = 0u;
    }
    // this thread's share of the softmax partials
    float2 ms = make_float2(-INFINITY, 0.0f);
    for (int g = tid; g < G; g += 256)
        ms = ms_combine(ms, __ldcg(part_ms + static_cast<size_t>(g) * batch_total + b), invT);
    __syncthreads();
    // A. lists warp, warp + W, ...; lane walks entries lane, lane + 32, ...
    //    of the warp's concatenated lists
    const int ngw = warp < G ? (G - warp + W - 1) / W : 0;
    const int tot = ngw * len;
    int li = lane / len, lj = lane % len;
    unsigned lo = 0xFFFFFFFFu, hi = 0u;
    for (int base = 0; base < tot; base += 32 * U) {
        uint64_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            v[u] = 0ull;
            if (base + 32 * u + lane < tot)
                v[u] = __ldcg(part_keys + (static_cast<size_t>(warp + W * li) * batch_total + b) * stride + lj);
            lj += 32;
            while (lj >= len) {
                lj -= len;
                ++li;
            }
        }
        unsigned m[U];
        int cnt = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            m[u] = __ballot_sync(0xFFFFFFFFu, v[u] != 0ull);
            cnt += __popc(m[u]);
        }
        if (cnt == 0) continue;  // warp-uniform
        int pos = 0;
        if (lane == 0) pos = atomicAdd(&h.n, cnt);
        pos = __shfl_sync(0xFFFFFFFFu, pos, 0);
        const unsigned below = (1u << lane) - 1u;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (v[u] != 0ull) {
                keys[pos + __popc(m[u] & below)] = v[u];
                const unsigned up = static_cast<unsigned>(v[u] >> 32);
                lo = min(lo, up);
                hi = max(hi, up);
            }
            pos += __popc(m[u]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
    }
    if (lane == 0 && lo <= hi) {
        atomicMin(&h.lo, lo);
        atomicMax(&h.hi, hi);
    }
    {
        float mx = ms.x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (lane == 0) h.wmax[warp] = mx;
    }
    __syncthreads();
    const int n = h.n;
    if (n < k) {
        __syncthreads();  // every thread has read h.n before the radix select reuses h
        merge_column(part_keys, part_ms, G, stride, len, batch_total, b, k, invT, out_ids, out_logits,
                     out_probs, h, keys, tid, 1);
        return;
    }
    // the softmax sum rescaled to the overall max, one term per thread
    float M = h.wmax[0];
#pragma unroll
    for (int q = 1; q < W; ++q) M = fmaxf(M, h.wmax[q]);
    {
        float t = ms.x == M ? ms.y : (ms.x == -INFINITY ? 0.0f : ms.y * expf((ms.x - M) * invT));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
        if (lane == 0) h.wsum[warp] = t;
    }
    // B, C. window [base, base + span), bins of 2^sh order keys; keys above
    // the window are counted in `above` (all candidates), `need` of the
    // top-k are still inside it
    unsigned base = h.lo;
    const unsigned range = h.hi - base;
    uint64_t span = static_cast<uint64_t>(range) + 1;
    int sh = range < 256u ? 0 : 24 - __clz(range);  // (range >> sh) < 256
    int need = k, above = 0;
    unsigned edge;
    int ncand;
    for (;;) {
        h.hist[tid] = 0u;
        __syncthreads();
        for (int i = tid; i < n; i += 256) {
            const unsigned up = static_cast<unsigned>(keys[i] >> 32);
            if (up >= base && static_cast<uint64_t>(up - base) < span) atomicAdd(&h.hist[(up - base) >> sh], 1u);
        }
        __syncthreads();
        // warp 0: lane L owns bins 255-8L ... 248-8L, highest first
        if (warp == 0) {
            unsigned c[8];
            unsigned lsum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = h.hist[255 - 8 * lane - i];
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
                        h.bin = 255 - 8 * lane - i;
                        h.above = static_cast<int>(run);
                        break;
                    }
                    run += c[i];
                }
            }
        }
        __syncthreads();
        const int bin = h.bin, in_above = h.above;
        const int in_bin = static_cast<int>(h.hist[bin]);
        edge = base + (static_cast<unsigned>(bin) << sh);
        ncand = above + in_above + in_bin;
        if (ncand <= kMergeRankDirect || sh == 0) break;
        // refine inside the bin: at most 256 sub-bins of it
        above += in_above;
        need -= in_above;
        base = edge;
        span = static_cast<uint64_t>(1) << sh;
        sh = sh > 8 ? sh - 8 : 0;
        __syncthreads();  // every thread has read hist / bin before they change
    }
    if (ncand > kMergeHistCand) {
        __syncthreads();  // h is read; the radix select reuses it
        merge_column(part_keys, part_ms, G, stride, len, batch_total, b, k, invT, out_ids, out_logits,
                     out_probs, h, keys, tid, 1);
        return;
    }
    // D. gather the candidates (order key >= edge), then rank them
    for (int i0 = 0; i0 < n; i0 += 256) {
        const int i = i0 + tid;
        const bool c = i < n && static_cast<unsigned>(keys[i] >> 32) >= edge;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, c);
        if (m == 0u) continue;
        int pos = 0;
        if (lane == 0) pos = atomicAdd(&h.ncand, __popc(m));
        pos = __shfl_sync(0xFFFFFFFFu, pos, 0);
        if (c) h.cand[pos + __popc(m & ((1u << lane) - 1u))] = keys[i];
    }
    float S = 0.0f;
#pragma unroll
    for (int q = 0; q < W; ++q) S += h.wsum[q];
    __syncthreads();
    for (int i = tid; i < ncand; i += 256) {
        const uint64_t x = h.cand[i];
        int rank = 0;
#pragma unroll 4
        for (int q = 0; q < ncand; ++q) rank += h.cand[q] > x;
        if (rank < k) {
            const size_t o = static_cast<size_t>(b) * k + rank;
            const float v = key_value(x);
            out_ids[o] = key_id(x);
            out_logits[o] = v;
            if (out_probs) out_probs[o] = expf((v - M) * invT) / S;
        }
    }
}

__global__ void __launch_bounds__(256)
    merge_kernel(const uint64_t *__restrict__ part_keys, const float2 *__restrict__ part_ms, int G,
                 int stride, int len, int batch_total, int k, float invT, int32_t *__restrict__ out_ids,
                 float *__restrict__ out_logits, float *__restrict__ out_probs) {
    extern __shared__ uint8_t dyn_smem[];
    MergeSmemHead &h = *reinterpret_cast<MergeSmemHead *>(dyn_smem);
    uint64_t *keys = reinterpret_cast<uint64_t *>(dyn_smem + ((sizeof(MergeSmemHead) + 15) & ~size_t(15)));
    pdl_trigger();
    pdl_wait();
    merge_column_hist(part_keys, part_ms, G, stride, len, batch_total, blockIdx.x, k, invT, out_ids,
                      out_logits, out_probs, h, keys, threadIdx.x);
}

// Merge of the GEMV kernels' sorted lists, one block per residual.  The
// host guarantees G <= kMergeThreads and R = merge_stage_entries(G, k).
__global__ void __launch_bounds__(kMergeThreads)
    merge_sorted_kernel(const uint64_t *__restrict__ part_keys, const float2 *__restrict__ part_ms,
                        int G, int batch_total, int k, int R, float invT, int32_t *__restrict__ out_ids,
                        float *__restrict__ out_logits, float *__restrict__ out_probs) {
    __shared__ MergeWork w;
    extern __shared__ uint64_t lists[];  // [G][R], then G float2
    float2 *sms = reinterpret_cast<float2 *>(lists + G * R);
    pdl_trigger();
    w.hist[threadIdx.x] = 0u;  // kMergeThreads == 256 bins
    if (threadIdx.x == 0) {
        w.lo = 0xFFFFFFFFu;
        w.hi = 0u;
    }
    pdl_wait();
    stage_sorted_lists(part_keys, part_ms, G, k, R, batch_total, blockIdx.x, lists, sms, threadIdx.x,
                       kMergeThreads);
    __syncthreads();
    merge_column_sorted(lists, R, sms, G, k, invT, part_keys, batch_total, blockIdx.x, out_ids, out_logits,
                        out_probs, w, threadIdx.x, 1);
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D map over a row-major [rows x cols] 16-bit matrix with a given row
// pitch; box = box_cols x box_rows, 128-byte swizzle, zero fill outside.
bool make_tma_map_16bit(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                    uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, bool bf16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                          const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tma_map_u16_plain(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                            uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// dynamic shared memory of the tensor-core GEMV with nst stages and passes
// of up to bc residuals: alignment slack + layout
size_t tc_smem_bytes(bool xres, int kpad, int nst, int bc) {
    const size_t x_off = nst == kStagesCompact ? tc_x_offset<kStagesCompact>()
                         : nst == kStagesRing  ? tc_x_offset<kStagesRing>()
                                               : tc_x_offset<kStagesResident>();
    return 1024 + x_off +
           (xres ? static_cast<size_t>(kpad / BK) * xres_rows(bc) * 128 : static_cast<size_t>(nst) * kXStageBytes);
}
constexpr size_t kSimtXBytesMax = 96 * 1024;

size_t simt_smem_bytes(int Bc, int K) {
    return ((sizeof(TopkShared) + 15) & ~size_t(15)) + static_cast<size_t>(Bc) * K * 4;
}
size_t bulk_smem_bytes(int64_t row_bytes, int Bc, int K) {
    return 128 + bulk_xs_offset(row_bytes) + static_cast<size_t>(Bc) * K * 4;
}
size_t merge_smem_bytes(int G, int k) {
    return ((sizeof(MergeSmemHead) + 15) & ~size_t(15)) + static_cast<size_t>(G) * k * 8;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }


}  // namespace

int plan_lm_head(const lhs_table &t, int32_t batch, int32_t k, int32_t resid_dtype,
                 const DeviceInfo &dev, LmHeadPlan *plan) {
    LmHeadPlan p{};
    // tensor-core path: 16-bit table, TMA-able rows (16-byte pitch), and at
    // least one full box in each dimension
    const bool tc = (t.dtype == LHS_F16 || t.dtype == LHS_BF16) && (t.hidden % 8 == 0) &&
                    t.hidden >= BK && t.vocab >= BM;
    // batches beyond one GEMV pass, with operands that are exact in bf16,
    // are a dense contraction: tcgen05 GEMM
    bool gemm = tc && t.dtype == LHS_BF16 && resid_dtype == LHS_BF16 && batch > kBatchChunk &&
                dev.num_sms >= 2;
    const int64_t units = (t.vocab + 15) / 16;
    p.kpad = static_cast<int>(align_up(t.hidden, BK));
    int clusters = 0;
    if (gemm) {
        clusters = gemm_lm_head_clusters(dev);
        // the epilogue stores vocab rows as 16-bit offsets within a cluster's range
        const int64_t tiles = (t.vocab + 255) / 256;
        if ((tiles + clusters - 1) / clusters * 256 > 65535) gemm = false;
    }
    // Q8_0 tables whose rows are whole 256-value stages (272-byte multiples,
    // a TMA pitch), 16-byte aligned, with a ring of at least two stages
    const int bc1 = batch < 1 ? 1 : (batch < kBatchChunk ? batch : kBatchChunk);
    const int q8_nst = (t.dtype == LHS_Q8_0 && t.hidden % 256 == 0 && t.vocab >= BM &&
                        reinterpret_cast<uintptr_t>(t.data) % 16 == 0)
                           ? gemv_q8_stages(t.hidden, bc1, dev.max_smem_optin)
                           : 0;
    // f32 tables with short 16-byte-multiple rows: bulk-stream GEMV
    const bool bulk = !tc && t.dtype == LHS_F32 && t.hidden % 8 == 0 &&
                      t.row_bytes % 16 == 0 && t.row_bytes <= kBulkRowBytesMax &&
                      bulk_smem_bytes(t.row_bytes, kBatchChunk, t.hidden) <= static_cast<size_t>(dev.max_smem_optin);
    p.path = gemm ? 2 : (tc ? 0 : (q8_nst ? 4 : (bulk ? 3 : 1)));
    if (gemm) {
        p.grid = clusters;  // partial lists: one per cluster
        // a cluster covers 2 x 128 residuals (one TMEM lane each): larger
        // batches run as successive passes of that many
        p.batch_chunk = batch < gemm_lm_head_max_batch() ? batch : gemm_lm_head_max_batch();
    } else {
        // with top-k, one SM stays free for the merge kernel: it cannot share
        // an SM with a GEMV CTA (shared memory), so it runs there while the
        // next call's CTAs already stream on the others
        const int ctas = (k > 0 && dev.num_sms > 1) ? dev.num_sms - 1 : dev.num_sms;
        p.grid = static_cast<int>(units < ctas ? units : ctas);
    }
    if (gemm) {
        // nothing else to size: the GEMM reads the residuals in place
    } else if (p.path == 3) {
        p.batch_chunk = kBatchChunk;
    } else if (p.path == 4) {
        p.batch_chunk = kBatchChunk;
        p.nst = q8_nst;
    } else if (tc) {
        p.batch_chunk = kBatchChunk;
        // the deepest ring that fits: the resident operand (compact for up
        // to 3 residuals) if it fits beside 10 stages or more, else the
        // operand streamed beside the table
        const int bc = batch < 1 ? 1 : (batch < kBatchChunk ? batch : kBatchChunk);
        const size_t lim = static_cast<size_t>(dev.max_smem_optin);
        p.xres = true;
        p.nst = xres_rows(bc) < 16 ? kStagesCompact : kStagesResident;
        if (tc_smem_bytes(true, p.kpad, p.nst, bc) > lim) p.nst = kStagesResident;
        if (tc_smem_bytes(true, p.kpad, p.nst, bc) > lim) {
            p.xres = false;
            p.nst = kStagesRing;
        }
        if (tc_smem_bytes(p.xres, p.kpad, p.nst, bc) > lim) return LHS_ERR_UNSUPPORTED;
    } else {
        int bc = static_cast<int>(kSimtXBytesMax / (static_cast<size_t>(t.hidden) * 4));
        if (bc > kBatchChunk) bc = kBatchChunk;
        if (bc < 1) bc = 1;
        p.batch_chunk = bc;
        if (simt_smem_bytes(bc, t.hidden) > static_cast<size_t>(dev.max_smem_optin))
            return LHS_ERR_UNSUPPORTED;
    }
    const int kk = k > 0 ? k : 1;
    if (k > 0 && merge_smem_bytes(p.grid, k > 32 ? k : 32) > static_cast<size_t>(dev.max_smem_optin))
        return LHS_ERR_UNSUPPORTED;
    size_t off = 0;
    p.off_x = off;
    off += (tc && !gemm) ? align_up(static_cast<size_t>(16) * p.kpad * 2, 1024) : 0;
    p.key_stride = gemm ? gemm_lm_head_cap(kk) : kk;
    const int wb = gemm ? p.batch_chunk : batch;  // residuals whose lists the workspace holds at once
    p.off_keys = off;
    off += align_up(static_cast<size_t>(p.grid) * wb * p.key_stride * 8, 256);
    p.off_ms = off;
    off += align_up(static_cast<size_t>(p.grid) * wb * 8, 256);
    // GEMM sample: the first tile of each cluster, worth it when each
    // cluster owns at least two tiles
    p.sample = gemm && k > 0 && (t.vocab + 255) / 256 >= 2 * static_cast<int64_t>(p.grid);
    p.off_sample = p.off_bound = p.off_sync = off;
    if (p.sample) {
        p.off_sample = off;
        off += align_up(static_cast<size_t>(wb) * p.grid * gemm_lm_head_sample_groups() * 4, 256);
        p.off_bound = off;
        off += align_up(static_cast<size_t>(wb) * 4, 256);
        p.off_sync = off;
        off += 256;
    }
    p.bytes = off;
    *plan = p;
    return LHS_OK;
}

int lm_head_launches(const LmHeadPlan &plan, int32_t batch, bool raw) {
    const int chunks = (batch + plan.batch_chunk - 1) / plan.batch_chunk;
    if (plan.path == 2) return chunks * (raw ? 1 : (plan.sample ? 3 : 2));  // (counter reset +) GEMM + merge
    const int per_chunk = (plan.path == 0 && !plan.xres) ? 2 : 1;  // (prep +) projection
    return chunks * per_chunk + (raw ? 0 : 1);
}

cudaError_t launch_lm_head(const lhs_table &t, const LmHeadPlan &plan, const void *resid,
                           int32_t resid_dtype, int32_t batch, int32_t k, float temperature,
                           int32_t *ids, float *logits_out, float *probs, float *raw_logits,
                           void *ws, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    const bool raw = raw_logits != nullptr;
    const float invT = 1.0f / temperature;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    uint64_t *part_keys = reinterpret_cast<uint64_t *>(wsb + plan.off_keys);
    float2 *part_ms = reinterpret_cast<float2 *>(wsb + plan.off_ms);
    const size_t relt = resid_dtype == LHS_F32 ? 4 : 2;

    if (plan.path == 2) {
        GemmBuffers gb;
        gb.sample = plan.sample ? reinterpret_cast<uint32_t *>(wsb + plan.off_sample) : nullptr;
        gb.bound = reinterpret_cast<uint32_t *>(wsb + plan.off_bound);
        gb.sync = reinterpret_cast<uint32_t *>(wsb + plan.off_sync);
        gb.cand = part_keys;
        gb.ms = part_ms;
        gb.cap = plan.key_stride;
        for (int c0 = 0; c0 < batch; c0 += plan.batch_chunk) {
            const int Bc = batch - c0 < plan.batch_chunk ? batch - c0 : plan.batch_chunk;
            const void *rc = static_cast<const uint8_t *>(resid) + static_cast<size_t>(c0) * t.hidden * relt;
            float *rawc = raw ? raw_logits + static_cast<size_t>(c0) * t.vocab : nullptr;
            e = launch_gemm_lm_head(t, rc, Bc, k, invT, rawc, gb, err, plan.grid, dev, stream);
            if (e != cudaSuccess) return e;
            if (!raw) {
                const size_t o = static_cast<size_t>(c0) * k;
                e = launch_merge(part_keys, part_ms, plan.grid, plan.key_stride, k, Bc, k, invT, ids + o,
                                 logits_out + o, probs ? probs + o : nullptr, dev, stream);
                if (e != cudaSuccess) return e;
            }
        }
        return cudaSuccess;
    } else if (plan.path == 0) {
        const bool bf16 = t.dtype == LHS_BF16;
        uint16_t *xs = reinterpret_cast<uint16_t *>(wsb + plan.off_x);
        CUtensorMap tm_a, tm_a16, tm_x;
        if (!make_tma_map_16bit(&tm_a, t.data, t.hidden, t.vocab, t.row_bytes, BK, BM, bf16) ||
            !make_tma_map_16bit(&tm_a16, t.data, t.hidden, t.vocab, t.row_bytes, BK, kBoxRowsSmall, bf16) ||
            !make_tma_map_16bit(&tm_x, xs, plan.kpad, 16, static_cast<uint64_t>(plan.kpad) * 2, BK, 16, bf16))
            return cudaErrorInvalidValue;
        using TcKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const TcParams);
        // variants: operand streamed (kStagesRing), resident (kStagesResident
        // or, compact, kStagesCompact)
#define LHS_TC(BF, R)                                                                              \
    {gemv_tc_kernel<BF, R, false, kStagesRing>, gemv_tc_kernel<BF, R, true, kStagesResident>, \
     gemv_tc_kernel<BF, R, true, kStagesCompact>}
        static const TcKernel kTable[2][2][3] = {{LHS_TC(false, false), LHS_TC(false, true)},
                                                 {LHS_TC(true, false), LHS_TC(true, true)}};
#undef LHS_TC
        const int variant = !plan.xres ? 0 : (plan.nst == kStagesCompact ? 2 : 1);
        const TcKernel kern = kTable[bf16][raw][variant];
        const size_t smem = tc_smem_bytes(plan.xres, plan.kpad, plan.nst,
                                          batch < plan.batch_chunk ? batch : plan.batch_chunk);
        {
            // one attribute flag per instantiation: the largest size this device allows
            static std::mutex mu;
            static bool done[12][64] = {};
            const int which = (bf16 ? 6 : 0) + (raw ? 3 : 0) + variant;
            std::lock_guard<std::mutex> lock(mu);
            if (!done[which][dev.device]) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin);
                if (e != cudaSuccess) return e;
                done[which][dev.device] = true;
            }
        }
        for (int c0 = 0; c0 < batch; c0 += plan.batch_chunk) {
            const int Bc = batch - c0 < plan.batch_chunk ? batch - c0 : plan.batch_chunk;
            const void *rc = static_cast<const uint8_t *>(resid) + static_cast<size_t>(c0) * t.hidden * relt;
            if (!plan.xres) {
                const int pgrid = static_cast<int>((static_cast<int64_t>(8) * plan.kpad + 255) / 256);
                auto prep = bf16 ? (resid_dtype == LHS_F32 ? prep_kernel<true, LHS_F32> : prep_kernel<true, LHS_BF16>)
                                 : (resid_dtype == LHS_F32 ? prep_kernel<false, LHS_F32> : prep_kernel<false, LHS_BF16>);
                e = launch_pdl(prep, dim3(pgrid), dim3(256), 0, stream, rc, Bc, static_cast<int>(t.hidden),
                               plan.kpad, xs, err);
                if (e != cudaSuccess) return e;
            }
            TcParams p;
            p.V = t.vocab;
            p.K = t.hidden;
            p.nk = plan.kpad / BK;
            p.Bc = Bc;
            p.b_off = c0;
            p.batch_total = batch;
            p.k = k;
            p.invT = invT;
            p.raw = raw_logits;
            p.part_keys = part_keys;
            p.part_ms = part_ms;
            p.resid = rc;
            p.resid_f32 = resid_dtype == LHS_F32;
            p.err = err;
            e = launch_pdl(kern, dim3(plan.grid), dim3(kTcThreads), smem, stream, tm_a, tm_a16, tm_x, p);
            if (e != cudaSuccess) return e;
        }
    } else if (plan.path == 4) {
        e = launch_gemv_q8(t, plan.nst, resid, resid_dtype, batch, k, invT, raw_logits, part_keys, part_ms, err,
                           plan.grid, dev, stream);
        if (e != cudaSuccess) return e;
    } else if (plan.path == 3) {
        using BulkKernel = void (*)(const BulkParams);
        static const BulkKernel kTable[2][4] = {
            {gemv_bulk_kernel<LHS_F32, false, 1>, gemv_bulk_kernel<LHS_F32, false, 2>,
             gemv_bulk_kernel<LHS_F32, false, 4>, gemv_bulk_kernel<LHS_F32, false, 8>},
            {gemv_bulk_kernel<LHS_F32, true, 1>, gemv_bulk_kernel<LHS_F32, true, 2>,
             gemv_bulk_kernel<LHS_F32, true, 4>, gemv_bulk_kernel<LHS_F32, true, 8>}};
        {
            static std::mutex mu;
            static bool done[8][64] = {};
            std::lock_guard<std::mutex> lock(mu);
            for (int r = 0; r < 2; ++r)
                for (int c = 0; c < 4; ++c) {
                    const int which = r * 4 + c;
                    if (!done[which][dev.device]) {
                        e = cudaFuncSetAttribute(kTable[r][c], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 dev.max_smem_optin);
                        if (e != cudaSuccess) return e;
                        done[which][dev.device] = true;
                    }
                }
        }
        for (int c0 = 0; c0 < batch; c0 += plan.batch_chunk) {
            const int Bc = batch - c0 < plan.batch_chunk ? batch - c0 : plan.batch_chunk;
            const BulkKernel kern = kTable[raw][Bc <= 1 ? 0 : (Bc <= 2 ? 1 : (Bc <= 4 ? 2 : 3))];
            BulkParams p;
            p.table = static_cast<const uint8_t *>(t.data);
            p.V = t.vocab;
            p.K = t.hidden;
            p.row_bytes = t.row_bytes;
            p.resid = static_cast<const uint8_t *>(resid) + static_cast<size_t>(c0) * t.hidden * relt;
            p.resid_dtype = resid_dtype;
            p.Bc = Bc;
            p.b_off = c0;
            p.batch_total = batch;
            p.k = k;
            p.invT = invT;
            p.raw = raw_logits;
            p.part_keys = part_keys;
            p.part_ms = part_ms;
            p.err = err;
            e = launch_pdl(kern, dim3(plan.grid), dim3(kBulkThreads), bulk_smem_bytes(t.row_bytes, Bc, t.hidden),
                           stream, p);
            if (e != cudaSuccess) return e;
        }
    } else {
        const size_t smem = simt_smem_bytes(plan.batch_chunk, t.hidden);
        // 8-element steps: K % 8 == 0, rows 16-byte aligned (Q8_0: 2-byte, always)
        bool vec = t.hidden % 8 == 0;
        if (t.dtype != LHS_Q8_0)
            vec = vec && reinterpret_cast<uintptr_t>(t.data) % 16 == 0 && t.row_bytes % 16 == 0;
        void (*kern)(const SimtParams);
#define LHS_SIMT(DT) (raw ? (vec ? gemv_simt_kernel<DT, true, true> : gemv_simt_kernel<DT, true, false>) \
                          : (vec ? gemv_simt_kernel<DT, false, true> : gemv_simt_kernel<DT, false, false>))
        switch (t.dtype) {
        case LHS_F32: kern = LHS_SIMT(LHS_F32); break;
        case LHS_F16: kern = LHS_SIMT(LHS_F16); break;
        case LHS_BF16: kern = LHS_SIMT(LHS_BF16); break;
        default: kern = LHS_SIMT(LHS_Q8_0); break;
        }
#undef LHS_SIMT
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        for (int c0 = 0; c0 < batch; c0 += plan.batch_chunk) {
            const int Bc = batch - c0 < plan.batch_chunk ? batch - c0 : plan.batch_chunk;
            SimtParams p;
            p.table = static_cast<const uint8_t *>(t.data);
            p.V = t.vocab;
            p.K = t.hidden;
            p.row_bytes = t.row_bytes;
            p.resid = static_cast<const uint8_t *>(resid) + static_cast<size_t>(c0) * t.hidden * relt;
            p.resid_dtype = resid_dtype;
            p.Bc = Bc;
            p.b_off = c0;
            p.batch_total = batch;
            p.k = k;
            p.invT = invT;
            p.raw = raw_logits;
            p.part_keys = part_keys;
            p.part_ms = part_ms;
            p.err = err;
            e = launch_pdl(kern, dim3(plan.grid), dim3(kSimtThreads), smem, stream, p);
            if (e != cudaSuccess) return e;
        }
    }
    if (raw) return cudaSuccess;
    if (plan.path != 2 && plan.grid <= kMergeThreads) {
        const int R = merge_stage_entries(plan.grid, k);
        return launch_pdl(merge_sorted_kernel, dim3(batch), dim3(kMergeThreads),
                          static_cast<size_t>(plan.grid) * (R + 1) * 8, stream,
                          static_cast<const uint64_t *>(part_keys), static_cast<const float2 *>(part_ms),
                          plan.grid, static_cast<int>(batch), static_cast<int>(k), R, invT, ids, logits_out,
                          probs);
    }
    return launch_merge(part_keys, part_ms, plan.grid, plan.key_stride, k, batch, k, invT, ids,
                        logits_out, probs, dev, stream);
}

cudaError_t launch_merge(const uint64_t *part_keys, const float2 *part_ms, int G, int stride,
                         int len, int batch, int k, float invT, int32_t *ids, float *logits,
                         float *probs, const DeviceInfo &dev, cudaStream_t stream) {
    const size_t msmem = merge_smem_bytes(G, len);
    {
        static std::mutex mu;
        static bool done[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev.device]) {
            const cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       dev.max_smem_optin);
            if (e != cudaSuccess) return e;
            done[dev.device] = true;
        }
    }
    return launch_pdl(merge_kernel, dim3(batch), dim3(256), msmem, stream, part_keys, part_ms, G,
                      stride, len, batch, k, invT, ids, logits, probs);
}

// ---------------------------------------------------------------------------
// bounded-wait self test
// ---------------------------------------------------------------------------
namespace {
__global__ void selftest_wait_kernel(int32_t *err, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing ever arrives on `bar`: phase 0 never completes
        if (!mbar_wait(&bar, 0, timeout_ns)) set_err(err, LHS_ERRBIT_TIMEOUT);
    }
}
}  // namespace

cudaError_t launch_selftest_wait(int32_t *err, int64_t timeout_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, static_cast<uint64_t>(timeout_ns));
    return cudaGetLastError();
}

}  // namespace lhs
