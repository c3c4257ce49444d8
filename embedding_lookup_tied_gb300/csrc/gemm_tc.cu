// gemm_tc.cu — batched tied lm_head on the 5th-generation tensor cores
// (tcgen05 + TMEM), with the top-k and the online softmax fused into the
// epilogue.
//
// ADR-0008 "Remote Embeddings and lm_head Service", POST /v1/logits
// (residual @ lm_head.T, top_k {token_id, prob}) for a batch of residuals:
// with hundreds of residuals the projection is a dense contraction
// (2*batch FLOP per table element), so it runs as a GEMM.
//
// Orientation: D[m][n] = sum_k X[m][k] * T[n][k].  The residuals are M (one
// TMEM lane each, 128 per CTA), the vocab rows are N (256 per tile), both
// operands K-major bf16 staged by TMA with 128-byte swizzle, the f32
// accumulator lives in TMEM (2 x 256 columns, double-buffered so the MMAs
// of the next tile overlap the epilogue of this one).  An epilogue thread
// therefore owns one residual: it keeps its own running (max, sum exp) and
// its own sorted top-k list in shared memory, with no cross-thread
// reduction.
//
// CTAs run in clusters of two, one per half of the residuals.  Both need the
// same 256-row table tile per stage: each CTA loads 128 rows and multicasts
// them to both, so HBM reads every table row once per call.
//
// Roles (192 threads): warp 0 — TMA producer; warp 1 — TMEM allocation and
// the single MMA-issuing thread; warps 2..5 — epilogue (TMEM lane quarter =
// warp % 4).  Every mbarrier wait is bounded; on expiry the kernel records
// LHS_ERRBIT_TIMEOUT, every role skips its remaining waits, and the CTA
// still frees its TMEM and meets its peer at the final cluster barrier.
#include <cuda_bf16.h>

#include <mutex>

#include "lhs_internal.cuh"

namespace lhs {
namespace {

constexpr int GM = 128;                      // residuals per CTA (TMEM lanes)
constexpr int GN = 256;                      // vocab rows per tile
constexpr int GK = 64;                       // k per stage: 128 bytes of bf16
constexpr int kGemmThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kAccCols = 256;                // f32 columns per accumulator buffer
constexpr int kTmemCols = 512;               // two buffers
constexpr int kAStageBytes = GM * GK * 2;    // 16 KB: this CTA's residuals
constexpr int kBStageBytes = GN * GK * 2;    // 32 KB: the whole table tile
constexpr int kBHalfBytes = kBStageBytes / 2;

struct GemmParams {
    int64_t V;
    int K;
    int B;            // residuals in the call
    int k;            // top-k (0 = raw mode)
    float invT;
    int tiles;        // ceil(V / GN)
    int clusters;     // clusters in the grid
    float *raw;       // raw mode: [B x V]
    uint64_t *part_keys;
    float2 *part_ms;
    int32_t *err;
};

template <int S>
struct GemmSmem {
    uint8_t a[S][kAStageBytes];
    uint8_t b[S][kBStageBytes];
    uint64_t full[S];
    uint64_t empty[S];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int abort_flag;
    // followed by the top-k lists: list[i * GM + row], i < k
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// TMA load of a box into the same shared-memory offset of every CTA in
// `mask`, completing transaction bytes on the barrier at that offset in each.
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *map, uint64_t *bar,
                                               int32_t c0, int32_t c1, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "h"(mask)
        : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the layout TMA writes for a box 64 bf16 wide).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor, kind::f16: bf16 x bf16 -> f32, both K-major.
constexpr uint32_t kIdesc = (1u << 4)                        // D = f32
                            | (1u << 7) | (1u << 10)         // A, B = bf16
                            | (static_cast<uint32_t>(GN >> 3) << 17)   // N
                            | (static_cast<uint32_t>(GM >> 4) << 24);  // M
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void umma_commit_mc(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ int ld_vol(const int *p) { return *reinterpret_cast<const volatile int *>(p); }

// The bits of `mask` whose (logit, vocab row) key beats `tau` exactly.
// Static indices only, so vals[] stays in registers.
__device__ __forceinline__ uint32_t exact_mask(const float (&vals)[32], uint32_t mask, int64_t vc,
                                               uint64_t tau) {
    uint32_t exact = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if ((mask >> j) & 1u)
            if (topk_key(vals[j], static_cast<int32_t>(vc + j)) > tau) exact |= 1u << j;
    return exact;
}

// 2^x with the hardware approximation (relative error ~2^-22), enough for
// the softmax normaliser (probabilities are checked to 1e-5).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bounded wait that gives up at once when the CTA has already aborted
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, int *abort_flag,
                                              int32_t *err) {
    if (ld_vol(abort_flag)) return false;
    if (mbar_wait(bar, parity, kWaitTimeoutNs)) return true;
    set_err(err, LHS_ERRBIT_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
    return false;
}

// Candidate buffers of the top-k epilogue.  Residual `row` of the CTA owns
// entries [0, cnt) of keys32[i * GM + row] (order key of the logit) and
// offs[i * GM + row] (vocab row - first row of the cluster's range), 6 bytes
// per entry.  Each epilogue thread appends its own residual's candidates;
// when a buffer could overflow, the warp cuts it back to the k best with a
// bitonic sort in registers (E entries per lane).
template <int S>
struct TopkCap {
    // entries per residual that fit beside S stages in 227 KB
    static constexpr int value = S >= 4 ? 44 : (S == 3 ? 108 : 172);
    static constexpr int sortn = value <= 64 ? 64 : (value <= 128 ? 128 : 256);
};

constexpr size_t kSmemOptin = 232448;  // 227 KB per CTA on sm_103a
static_assert(1024 + sizeof(GemmSmem<4>) + 16 + TopkCap<4>::value * GM * 6 <= kSmemOptin, "S=4");
static_assert(1024 + sizeof(GemmSmem<3>) + 16 + TopkCap<3>::value * GM * 6 <= kSmemOptin, "S=3");
static_assert(1024 + sizeof(GemmSmem<2>) + 16 + TopkCap<2>::value * GM * 6 <= kSmemOptin, "S=2");
static_assert(kMaxK + 32 <= TopkCap<2>::value, "largest k fits the two-stage buffers");

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), m);
    const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), src);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// One compare-exchange stage of a descending bitonic sort of N keys held E
// per lane (index i = lane * E + e), then the next stage: the network is
// unrolled at compile time so v[] stays in registers.
template <int N, int LS, int LD>
struct BitonicStage {
    static __device__ __forceinline__ void run(uint64_t (&v)[N / 32], int lane) {
        constexpr int E = N / 32;
        constexpr int size = 1 << LS, d = 1 << LD;
        constexpr int LOGN = N == 64 ? 6 : (N == 128 ? 7 : 8);
        if constexpr (d >= E) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int i = lane * E + e;
                const uint64_t other = shfl_xor_u64(v[e], d / E);
                const bool take_max = ((i & d) == 0) == ((i & size) == 0);
                v[e] = take_max ? (v[e] > other ? v[e] : other) : (v[e] < other ? v[e] : other);
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if (e & d) continue;
                const bool desc = ((lane * E + e) & size) == 0;
                const uint64_t a = v[e], b = v[e | d];
                const bool sw = desc ? (a < b) : (a > b);
                v[e] = sw ? b : a;
                v[e | d] = sw ? a : b;
            }
        }
        if constexpr (LD > 0) BitonicStage<N, LS, LD - 1>::run(v, lane);
        else if constexpr (LS < LOGN) BitonicStage<N, LS + 1, LS>::run(v, lane);
    }
};

// Warp-collective: sort the n entries of residual `row` (full 64-bit keys,
// id = id_base + off) descending and keep the first kk in the buffer.
// Returns the kk-th key (0 when n < kk) in every lane.
template <int N>
__device__ __forceinline__ uint64_t warp_cut(uint32_t *keys32, uint16_t *offs, int row, int n, int kk,
                             uint32_t id_base, int lane) {
    constexpr int E = N / 32;
    uint64_t v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = lane * E + e;
        v[e] = i < n ? (static_cast<uint64_t>(keys32[i * GM + row]) << 32) |
                           (0xFFFFFFFFu - (id_base + offs[i * GM + row]))
                     : 0ull;
    }
    BitonicStage<N, 1, 0>::run(v, lane);  // descending
    __syncwarp();  // every lane has read the buffer before it is rewritten
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = lane * E + e;
        if (i < kk && i < n) {
            keys32[i * GM + row] = static_cast<uint32_t>(v[e] >> 32);
            offs[i * GM + row] =
                static_cast<uint16_t>((0xFFFFFFFFu - static_cast<uint32_t>(v[e])) - id_base);
        }
    }
    __syncwarp();
    if (n < kk) return 0ull;
    const int idx = kk - 1;
    // fetch element idx from its lane without indexing v[] at run time
    uint64_t sel = 0ull;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const uint64_t t = shfl_u64(v[e], idx / E);
        if (e == idx % E) sel = t;
    }
    return sel;
}

template <int S, bool RAW>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_t,
                   const GemmParams p) {
    extern __shared__ uint8_t dyn_smem[];
    GemmSmem<S> &sm = *reinterpret_cast<GemmSmem<S> *>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int CAP = TopkCap<S>::value;
    uint32_t *keys32 = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(&sm) +
                                                    ((sizeof(GemmSmem<S>) + 15) & ~size_t(15)));
    uint16_t *offs = reinterpret_cast<uint16_t *>(keys32 + CAP * GM);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();          // residual half
    const int cl = blockIdx.x >> 1;                   // cluster index
    const int t0 = static_cast<int>((static_cast<int64_t>(p.tiles) * cl) / p.clusters);
    const int t1 = static_cast<int>((static_cast<int64_t>(p.tiles) * (cl + 1)) / p.clusters);
    const int nk = (p.K + GK - 1) / GK;
    const uint32_t total = static_cast<uint32_t>(t1 - t0) * nk;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 2);       // one MMA commit from each CTA of the pair
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tmem_full[i], 1);
            mbar_init(&sm.tmem_empty[i], kEpiThreads / 32);
        }
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();  // the peer's barriers exist before anything is multicast to them
    pdl_trigger();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            tma_prefetch_map(&tm_x);
            tma_prefetch_map(&tm_t);
            const uint16_t both = 0x3;
            auto issue_t = [&](uint32_t j) {
                const int s = j % S;
                const int tile = t0 + static_cast<int>(j / nk), kc = static_cast<int>(j % nk);
                tma_load_2d_mc(sm.b[s] + rank * kBHalfBytes, &tm_t, &sm.full[s], kc * GK,
                               tile * GN + static_cast<int>(rank) * (GN / 2), both);
            };
            auto issue_x = [&](uint32_t j) {
                const int s = j % S;
                tma_load_2d(sm.a[s], &tm_x, &sm.full[s], static_cast<int>(j % nk) * GK,
                            static_cast<int>(rank) * GM);
            };
            // table tiles first (never written by an earlier kernel), then
            // wait for the residuals' producer
            const uint32_t pre = total < static_cast<uint32_t>(S) ? total : S;
            for (uint32_t j = 0; j < pre; ++j) {
                mbar_arrive_expect_tx(&sm.full[j], kAStageBytes + kBStageBytes);
                issue_t(j);
            }
            pdl_wait();
            for (uint32_t j = 0; j < pre; ++j) issue_x(j);
            uint32_t it = pre;
            for (; it < total; ++it) {
                const int s = it % S;
                if (!wait_or_abort(&sm.empty[s], ((it / S) & 1) ^ 1, &sm.abort_flag, p.err)) break;
                mbar_arrive_expect_tx(&sm.full[s], kAStageBytes + kBStageBytes);
                issue_t(it);
                issue_x(it);
            }
            // drain: both CTAs have consumed every issued stage, so no copy
            // or remote arrive is still headed for either CTA
            for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0); j < it; ++j)
                if (!wait_or_abort(&sm.empty[j % S], (j / S) & 1, &sm.abort_flag, p.err)) break;
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            uint32_t it = 0;
            const uint16_t both = 0x3;
            for (int tile = t0, ti = 0; tile < t1; ++tile, ++ti) {
                const int buf = ti & 1;
                if (!wait_or_abort(&sm.tmem_empty[buf], ((ti >> 1) & 1) ^ 1, &sm.abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * kAccCols;
                bool ok = true;
                for (int kc = 0; kc < nk; ++kc, ++it) {
                    const int s = it % S;
                    if (!wait_or_abort(&sm.full[s], (it / S) & 1, &sm.abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sm.a[s]), b0 = smem_u32(sm.b[s]);
#pragma unroll
                    for (int ks = 0; ks < GK / 16; ++ks)
                        umma_bf16(d, desc_sw128(a0 + ks * 32), desc_sw128(b0 + ks * 32),
                                  (kc | ks) != 0);
                    umma_commit_mc(&sm.empty[s], both);  // frees the stage in both CTAs
                }
                if (!ok) break;
                umma_commit(&sm.tmem_full[buf]);
            }
        }
    } else {
        // ---------------- epilogue ----------------
        pdl_wait();  // partial lists may still be read by the previous merge
        const int q = warp & 3;                       // TMEM lane quarter
        const int row = q * 32 + lane;                // this thread's residual in the CTA
        const int b = static_cast<int>(rank) * GM + row;
        const bool valid = b < p.B;
        float m_run = -INFINITY, s_run = 0.0f;
        int cnt = 0;          // entries in this residual's buffer
        uint64_t tau = 0ull;  // a key every kept entry beats (the k-th best after a cut)
        float tau_val = -INFINITY;  // the logit of tau
        const float l2e_invT = 1.4426950408889634f * p.invT;
        const uint32_t id_base = static_cast<uint32_t>(t0) * GN;
        for (int tile = t0, ti = 0; tile < t1; ++tile, ++ti) {
            const int buf = ti & 1;
            // the decision must be warp-uniform: tcgen05.ld is warp-collective
            const bool ok = wait_or_abort(&sm.tmem_full[buf], (ti >> 1) & 1, &sm.abort_flag, p.err);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const int64_t v0 = static_cast<int64_t>(tile) * GN;
            for (int c = 0; c < kAccCols / 32; ++c) {
                float vals[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kAccCols + c * 32, vals);
                const int64_t vc = v0 + c * 32;
                if (RAW) {
                    if (valid)
                        for (int j = 0; j < 32; ++j)
                            if (vc + j < p.V) p.raw[static_cast<int64_t>(b) * p.V + vc + j] = vals[j];
                    continue;
                }
                const int nvalid = valid ? static_cast<int>(p.V - vc < 32 ? (p.V - vc) : 32) : 0;
                const uint32_t vmask = nvalid >= 32 ? 0xFFFFFFFFu : ((1u << nvalid) - 1u);
                if (nvalid > 0) {
                    float cmax = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if ((vmask >> j) & 1u) cmax = fmaxf(cmax, vals[j]);
                    const float mn = fmaxf(m_run, cmax);
                    if (mn != -INFINITY) {
                        // exp((v - mn) / T) = 2^((v - mn) * log2(e) / T)
                        float acc = s_run * ex2_approx((m_run - mn) * l2e_invT);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if ((vmask >> j) & 1u) acc += ex2_approx((vals[j] - mn) * l2e_invT);
                        s_run = acc;
                        m_run = mn;
                    }
                }
                const uint32_t off0 = static_cast<uint32_t>(vc) - id_base;
                // candidates: logits not below the threshold's value (NaN
                // passes), then the exact (value, id) order for those only
                uint32_t mask = 0;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (!(vals[j] < tau_val)) mask |= 1u << j;
                mask &= vmask;
                if (mask) mask = exact_mask(vals, mask, vc, tau);
                // cut every buffer of the warp that this chunk could overflow
                unsigned need = __ballot_sync(0xFFFFFFFFu, cnt + __popc(mask) > CAP);
                while (need) {
                    const int L = __ffs(need) - 1;
                    need &= need - 1;
                    const int nL = __shfl_sync(0xFFFFFFFFu, cnt, L);
                    const uint64_t kth = warp_cut<TopkCap<S>::sortn>(keys32, offs, q * 32 + L, nL,
                                                                     p.k, id_base, lane);
                    if (lane == L) {
                        cnt = nL < p.k ? nL : p.k;
                        tau = kth;
                        tau_val = kth ? key_value(kth) : -INFINITY;
                        // keep only what still beats the new k-th best
                        if (mask) mask = exact_mask(vals, mask, vc, tau);
                    }
                }
                if (mask) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if ((mask >> j) & 1u) {
                            keys32[cnt * GM + row] = order_key32(vals[j]);
                            offs[cnt * GM + row] = static_cast<uint16_t>(off0 + j);
                            ++cnt;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tmem_empty[buf]);
        }
        if (!RAW && !ld_vol(&sm.abort_flag)) {
            // final cut of every buffer in the warp, then the partial list
            unsigned need = __ballot_sync(0xFFFFFFFFu, cnt > p.k);
            while (need) {
                const int L = __ffs(need) - 1;
                need &= need - 1;
                const int nL = __shfl_sync(0xFFFFFFFFu, cnt, L);
                warp_cut<TopkCap<S>::sortn>(keys32, offs, q * 32 + L, nL, p.k, id_base, lane);
                if (lane == L) cnt = nL < p.k ? nL : p.k;
            }
            if (valid) {
                uint64_t *dst = p.part_keys + (static_cast<size_t>(cl) * p.B + b) * p.k;
                for (int i = 0; i < p.k; ++i)
                    dst[i] = i < cnt ? (static_cast<uint64_t>(keys32[i * GM + row]) << 32) |
                                           (0xFFFFFFFFu - (id_base + offs[i * GM + row]))
                                     : 0ull;
                p.part_ms[static_cast<size_t>(cl) * p.B + b] = make_float2(m_run, s_run);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync_all();  // neither CTA leaves while its peer may still address it
}

template <int S>
size_t gemm_smem_bytes(bool raw) {
    return 1024 + ((sizeof(GemmSmem<S>) + 15) & ~size_t(15)) +
           (raw ? 0 : static_cast<size_t>(TopkCap<S>::value) * GM * 6);
}

template <int S, bool RAW>
cudaError_t launch_s(const lhs_table &t, const void *resid, int batch, int k, float invT, float *raw,
                     uint64_t *part_keys, float2 *part_ms, int32_t *err, int clusters,
                     const DeviceInfo &dev, cudaStream_t stream) {
    CUtensorMap tm_x, tm_t;
    if (!make_tma_map_16bit(&tm_x, resid, t.hidden, batch, static_cast<uint64_t>(t.hidden) * 2, GK, GM,
                            true) ||
        !make_tma_map_16bit(&tm_t, t.data, t.hidden, t.vocab, t.row_bytes, GK, GN / 2, true))
        return cudaErrorInvalidValue;
    const size_t smem = gemm_smem_bytes<S>(RAW);
    auto kern = gemm_tc_kernel<S, RAW>;
    {
        static std::mutex mu;
        static bool done[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev.device]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 dev.max_smem_optin);
            if (e != cudaSuccess) return e;
            done[dev.device] = true;
        }
    }
    GemmParams p;
    p.V = t.vocab;
    p.K = t.hidden;
    p.B = batch;
    p.k = k;
    p.invT = invT;
    p.tiles = static_cast<int>((t.vocab + GN - 1) / GN);
    p.clusters = clusters;
    p.raw = raw;
    p.part_keys = part_keys;
    p.part_ms = part_ms;
    p.err = err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_t, p);
}

}  // namespace

// Stage count: as many as leave each residual's buffer room for k entries
// plus one full 32-column chunk.
static int gemm_stages(int k) {
    if (k + 32 <= TopkCap<4>::value) return 4;
    if (k + 32 <= TopkCap<3>::value) return 3;
    return 2;
}

size_t gemm_lm_head_smem(int k) {
    switch (gemm_stages(k)) {
    case 4: return gemm_smem_bytes<4>(false);
    case 3: return gemm_smem_bytes<3>(false);
    default: return gemm_smem_bytes<2>(false);
    }
}

// Clusters of two that can be resident at once (one CTA per SM), so the
// grid is one wave.  Cached per device.
int gemm_lm_head_clusters(const DeviceInfo &dev, int k) {
    static std::mutex mu;
    static int cache[64][3] = {};
    const int kk = k < 1 ? 1 : k;
    const int si = gemm_stages(kk) == 4 ? 0 : (gemm_stages(kk) == 3 ? 1 : 2);
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev.device][si]) return cache[dev.device][si];
    int n = dev.num_sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * n);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = gemm_lm_head_smem(kk);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    const void *fn = si == 0 ? reinterpret_cast<const void *>(gemm_tc_kernel<4, false>)
                   : si == 1 ? reinterpret_cast<const void *>(gemm_tc_kernel<3, false>)
                             : reinterpret_cast<const void *>(gemm_tc_kernel<2, false>);
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin);
    if (cudaOccupancyMaxActiveClusters(&active, fn, &cfg) == cudaSuccess && active > 0 && active < n)
        n = active;
    (void)cudaGetLastError();
    if (n < 1) n = 1;
    cache[dev.device][si] = n;
    return n;
}

cudaError_t launch_gemm_lm_head(const lhs_table &t, const void *resid, int batch, int k, float invT,
                                float *raw, uint64_t *part_keys, float2 *part_ms, int32_t *err,
                                int clusters, const DeviceInfo &dev, cudaStream_t stream) {
    const bool is_raw = raw != nullptr;
    const int kk = is_raw ? 1 : k;
    switch (gemm_stages(kk)) {
    case 4:
        return is_raw ? launch_s<4, true>(t, resid, batch, kk, invT, raw, part_keys, part_ms, err, clusters, dev, stream)
                      : launch_s<4, false>(t, resid, batch, kk, invT, raw, part_keys, part_ms, err, clusters, dev, stream);
    case 3:
        return launch_s<3, false>(t, resid, batch, kk, invT, raw, part_keys, part_ms, err, clusters, dev, stream);
    default:
        return launch_s<2, false>(t, resid, batch, kk, invT, raw, part_keys, part_ms, err, clusters, dev, stream);
    }
}

}  // namespace lhs
