// gemm_tc.cu — batched tied lm_head on the 5th-generation tensor cores
// (tcgen05 + TMEM), with the top-k and the online softmax fused into the
// epilogue.
//
// ADR-0008 "Remote Embeddings and lm_head Service", POST /v1/logits
// (residual @ lm_head.T, top_k {token_id, prob}) for a batch of residuals:
// with hundreds of residuals the projection is a dense contraction
// (2*batch FLOP per table element), so it runs as a GEMM.
//
// Orientation: D[m][n] = sum_k X[m][k] * T[n][k].  The residuals are M, the
// vocab rows are N (256 per tile), both operands K-major bf16 staged by TMA
// with 128-byte swizzle, the f32 accumulator in TMEM (2 x 256 columns,
// double-buffered so the MMAs of the next tile overlap the epilogue of this
// one).  An epilogue thread owns one residual (one TMEM lane): its running
// (max, sum exp) and its top-k candidates need no reduction across threads.
//
// CTAs run in pairs (clusters of two) and the leader CTA issues one M = 256
// MMA (tcgen05 cta_group::2) for the pair: each CTA stages its own 128
// residuals and its own 128 of the tile's 256 table rows, and receives the
// 128 x 256 accumulator of its residuals in its TMEM.  HBM reads every table
// row once per call, and a stage costs each CTA 32 KB of shared memory, so
// the ring holds seven stages in flight.  Both CTAs' copies of a stage complete
// on the leader's barrier; the leader's commits free the stage, and hand an
// accumulator to the epilogue, in both CTAs.
//
// Top-k in one pass with a bound taken from a sample of the logits, so that
// almost nothing is kept:
//  * every cluster's first tile is the sample (clusters x 256 vocab rows,
//    spread evenly over the vocabulary).  Each epilogue thread folds its
//    residual's 256 logits of that tile into 16 column-group maxima and
//    publishes them; the tile's accumulator stays in TMEM while the tensor
//    cores go on with the second tile in the other buffer.
//  * once every CTA has published (an arrival counter in global memory),
//    one warp per residual finds the k-th largest of that residual's
//    clusters x 16 group maxima.  It is a lower bound of the final k-th
//    logit (the k-th largest of any subset of the logits never exceeds the
//    k-th largest of all of them), and close to it, since the sample's best
//    logits rarely share a group.  A second counter tells every thread that
//    all bounds are written.
//  * every logit below its residual's bound is then dropped at once, the
//    first tile's included (read again from TMEM); the few others go to a
//    per-(cluster, residual) candidate buffer in global memory, cut back to
//    k by a warp-cooperative bitonic sort if it would overflow.  A merge
//    kernel selects the final top-k from the buffers.
// The exchange needs every CTA of the grid resident at once, which the
// launch sizes for (one wave of clusters); its waits are bounded, and a wait
// that runs out only drops the bound (every logit is then a candidate), so
// the result stays exact.  A CTA lets the next kernel launch only after it
// has published, so a dependent kernel never takes the SM of a CTA that the
// exchange still waits for.  The two counters are zeroed by a one-thread
// kernel launched just before, so the workspace may hold anything on entry.
// Vocabularies under two tiles per cluster skip the sample: no bound.
//
// Roles (192 threads): warp 0 — TMA producer; warp 1 — TMEM allocation
// (with the peer's warp 1) and, in the leader, the single MMA-issuing
// thread; warps 2..5 — epilogue (TMEM lane quarter = warp % 4).  Every
// mbarrier wait is bounded; on expiry the kernel records LHS_ERRBIT_TIMEOUT,
// every role skips its remaining waits, and the CTA still frees its TMEM and
// meets its peer at the final cluster barrier.
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
constexpr int kBHalfBytes = GN / 2 * GK * 2; // 16 KB: this CTA's half of the table tile
constexpr int kStagesG = 7;                  // ring stages (a residual box and a table box each)
constexpr int kPairStageBytes = 2 * (kAStageBytes + kBHalfBytes);  // one stage of both CTAs

enum { kModeRaw = 0, kModeMain = 1, kModeFused = 2 };
constexpr int kSampleGroups = 16;            // group maxima per (residual, cluster)
constexpr int kBoundPerLane = 48;            // sample entries per lane of a bound warp: all of them
                                             // up to 96 clusters, the first 1,536 beyond (a subset
                                             // still bounds the k-th logit from below)

struct GemmParams {
    int64_t V;
    int K;
    int B;                       // residuals in the call
    int k;                       // top-k
    float invT;
    int tiles;                   // ceil(V / GN)
    int clusters;                // clusters in the grid
    float *raw;                  // raw: [B x V]
    uint64_t *keys;              // main / fused: candidate buffers [clusters][B][cap]
    float2 *ms;                  // [clusters][B]
    int cap;                     // candidate buffer entries per (cluster, residual)
    uint32_t *sample;            // fused: [B][clusters][kSampleGroups] order keys of the first tile's
                                 // group maxima
    uint32_t *bound;             // fused: [B] order key of each residual's bound (0: none)
    uint32_t *sync;              // fused: arrival counters sync[0] (CTAs that published their
                                 // sample) and sync[32] (bound warps done), zeroed before the launch
    int32_t *err;
};

struct GemmSmem {
    uint8_t a[kStagesG][kAStageBytes];
    uint8_t b[kStagesG][kBHalfBytes];
    uint64_t full[kStagesG];
    uint64_t empty[kStagesG];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t kGemmSmemBytes = 1024 + sizeof(GemmSmem);

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// The shared::cluster address of the variable at `smem_addr` in CTA `cta`
// of this cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t smem_addr, uint32_t cta) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(cta));
    return r;
}
// TMA load of a box into this CTA's shared memory whose completion is
// counted on an mbarrier of either CTA of the pair (a shared::cluster
// address): both CTAs' copies of a stage complete on the leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}
// Arrive on an mbarrier of either CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the layout TMA writes for a box 64 bf16 wide).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor, kind::f16: bf16 x bf16 -> f32, both K-major;
// M = 256 over the CTA pair (128 TMEM lanes in each), N = 256.
constexpr uint32_t kIdesc = (1u << 4)                        // D = f32
                            | (1u << 7) | (1u << 10)         // A, B = bf16
                            | (static_cast<uint32_t>(GN >> 3) << 17)        // N
                            | (static_cast<uint32_t>((2 * GM) >> 4) << 24); // M
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit_mc(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
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

// bounded wait that gives up at once when the CTA has already aborted
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, int *abort_flag,
                                              int32_t *err) {
    if (ld_vol(abort_flag)) return false;
    if (mbar_wait(bar, parity, kWaitTimeoutNs)) return true;
    set_err(err, LHS_ERRBIT_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
    return false;
}

// 2^x with the hardware approximation (relative error ~2^-22), enough for
// the softmax normaliser (probabilities are checked to 1e-5).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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

// Warp-collective: sort the n keys of one candidate buffer (global memory)
// descending and keep the first kk.  Returns the kk-th key (0 when n < kk).
template <int N>
__device__ __forceinline__ uint64_t warp_cut(uint64_t *buf, int n, int kk, int lane) {
    constexpr int E = N / 32;
    uint64_t v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = lane * E + e;
        v[e] = i < n ? buf[i] : 0ull;
    }
    BitonicStage<N, 1, 0>::run(v, lane);
    __syncwarp();  // every lane has read the buffer before it is rewritten
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = lane * E + e;
        if (i < kk && i < n) buf[i] = v[e];
    }
    __syncwarp();
    if (n < kk) return 0ull;
    const int idx = kk - 1;
    uint64_t sel = 0ull;
#pragma unroll
    for (int e = 0; e < E; ++e) {  // element idx from its lane, no run-time index into v[]
        const uint64_t t = shfl_u64(v[e], idx / E);
        if (e == idx % E) sel = t;
    }
    return sel;
}

// Grid-wide arrival counters of the fused pass (global memory, gpu scope).
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Warp-collective: wait until *ctr >= target, for at most kWaitTimeoutNs.
// Lane 0 polls; every lane then takes its own acquire, so its later loads
// see what the arrivals published.  False when the limit ran out.
__device__ __forceinline__ bool wait_count(const uint32_t *ctr, uint32_t target, int lane) {
    int ok = 1;
    if (lane == 0 && ld_acquire_u32(ctr) < target) {
        const uint64_t t0 = global_ns();
        while (ld_acquire_u32(ctr) < target) {
            if (global_ns() - t0 > kWaitTimeoutNs) {
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (ok) (void)ld_acquire_u32(ctr);
    return ok != 0;
}
// Warp-collective: the k-th largest of the n order keys at src, counted with
// multiplicity (0 when fewer than k are nonzero).  Each lane holds up to
// kBoundPerLane of them; the result is built bit by bit from the top, a bit
// kept when at least k keys are >= the prefix with it set.
__device__ __forceinline__ uint32_t sample_kth(const uint32_t *src, int n, int k, int lane) {
    uint32_t v[kBoundPerLane];
#pragma unroll
    for (int e = 0; e < kBoundPerLane; ++e) {
        const int i = e * 32 + lane;
        v[e] = i < n ? __ldcg(src + i) : 0u;
    }
    uint32_t T = 0u;
#pragma unroll 1
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t c = T | (1u << bit);
        uint32_t cnt = 0u;
#pragma unroll
        for (int e = 0; e < kBoundPerLane; ++e) cnt += v[e] >= c ? 1u : 0u;
        cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (cnt >= static_cast<uint32_t>(k)) T = c;
    }
    return T;
}

// Zeroes the fused pass's two arrival counters, after every earlier kernel
// of the stream (the previous call's pass and merge) has completed.
__global__ void gemm_sync_reset_kernel(uint32_t *sync) {
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) {
        sync[0] = 0u;
        sync[32] = 0u;
    }
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_t,
                   const GemmParams p) {
    constexpr int S = kStagesG;
    extern __shared__ uint8_t dyn_smem[];
    GemmSmem &sm = *reinterpret_cast<GemmSmem *>(smem_align<1024>(dyn_smem));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();          // residual half
    const int cl = blockIdx.x >> 1;                   // cluster index
    const int t0 = static_cast<int>((static_cast<int64_t>(p.tiles) * cl) / p.clusters);
    const int t1 = static_cast<int>((static_cast<int64_t>(p.tiles) * (cl + 1)) / p.clusters);
    const int nk = (p.K + GK - 1) / GK;
    const uint32_t total = static_cast<uint32_t>(t1 - t0) * nk;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);        // leader: its producer's expect_tx; both CTAs' bytes
            mbar_init(&sm.empty[s], 1);       // the leader's MMA commit, multicast to both CTAs
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tmem_full[i], 1);
            mbar_init(&sm.tmem_empty[i], 2 * kEpiThreads / 32);  // leader: both CTAs' epilogue warps
        }
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {  // with the peer's warp 1: the pair's accumulator columns
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();  // the peer's barriers exist before anything is multicast to them
    if (MODE != kModeFused) pdl_trigger();  // fused: after this CTA has published its sample
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            tma_prefetch_map(&tm_x);
            tma_prefetch_map(&tm_t);
            // each CTA loads its residuals and its half of the table tile
            // into its own shared memory; both complete on the leader's
            // barrier, which the leader's producer arms for the pair
            auto issue = [&](uint32_t j, bool table, bool resid) {
                const int s = j % S;
                const int tile = t0 + static_cast<int>(j / nk), kc = static_cast<int>(j % nk);
                const uint32_t bar = cluster_addr(smem_u32(&sm.full[s]), 0);
                if (table) {
                    if (rank == 0) mbar_arrive_expect_tx(&sm.full[s], kPairStageBytes);
                    tma_load_2d_pair(sm.b[s], &tm_t, bar, kc * GK, tile * GN + static_cast<int>(rank) * (GN / 2));
                }
                if (resid) tma_load_2d_pair(sm.a[s], &tm_x, bar, kc * GK, static_cast<int>(rank) * GM);
            };
            // table boxes first (never written by an earlier kernel), then
            // wait for the residuals' producer
            const uint32_t pre = total < static_cast<uint32_t>(S) ? total : S;
            for (uint32_t j = 0; j < pre; ++j) issue(j, true, false);
            pdl_wait();
            for (uint32_t j = 0; j < pre; ++j) issue(j, false, true);
            uint32_t it = pre;
            for (; it < total; ++it) {
                if (!wait_or_abort(&sm.empty[it % S], ((it / S) & 1) ^ 1, &sm.abort_flag, p.err)) break;
                issue(it, true, true);
            }
            // drain: the pair has consumed every issued stage, so no copy,
            // completion or commit is still headed for either CTA
            for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0); j < it; ++j)
                if (!wait_or_abort(&sm.empty[j % S], (j / S) & 1, &sm.abort_flag, p.err)) break;
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (the leader CTA only) ----------------
        if (lane == 0 && rank == 0) {
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
                umma_commit_mc(&sm.tmem_full[buf], both);
            }
        }
    } else {
        // ---------------- epilogue ----------------
        pdl_wait();  // outputs may still be read, and the sample bound written, by earlier kernels
        const int q = warp & 3;                       // TMEM lane quarter
        const int row = q * 32 + lane;                // this thread's residual in the CTA
        const int b = static_cast<int>(rank) * GM + row;
        const bool valid = b < p.B;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;

        if (MODE == kModeRaw) {
            for (int tile = t0, ti = 0; tile < t1; ++tile, ++ti) {
                const int buf = ti & 1;
                const bool ok = wait_or_abort(&sm.tmem_full[buf], (ti >> 1) & 1, &sm.abort_flag, p.err);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;  // tcgen05.ld is warp-collective
                tc_fence_after();
                const int64_t v0 = static_cast<int64_t>(tile) * GN;
                for (int c = 0; c < kAccCols / 32; ++c) {
                    float vals[32];
                    tmem_ld32(tmem + lane_base + buf * kAccCols + c * 32, vals);
                    const int64_t vc = v0 + c * 32;
                    if (!valid) continue;
                    float *dst = p.raw + static_cast<int64_t>(b) * p.V + vc;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (vc + j < p.V) dst[j] = vals[j];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(&sm.tmem_empty[buf]), 0));
            }
        } else {
            // running softmax; candidates not below the bound into this
            // residual's buffer in global memory
            float m_run = -INFINITY, s_run = 0.0f;
            int cnt = 0;
            uint64_t tau = 0ull;       // exact key every kept entry beats (after a cut)
            float tau_val = -INFINITY; // the logit below which nothing can be kept
            const float l2e_invT = 1.4426950408889634f * p.invT;
            uint64_t *cand = p.keys + (static_cast<size_t>(cl) * p.B + (valid ? b : 0)) * p.cap;
            uint64_t *cand_lane0 =
                p.keys + (static_cast<size_t>(cl) * p.B + static_cast<int>(rank) * GM + q * 32) * p.cap;
            // one 32-column chunk of this residual's logits: running softmax,
            // then the candidates (warp-collective: every lane calls it)
            auto chunk = [&](const float (&vals)[32], int64_t vc) {
                const int nvalid = valid ? static_cast<int>(p.V - vc < 32 ? (p.V - vc) : 32) : 0;
                const uint32_t vmask = nvalid >= 32 ? 0xFFFFFFFFu
                                                    : (nvalid > 0 ? ((1u << nvalid) - 1u) : 0u);
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
                // candidates: not below the bound's value (NaN passes),
                // then the exact (value, id) order for those only
                uint32_t mask = 0;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (!(vals[j] < tau_val)) mask |= 1u << j;
                mask &= vmask;
                if (mask) mask = exact_mask(vals, mask, vc, tau);
                // cut every buffer of the warp this chunk could overflow
                unsigned need = __ballot_sync(0xFFFFFFFFu, cnt + __popc(mask) > p.cap);
                while (need) {
                    const int L = __ffs(need) - 1;
                    need &= need - 1;
                    const int nL = __shfl_sync(0xFFFFFFFFu, cnt, L);
                    uint64_t *bufL = cand_lane0 + static_cast<size_t>(L) * p.cap;
                    const uint64_t kth = p.cap <= 128 ? warp_cut<128>(bufL, nL, p.k, lane)
                                                      : warp_cut<256>(bufL, nL, p.k, lane);
                    if (lane == L) {
                        cnt = nL < p.k ? nL : p.k;
                        if (kth) {
                            tau = kth;
                            tau_val = fmaxf(tau_val, key_value(kth));
                        }
                        if (mask) mask = exact_mask(vals, mask, vc, tau);
                    }
                }
                if (mask) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if ((mask >> j) & 1u) cand[cnt++] = topk_key(vals[j], static_cast<int32_t>(vc + j));
                }
            };
            int ti_first = 0;  // first tile the loop below takes from TMEM
            if (MODE == kModeFused) {
                // (1) the first tile's 16 column-group maxima (groups
                // {j, j+16, j+32, ...}) as order keys: this thread's part of
                // the sample.  The accumulator stays in TMEM.
                const bool ok = t1 > t0 && wait_or_abort(&sm.tmem_full[0], 0, &sm.abort_flag, p.err);
                const bool ok_all = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.ld is warp-collective
                const int64_t v0 = static_cast<int64_t>(t0) * GN;
                uint32_t g[kSampleGroups];
#pragma unroll
                for (int j = 0; j < kSampleGroups; ++j) g[j] = 0u;
                if (ok_all) {
                    tc_fence_after();
                    for (int c = 0; c < kAccCols / 32; ++c) {
                        float vals[32];
                        tmem_ld32(tmem + lane_base + c * 32, vals);
                        const int64_t vc = v0 + c * 32;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (vc + j < p.V) g[j % kSampleGroups] = max(g[j % kSampleGroups], order_key32(vals[j]));
                    }
                }
                if (valid) {  // zeros (no entry) if the pipeline gave up
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        p.sample + (static_cast<size_t>(b) * p.clusters + cl) * kSampleGroups);
#pragma unroll
                    for (int j = 0; j < kSampleGroups / 4; ++j)
                        dst[j] = make_uint4(g[4 * j], g[4 * j + 1], g[4 * j + 2], g[4 * j + 3]);
                }
                __threadfence();
                named_bar_sync(1, kEpiThreads);  // the CTA's sample is written
                if (tid == 2 * 32) {
                    red_release_add(p.sync, 1u);
                    pdl_trigger();
                }
                // (2) one warp per residual: its bound, once every CTA has
                // published
                const int nw = static_cast<int>(gridDim.x) * (kEpiThreads / 32);
                const int gw = static_cast<int>(blockIdx.x) * (kEpiThreads / 32) + (warp - 2);
                if (gw < p.B) {
                    const bool all_in = wait_count(p.sync, gridDim.x, lane);
                    for (int rb = gw; rb < p.B; rb += nw) {
                        const uint32_t T =
                            all_in ? sample_kth(p.sample + static_cast<size_t>(rb) * p.clusters * kSampleGroups,
                                                p.clusters * kSampleGroups, p.k, lane)
                                   : 0u;
                        if (lane == 0) p.bound[rb] = T;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        red_release_add(p.sync + 32, 1u);
                    }
                }
                // (3) this residual's bound (none if the exchange ran out of time)
                const bool bounds_in = wait_count(p.sync + 32, static_cast<uint32_t>(p.B < nw ? p.B : nw), lane);
                if (bounds_in && valid) {
                    const uint32_t T = __ldcg(p.bound + b);
                    if (T) tau_val = key_value(static_cast<uint64_t>(T) << 32);
                }
                // (4) the first tile, filtered by the bound
                if (ok_all) {
                    for (int c = 0; c < kAccCols / 32; ++c) {
                        float vals[32];
                        tmem_ld32(tmem + lane_base + c * 32, vals);
                        chunk(vals, v0 + c * 32);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(&sm.tmem_empty[0]), 0));
                }
                ti_first = 1;
            }
            for (int tile = t0 + ti_first, ti = ti_first; tile < t1; ++tile, ++ti) {
                const int buf = ti & 1;
                const bool ok = wait_or_abort(&sm.tmem_full[buf], (ti >> 1) & 1, &sm.abort_flag, p.err);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;  // tcgen05.ld is warp-collective
                tc_fence_after();
                const int64_t v0 = static_cast<int64_t>(tile) * GN;
                for (int c = 0; c < kAccCols / 32; ++c) {
                    float vals[32];
                    tmem_ld32(tmem + lane_base + buf * kAccCols + c * 32, vals);
                    chunk(vals, v0 + c * 32);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(&sm.tmem_empty[buf]), 0));
            }
            if (!ld_vol(&sm.abort_flag)) {
                // cut buffers holding more than k, then pad to k
                unsigned need = __ballot_sync(0xFFFFFFFFu, cnt > p.k);
                while (need) {
                    const int L = __ffs(need) - 1;
                    need &= need - 1;
                    const int nL = __shfl_sync(0xFFFFFFFFu, cnt, L);
                    uint64_t *bufL = cand_lane0 + static_cast<size_t>(L) * p.cap;
                    if (p.cap <= 128) warp_cut<128>(bufL, nL, p.k, lane);
                    else warp_cut<256>(bufL, nL, p.k, lane);
                    if (lane == L) cnt = p.k;
                }
                if (valid) {
                    for (int i = cnt; i < p.k; ++i) cand[i] = 0ull;
                    p.ms[static_cast<size_t>(cl) * p.B + b] = make_float2(m_run, s_run);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the pair is done with its accumulators and barriers
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync_all();  // neither CTA leaves while its peer may still address it
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap &tm_x, const CUtensorMap &tm_t, const GemmParams &p,
                        const DeviceInfo &dev, cudaStream_t stream) {
    auto kern = gemm_tc_kernel<MODE>;
    {
        static std::mutex mu;
        static bool done[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev.device]) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(kGemmSmemBytes));
            if (e != cudaSuccess) return e;
            done[dev.device] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * p.clusters);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kGemmSmemBytes;
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

size_t gemm_lm_head_smem() { return kGemmSmemBytes; }

// Residuals one launch covers: a cluster's two CTAs hold 128 each.
int gemm_lm_head_max_batch() { return 2 * GM; }

// Candidate buffer entries per (cluster, residual) in the main pass: room
// for k plus at least one full chunk of 32 after a cut.
int gemm_lm_head_cap(int k) { return k + 32 <= 128 ? 128 : 256; }

// Clusters of two that can be resident at once (one CTA per SM), so the
// grid is one wave.  Cached per device.
int gemm_lm_head_clusters(const DeviceInfo &dev) {
    static std::mutex mu;
    static int cache[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev.device]) return cache[dev.device];
    int n = dev.num_sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * n);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kGemmSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    const void *fn = reinterpret_cast<const void *>(gemm_tc_kernel<kModeMain>);
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kGemmSmemBytes));
    if (cudaOccupancyMaxActiveClusters(&active, fn, &cfg) == cudaSuccess && active > 0 && active < n)
        n = active;
    (void)cudaGetLastError();
    if (n < 1) n = 1;
    cache[dev.device] = n;
    return n;
}

int gemm_lm_head_sample_groups() { return kSampleGroups; }

cudaError_t launch_gemm_lm_head(const lhs_table &t, const void *resid, int batch, int k, float invT,
                                float *raw, const GemmBuffers &bufs, int32_t *err, int clusters,
                                const DeviceInfo &dev, cudaStream_t stream) {
    CUtensorMap tm_x, tm_t;
    if (!make_tma_map_16bit(&tm_x, resid, t.hidden, batch, static_cast<uint64_t>(t.hidden) * 2, GK, GM,
                            true) ||
        !make_tma_map_16bit(&tm_t, t.data, t.hidden, t.vocab, t.row_bytes, GK, GN / 2, true))
        return cudaErrorInvalidValue;
    GemmParams p = {};
    p.V = t.vocab;
    p.K = t.hidden;
    p.B = batch;
    p.k = k;
    p.invT = invT;
    p.tiles = static_cast<int>((t.vocab + GN - 1) / GN);
    p.clusters = clusters;
    p.err = err;

    if (raw) {
        p.raw = raw;
        return launch_mode<kModeRaw>(tm_x, tm_t, p, dev, stream);
    }
    p.keys = bufs.cand;
    p.ms = bufs.ms;
    p.cap = bufs.cap;
    if (!bufs.sample) return launch_mode<kModeMain>(tm_x, tm_t, p, dev, stream);
    p.sample = bufs.sample;
    p.bound = bufs.bound;
    p.sync = bufs.sync;
    const cudaError_t e = launch_pdl(gemm_sync_reset_kernel, dim3(1), dim3(32), 0, stream, bufs.sync);
    if (e != cudaSuccess) return e;
    return launch_mode<kModeFused>(tm_x, tm_t, p, dev, stream);
}

}  // namespace lhs
