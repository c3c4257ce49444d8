// gemv_q8.cu — steps 2+3 over a Q8_0 table: the lm_head projection on the
// tensor cores, with the fused top-k of lm_topk.cuh.
//
// ADR-0008 "Remote Embeddings and lm_head Service", POST /v1/logits: the
// projection residual @ lm_head.T over every vocab row.  "embedding-inference
// — Port Specification", Tensor inventory: the table stored as Q8_0, value =
// d * q with one f16 scale d per block of 32 int8 codes, 34-byte blocks
// {f16 d; int8 q[32]} laid end to end along a row.
//
// A logit is sum over blocks j of d[v][j] * (sum over the block's 32 values
// of q[v][i] * x[i]).  The inner sums run on mma.sync m16n8k16 with f16
// operands and f32 accumulation, exactly:
//  * a code q (-128..127) becomes the f16 1024 + (q + 128) by placing its
//    bits, sign bit flipped, under the exponent byte 0x64; subtracting 1152
//    leaves q exactly (every integer up to 2048 is an f16);
//  * each residual enters as four f16 columns, two levels of a hi/lo pair:
//    scaled by a power of two 2^e (exact) so that its largest finite
//    magnitude lies in [2^14, 2^15), a value x' = x 2^e with |x'| >= 2^-5
//    goes to level 0 as hi = rn16(x'), lo = rn16(x' - hi); a smaller one to
//    level 1, scaled by 2^20 more.  Each value within 2^-40 of the largest
//    is then held to a relative 2^-20 or better, with no f16 overflow
//    whatever the residual's range (smaller values keep an absolute error
//    below 2^-45 of the largest);
//  * products of two f16 are exact in f32.  A block's two MMAs start from
//    zero, and the block's f32 sum is scaled by d and added to the row's f32
//    accumulator (one FMA per block and column); the logit is
//    (hi0 + lo0) 2^-e + (hi1 + lo1) 2^-(e+20).
// The order of the 32 values inside a block is free (a sum), so each thread
// takes the same four consecutive codes of both 16-value halves for its A
// fragment as its B fragment holds: loads of 4-byte words with no bank
// conflicts (a row of a stage is 272 bytes: rows 8 apart differ by 4 banks).
// A non-finite residual value enters level 0's hi unscaled (inf or NaN,
// lo = 0), so such logits are inf or NaN as the products dictate.
//
// Layout: one CTA per SM, 8 consumer warps of 16 vocab rows each, one
// producer warp and one selection warp (lm_topk.cuh: the consumers only stage
// each block's logits; the selection warp keeps the top-k lists).  The producer keeps a ring of TMA tiles in flight: 128
// table rows x 8 Q8_0 blocks (256 values, 272 bytes, no swizzle); the CTA's
// 128-row blocks are those of the tensor-core GEMV (interleaved over the
// table, then an even share of the rest).  The residual operand is built by
// the consumers once per pass, in shared memory, already in B-fragment order
// (one 16-byte load per thread per block and column group).
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <mutex>

#include "lhs_internal.cuh"
#include "lm_topk.cuh"

namespace lhs {
namespace {

constexpr int kQBlk = 32;                                 // values per Q8_0 block
constexpr int kQBlkBytes = 34;                            // {f16 d; int8 q[32]}
constexpr int kQChunkBlocks = 8;                          // Q8_0 blocks per stage: 256 values
constexpr int kQChunkBytes = kQChunkBlocks * kQBlkBytes;  // 272
constexpr int kQChunkU16 = kQChunkBytes / 2;              // TMA box width in 16-bit units
constexpr int kQStageBytes = BM * kQChunkBytes;           // 34,816 = 34 KB
constexpr int kQBoxRowsSmall = 16;                        // box of the ragged last block
constexpr int kQWarps = 8;
constexpr int kQConsumers = kQWarps * 32;
constexpr int kQThreads = kQConsumers + 64;  // + the producer warp and the selection warp
constexpr int kQMaxStages = 8;
constexpr int kQFragBytes = 32 * 16;  // one B fragment set: 32 lanes x 4 registers

static_assert(kQStageBytes % 1024 == 0, "stages stay 1 KB aligned");
// residual values the prologue stages in the top-k state's candidate keys
// and the scratch keys that follow them
constexpr int kQStagedFloats = (kCandTotal + kBatchChunk * kMaxK) * 2;
static_assert(offsetof(TopkShared, scratch) == sizeof(uint64_t) * kCandTotal, "scratch follows the candidate keys");

struct Q8Params {
    int64_t V;
    int K;
    int nchunk;  // stages per 128-row block (K / 256)
    int nst;     // ring stages
    int Bc;      // residuals in this pass (<= 8)
    int b_off;
    int batch_total;
    int k;
    float invT;
    float *raw;
    uint64_t *part_keys;
    float2 *part_ms;
    const void *resid;  // this pass's residuals [Bc x K]
    int resid_f32;
    int32_t *err;
};

struct Q8Head {
    uint64_t full[kQMaxStages];
    uint64_t empty[kQMaxStages];
    // per residual and level l: 2^(e + 20 l) = up1 * up2, its inverse dn1 * dn2
    float up1[kBatchChunk][2], up2[kBatchChunk][2];
    float dn1[kBatchChunk][2], dn2[kBatchChunk][2];
    TopkShared tk;
};

// Shared memory: [ring nst x 34 KB][Q8Head][B fragments (K / 32) x NB x 512 B]
__host__ __device__ __forceinline__ size_t q8_head_offset(int nst) {
    return static_cast<size_t>(nst) * kQStageBytes;
}
__host__ __device__ __forceinline__ size_t q8_frag_offset(int nst) {
    return (q8_head_offset(nst) + sizeof(Q8Head) + 127) & ~size_t(127);
}
__host__ __device__ __forceinline__ size_t q8_smem_bytes(int nst, int K, int NB) {
    return 1024 + q8_frag_offset(nst) + static_cast<size_t>(K / kQBlk) * NB * kQFragBytes;
}

__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Two codes whose bytes sit at positions 0 and 2 of `h` (positions 1 and 3
// ignored) -> the f16 pair (q0, q1), exactly.  One lop3 flips the codes'
// sign bits and puts the exponent byte 0x64 above each: f16 1024 + (q + 128).
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t h) {
    uint32_t t;
    // out = mask ? (h ^ c) : c  with mask = 0x00FF00FF, c = 0x64806480
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(t) : "r"(h), "r"(0x00FF00FFu), "r"(0x64806480u));
    const __half2 v = __hsub2(*reinterpret_cast<const __half2 *>(&t), __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The code words of one Q8_0 block for the thread's rows (g: row, g+8:
// row8) and its four codes of each 16-value half (4c .. 4c+3 and
// 16+4c .. 16+4c+3).  ODD: the block starts 2 bytes past a 4-byte boundary,
// so its codes start on one and each half's four codes are one word;
// otherwise they straddle two words (codes 0,1 = bytes 2,3 of the first,
// codes 2,3 = bytes 0,1 of the second).
template <bool ODD>
struct Q8Words {
    uint32_t w[2][2][ODD ? 1 : 2];  // [half m][row g, g+8][word]
};
template <bool ODD>
__device__ __forceinline__ void q8_load_words(const uint8_t *row, const uint8_t *row8, int c, Q8Words<ODD> &q) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int o = 2 + 16 * m + 4 * c;  // first code of the thread's four
        if (ODD) {
            q.w[m][0][0] = lds32(row + o);
            q.w[m][1][0] = lds32(row8 + o);
        } else {
            q.w[m][0][0] = lds32(row + o - 2);
            q.w[m][0][1] = lds32(row + o + 2);
            q.w[m][1][0] = lds32(row8 + o - 2);
            q.w[m][1][1] = lds32(row8 + o + 2);
        }
    }
}
// A fragments: a[m] = {row g codes 0,1; row g+8 codes 0,1; row g codes 2,3;
// row g+8 codes 2,3}.
template <bool ODD>
__device__ __forceinline__ void q8_block_a(const Q8Words<ODD> &q, uint32_t (&a)[2][4]) {
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            uint32_t lo, hi;  // codes 0,1 / 2,3 in bytes 0 and 2
            if (ODD) {
                lo = __byte_perm(q.w[m][r][0], 0u, 0x1100);
                hi = __byte_perm(q.w[m][r][0], 0u, 0x3322);
            } else {
                lo = __byte_perm(q.w[m][r][0], 0u, 0x3322);
                hi = __byte_perm(q.w[m][r][1], 0u, 0x1100);
            }
            a[m][r] = codes_to_f16x2(lo);
            a[m][2 + r] = codes_to_f16x2(hi);
        }
}

// NB: column groups of 8: residuals 2 nb and 2 nb + 1, each as columns
// (hi, lo) of level 0 then (hi, lo) of level 1.  RAW: write the logits
// instead of the top-k lists (the selection warp then has nothing to do).
template <bool RAW, int NB>
__global__ void __launch_bounds__(kQThreads, 1)
    gemv_q8_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a16,
                   const Q8Params p) {
    extern __shared__ uint8_t dyn_smem[];
    uint8_t *base = smem_align<1024>(dyn_smem);
    Q8Head &hd = *reinterpret_cast<Q8Head *>(base + q8_head_offset(p.nst));
    uint4 *frag = reinterpret_cast<uint4 *>(base + q8_frag_offset(p.nst));
    TopkShared &tk = hd.tk;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nblk = tc_blocks(p.V, gridDim.x, blockIdx.x);
    const int nst = p.nst;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&hd.full[s], 1);
            mbar_init(&hd.empty[s], kQWarps);
        }
        sel_init(tk, kQWarps);
        fence_mbar_init();
    }
    if (tid < kQConsumers) topk_init(tk, tid, kQConsumers);
    __syncthreads();
    pdl_trigger();

    if (warp == kQWarps) {
        // ---------------- producer: the table only, never written by an earlier kernel
        if (lane == 0) {
            tma_prefetch_map(&tm_a);
            tma_prefetch_map(&tm_a16);
            const uint32_t total = static_cast<uint32_t>(nblk) * p.nchunk;
            auto issue = [&](uint32_t j, int s) {
                const int blk = j / p.nchunk, ch = j % p.nchunk;
                int64_t row0;
                int rows;
                tc_block(p.V, gridDim.x, blockIdx.x, blk, row0, rows);
                uint8_t *dst = base + static_cast<size_t>(s) * kQStageBytes;
                if (rows == BM) {
                    mbar_arrive_expect_tx(&hd.full[s], kQStageBytes);
                    tma_load_2d(dst, &tm_a, &hd.full[s], ch * kQChunkU16, static_cast<int32_t>(row0));
                } else {
                    const int n16 = (rows + kQBoxRowsSmall - 1) / kQBoxRowsSmall;
                    mbar_arrive_expect_tx(&hd.full[s], static_cast<uint32_t>(n16 * kQBoxRowsSmall * kQChunkBytes));
                    for (int u = 0; u < n16; ++u)
                        tma_load_2d(dst + u * kQBoxRowsSmall * kQChunkBytes, &tm_a16, &hd.full[s], ch * kQChunkU16,
                                    static_cast<int32_t>(row0 + u * kQBoxRowsSmall));
                }
            };
            const uint32_t pre = total < static_cast<uint32_t>(nst) ? total : static_cast<uint32_t>(nst);
            for (uint32_t j = 0; j < pre; ++j) issue(j, static_cast<int>(j));
            uint32_t it = pre;
            int s = static_cast<int>(pre % nst);
            uint32_t ph = (pre / nst) & 1;
            for (; it < total; ++it) {
                if (!mbar_wait(&hd.empty[s], ph ^ 1, kWaitTimeoutNs)) {
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    break;
                }
                if (ld_volatile(&tk.abort_flag)) break;
                issue(it, s);
                if (++s == nst) {
                    s = 0;
                    ph ^= 1;
                }
            }
            // drain: every issued stage must land before the CTA exits
            for (uint32_t j = (it > static_cast<uint32_t>(nst) ? it - nst : 0); j < it; ++j)
                if (!mbar_wait(&hd.full[j % nst], (j / nst) & 1, kWaitTimeoutNs)) {
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    break;
                }
        }
        return;
    }
    if (warp == kQWarps + 1) {
        // ---------------- selection: the CTA's top-k lists and (m, s)
        if (RAW) return;
        pdl_wait();  // the partial lists may still be read by the previous kernel
        sel_run(tk, nblk, [&](int blk, int64_t &row0, int &rows) { tc_block(p.V, gridDim.x, blockIdx.x, blk, row0, rows); },
                p.Bc, p.k, p.invT, p.b_off, p.batch_total, p.part_ms, p.err, lane);
        named_bar_sync(kBarFinal, kQConsumers + 32);
        return;
    }

    // ---------------- consumers
    const int g = lane >> 2, c = lane & 3;
    // the residuals may come from the previous kernel, and the partial lists
    // written below may still be read by it
    pdl_wait();
    // 0. the pass's residuals as f32, staged in the candidate-list bytes of
    //    the top-k state (unused until the first offer) when they fit: one
    //    round of wide loads instead of dependent scalar ones
    const bool staged = p.Bc * p.K <= kQStagedFloats;  // uniform
    float *xst = reinterpret_cast<float *>(tk.cand);
    if (staged) {
        const int total = p.Bc * p.K;
        const uintptr_t ra = reinterpret_cast<uintptr_t>(p.resid);
        if (p.resid_f32 && (p.K & 3) == 0 && (ra & 15) == 0) {
            for (int i = tid; i < total / 4; i += kQConsumers)
                reinterpret_cast<float4 *>(xst)[i] = ld_dep(static_cast<const float4 *>(p.resid) + i);
        } else if (!p.resid_f32 && (p.K & 3) == 0 && (ra & 7) == 0) {
            for (int i = tid; i < total / 4; i += kQConsumers) {
                const uint2 u = ld_dep(static_cast<const uint2 *>(p.resid) + i);
                reinterpret_cast<float4 *>(xst)[i] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                                                 __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
            }
        } else {
            for (int i = tid; i < total; i += kQConsumers)
                xst[i] = p.resid_f32 ? ld_dep(static_cast<const float *>(p.resid) + i)
                                     : __uint_as_float(static_cast<uint32_t>(ld_dep(static_cast<const unsigned short *>(p.resid) + i)) << 16);
        }
        named_bar_sync(kBarAll, kQConsumers);
    }
    auto xval = [&](int b, int kk) -> float {
        const int64_t i = static_cast<int64_t>(b) * p.K + kk;
        if (staged) return xst[i];
        return p.resid_f32 ? ld_dep(static_cast<const float *>(p.resid) + i)
                           : __uint_as_float(static_cast<uint32_t>(ld_dep(static_cast<const unsigned short *>(p.resid) + i)) << 16);
    };
    // 1. per residual (warp b): the power of two 2^e that brings its largest
    //    finite magnitude into [2^14, 2^15)
    if (warp < p.Bc) {
        float m = 0.0f;
        for (int kk = lane; kk < p.K; kk += 32) {
            const float a = fabsf(xval(warp, kk));
            if (a <= 3.402823466e38f) m = fmaxf(m, a);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) {
            int e = 0;
            if (m > 0.0f) {
                // m in [2^(E-1), 2^E), from its bits (normal or subnormal)
                const uint32_t bits = __float_as_uint(m);
                const int ef = static_cast<int>(bits >> 23);
                const int E = ef ? ef - 126 : (31 - __clz(static_cast<int>(bits & 0x7FFFFFu))) - 148;
                e = 15 - E;
            }
            // each factor 2^n with |n| <= 92 is a normal float: bits (127 + n) << 23
            auto pow2 = [](int n) { return __uint_as_float(static_cast<uint32_t>(127 + n) << 23); };
#pragma unroll
            for (int l = 0; l < 2; ++l) {
                const int el = e + 20 * l, e1 = el / 2, e2 = el - e1;
                hd.up1[warp][l] = pow2(e1);
                hd.up2[warp][l] = pow2(e2);
                hd.dn1[warp][l] = pow2(-e1);
                hd.dn2[warp][l] = pow2(-e2);
            }
        }
    }
    named_bar_sync(kBarAll, kQConsumers);
    // 2. the B fragments: entry (block j, group nb, lane ln) holds, for column
    //    n = ln / 4 (residual 2 nb + n / 4, level (n / 2) % 2, hi if n is
    //    even, else lo) and c = ln % 4, the values 16 m + 4 c .. 16 m + 4 c + 3
    //    of block j, m = 0, 1
    {
        const int nb32 = p.K / kQBlk;
        const int total = nb32 * NB * 32;
        for (int i = tid; i < total; i += kQConsumers) {
            const int j = i / (NB * 32), nb = (i / 32) % NB, ln = i % 32;
            const int n = ln >> 2, cc = ln & 3;
            const int b = 2 * nb + (n >> 2);
            const int lvl = (n >> 1) & 1;
            const bool lo_col = n & 1;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (b < p.Bc) {
                const float u10 = hd.up1[b][0], u20 = hd.up2[b][0];
                const float u11 = hd.up1[b][1], u21 = hd.up2[b][1];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float x = xval(b, j * kQBlk + 16 * m + 4 * cc + u);
                        uint16_t hbits = 0;
                        if (fabsf(x) <= 3.402823466e38f) {
                            const float x0 = (x * u10) * u20;
                            const int xl = fabsf(x0) >= 0.03125f ? 0 : 1;  // 2^-5
                            if (xl == lvl) {
                                const float xs = xl ? (x * u11) * u21 : x0;
                                const __half h = __float2half_rn(xs);
                                hbits = lo_col ? __half_as_ushort(__float2half_rn(xs - __half2float(h)))
                                               : __half_as_ushort(h);
                            }
                        } else if (lvl == 0 && !lo_col) {
                            hbits = __half_as_ushort(__float2half_rn(x));  // inf, NaN
                        }
                        // register 2m: values 0,1; register 2m+1: values 2,3
                        w[2 * m + (u >> 1)] |= static_cast<uint32_t>(hbits) << (16 * (u & 1));
                    }
            }
            frag[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    // the thread's columns 2c, 2c+1: residual 2 nb + c / 2, level c % 2
    float dn1[NB], dn2[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int b = 2 * nb + (c >> 1);
        dn1[nb] = b < p.Bc ? hd.dn1[b][c & 1] : 1.0f;
        dn2[nb] = b < p.Bc ? hd.dn2[b][c & 1] : 1.0f;
    }
    named_bar_sync(kBarAll, kQConsumers);

    int s = 0;
    uint32_t ph = 0;
    const uint4 *frag_l = frag + lane;
    for (int blk = 0; blk < nblk; ++blk) {
        int64_t row0;
        int rows;
        tc_block(p.V, gridDim.x, blockIdx.x, blk, row0, rows);
        const bool active = warp * 16 < rows;
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
        for (int ch = 0; ch < p.nchunk; ++ch) {
            if (!ld_volatile(&tk.abort_flag)) {
                if (!mbar_wait(&hd.full[s], ph, kWaitTimeoutNs)) {
                    if (lane == 0) {
                        set_err(p.err, LHS_ERRBIT_TIMEOUT);
                        tk.abort_flag = 1;
                    }
                } else if (active) {
                    const uint8_t *row = base + static_cast<size_t>(s) * kQStageBytes + (warp * 16 + g) * kQChunkBytes;
                    const uint8_t *row8 = row + 8 * kQChunkBytes;
                    const uint4 *fr = frag_l + static_cast<size_t>(ch) * kQChunkBlocks * NB * 32;
#pragma unroll
                    for (int jb = 0; jb < kQChunkBlocks; ++jb) {
                        const uint8_t *pb = row + jb * kQBlkBytes, *pb8 = row8 + jb * kQBlkBytes;
                        uint32_t a[2][4];
                        if (jb & 1) {
                            Q8Words<true> q;
                            q8_load_words<true>(pb, pb8, c, q);
                            q8_block_a<true>(q, a);
                        } else {
                            Q8Words<false> q;
                            q8_load_words<false>(pb, pb8, c, q);
                            q8_block_a<false>(q, a);
                        }
                        const float d = __half2float(*reinterpret_cast<const __half *>(pb));
                        const float d8 = __half2float(*reinterpret_cast<const __half *>(pb8));
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb) {
                            const uint4 bfv = fr[(jb * NB + nb) * 32];
                            float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            mma_f16(t, a[0][0], a[0][1], a[0][2], a[0][3], bfv.x, bfv.y);
                            mma_f16(t, a[1][0], a[1][1], a[1][2], a[1][3], bfv.z, bfv.w);
                            acc[nb][0] = fmaf(d, t[0], acc[nb][0]);
                            acc[nb][1] = fmaf(d, t[1], acc[nb][1]);
                            acc[nb][2] = fmaf(d8, t[2], acc[nb][2]);
                            acc[nb][3] = fmaf(d8, t[3], acc[nb][3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hd.empty[s]);
            if (++s == nst) {
                s = 0;
                ph ^= 1;
            }
        }
        // epilogue: thread holds rows (g, g+8) x columns (2c, 2c+1), the hi
        // and lo of residual 2 nb + c / 2 at level c % 2.  Both threads of a
        // pair form the logit, level-0 part + level-1 part (the same sum in
        // either order); the even one takes row g, the odd one row g+8.  The
        // logits are written out (raw) or staged for the selection warp.
        bool staged = RAW;
        if (!RAW && active && !ld_volatile(&tk.abort_flag)) {
            if (!sel_acquire(tk, blk)) {
                if (lane == 0) {
                    set_err(p.err, LHS_ERRBIT_TIMEOUT);
                    tk.abort_flag = 1;
                }
            } else {
                staged = true;
            }
        }
        if (active && staged) {
            float *st = RAW ? nullptr : sel_slot(tk, blk);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                float val[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float part = ((acc[nb][2 * r] + acc[nb][2 * r + 1]) * dn1[nb]) * dn2[nb];
                    val[r] = part + __shfl_xor_sync(0xFFFFFFFFu, part, 1);
                }
                const int r = c & 1;
                const float vr = r ? val[1] : val[0];  // a select: no indexed local array
                const int b = 2 * nb + (c >> 1);
                const int rr = warp * 16 + g + 8 * r;  // row within the block
                if (b < p.Bc) {
                    if (RAW) {
                        if (rr < rows) p.raw[static_cast<int64_t>(p.b_off + b) * p.V + row0 + rr] = vr;
                    } else {
                        st[b * BM + rr] = vr;
                    }
                }
            }
        }
        if (RAW) named_bar_sync(kBarAll, kQConsumers);
        else sel_publish(tk, blk, lane);
        // the flag only changes inside the stage loop or just above: every
        // consumer reads the same value here after the CTA barrier (raw), and
        // every lane of a warp after the warp barrier of sel_publish
        if (ld_volatile(&tk.abort_flag)) break;
    }
    if (RAW) return;
    // the CTA's partial lists, written by the consumers once the selection
    // warp has taken every block
    named_bar_sync(kBarFinal, kQConsumers + 32);
    if (ld_volatile(&tk.abort_flag)) return;
    topk_write_lists(tk, tid, kQConsumers, p.Bc, p.k, kCandTotal / pow2_at_least(p.Bc), p.b_off, p.batch_total,
                     p.part_keys);
}

}  // namespace

// Stages of the ring for passes of up to bc residuals over hidden K, as many
// as shared memory holds (at most kQMaxStages); 0 when fewer than 2 fit.
int gemv_q8_stages(int K, int bc, int max_smem) {
    const int NB = (bc + 1) / 2;
    int nst = kQMaxStages;
    while (nst >= 2 && q8_smem_bytes(nst, K, NB) > static_cast<size_t>(max_smem)) --nst;
    return nst >= 2 ? nst : 0;
}

cudaError_t launch_gemv_q8(const lhs_table &t, int nst, const void *resid, int32_t resid_dtype, int32_t batch,
                           int32_t k, float invT, float *raw, uint64_t *part_keys, float2 *part_ms,
                           int32_t *err, int grid, const DeviceInfo &dev, cudaStream_t stream) {
    CUtensorMap tm_a, tm_a16;
    const uint64_t cols = static_cast<uint64_t>(t.row_bytes) / 2;
    if (!make_tma_map_u16_plain(&tm_a, t.data, cols, t.vocab, t.row_bytes, kQChunkU16, BM) ||
        !make_tma_map_u16_plain(&tm_a16, t.data, cols, t.vocab, t.row_bytes, kQChunkU16, kQBoxRowsSmall))
        return cudaErrorInvalidValue;
    using Kern = void (*)(const CUtensorMap, const CUtensorMap, const Q8Params);
    // [raw][column groups - 1]
    static const Kern kTable[2][4] = {
        {gemv_q8_kernel<false, 1>, gemv_q8_kernel<false, 2>, gemv_q8_kernel<false, 3>, gemv_q8_kernel<false, 4>},
        {gemv_q8_kernel<true, 1>, gemv_q8_kernel<true, 2>, gemv_q8_kernel<true, 3>, gemv_q8_kernel<true, 4>}};
    const bool is_raw = raw != nullptr;
    {
        // one attribute flag per instantiation: the largest size this device allows
        static std::mutex mu;
        static bool done[8][64] = {};
        std::lock_guard<std::mutex> lock(mu);
        for (int r = 0; r < 2; ++r)
            for (int n = 0; n < 4; ++n)
                if (!done[r * 4 + n][dev.device]) {
                    const cudaError_t e = cudaFuncSetAttribute(kTable[r][n], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                               dev.max_smem_optin);
                    if (e != cudaSuccess) return e;
                    done[r * 4 + n][dev.device] = true;
                }
    }
    const size_t relt = resid_dtype == LHS_F32 ? 4 : 2;
    for (int c0 = 0; c0 < batch; c0 += kBatchChunk) {
        const int Bc = batch - c0 < kBatchChunk ? batch - c0 : kBatchChunk;
        const int NB = (Bc + 1) / 2;
        Q8Params p;
        p.V = t.vocab;
        p.K = t.hidden;
        p.nchunk = t.hidden / (kQChunkBlocks * kQBlk);
        p.nst = nst;
        p.Bc = Bc;
        p.b_off = c0;
        p.batch_total = batch;
        p.k = k;
        p.invT = invT;
        p.raw = raw;
        p.part_keys = part_keys;
        p.part_ms = part_ms;
        p.resid = static_cast<const uint8_t *>(resid) + static_cast<size_t>(c0) * t.hidden * relt;
        p.resid_f32 = resid_dtype == LHS_F32;
        p.err = err;
        const cudaError_t e = launch_pdl(kTable[is_raw][NB - 1], dim3(grid), dim3(kQThreads),
                                         q8_smem_bytes(nst, t.hidden, NB), stream, tm_a, tm_a16, p);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace lhs
