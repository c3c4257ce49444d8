// lhs_internal.cuh — device helpers and launcher prototypes shared by the
// kernels of the GB300 embed / tied lm_head library.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lhs.h"

namespace lhs {

// ---------------------------------------------------------------------------
// error word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_err(int32_t *err, int bits) {
    atomicOr(reinterpret_cast<int *>(err), bits);
}

// ---------------------------------------------------------------------------
// Total order of (logit, token id) used by top-k: logit descending, equal
// logits by id ascending, +0 == -0, NaN above every number.  The 64-bit key
// is larger for the better entry; 0 never encodes a real entry.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key32(float v) {
    uint32_t u = __float_as_uint(v);
    if (v != v) u = 0x7FC00000u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t topk_key(float v, int32_t id) {
    return (static_cast<uint64_t>(order_key32(v)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}
__device__ __forceinline__ float key_value(uint64_t key) {
    uint32_t k = static_cast<uint32_t>(key >> 32);
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}
__device__ __forceinline__ int32_t key_id(uint64_t key) {
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers, TMA, bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// `p` (a pointer into shared memory) advanced to the next multiple of ALIGN
// bytes of the shared window.  The offset is added to p itself, so the
// compiler still knows that the result points into shared memory and emits
// shared loads, stores and atomics through it; a round trip through an
// integer would leave a generic pointer, whose accesses take the slower
// generic path.
template <unsigned ALIGN>
__device__ __forceinline__ uint8_t *smem_align(uint8_t *p) {
    static_assert((ALIGN & (ALIGN - 1)) == 0, "a power of two");
    return p + ((ALIGN - (smem_u32(p) & (ALIGN - 1))) & (ALIGN - 1));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait until the barrier phase with the given parity completes, for at most
// timeout_ns.  Returns false when the limit ran out (the caller records
// LHS_ERRBIT_TIMEOUT and leaves its loop).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > timeout_ns) return false;
    }
}

// One contiguous bulk copy global -> shared, completing on `bar` (both
// addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :
                 : "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(gmem_src)), "r"(bytes),
                   "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled TMA load global -> shared, completion signalled on `bar` as
// transaction bytes.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// ---------------------------------------------------------------------------
// Element decode and wire encoding helpers shared by the gather, the wire
// codecs and the fused embed -> wire kernel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// Stored element j of a table row, widened exactly to binary32 (Q8_0: d*q,
// exact: an 11-bit by 8-bit significand product fits in 24 bits).
template <int DT>
__device__ __forceinline__ float row_element(const uint8_t *row, int j) {
    if (DT == LHS_F32) return __ldg(reinterpret_cast<const float *>(row) + j);
    if (DT == LHS_F16) return f16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short *>(row) + j));
    if (DT == LHS_BF16) return bf16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short *>(row) + j));
    const uint8_t *blk = row + (j >> 5) * 34;  // Q8_0 block: [f16 d][32 x int8]
    const float d = f16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short *>(blk)));
    const float q = static_cast<float>(static_cast<int8_t>(__ldg(blk + 2 + (j & 31))));
    return __fmul_rn(d, q);
}

// Elements 8g .. 8g+7 of a row (hidden % 8 == 0; f32/f16/bf16 rows 16-byte
// aligned; Q8_0 rows 2-byte aligned).
template <int DT>
__device__ __forceinline__ void row_elements8(const uint8_t *row, int g, float (&v)[8]) {
    if (DT == LHS_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(row) + 2 * g;
        const float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if (DT == LHS_F16 || DT == LHS_BF16) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(row) + g);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = DT == LHS_F16 ? f16_bits_to_f32(u[i] & 0xFFFFu) : bf16_bits_to_f32(u[i] & 0xFFFFu);
            v[2 * i + 1] = DT == LHS_F16 ? f16_bits_to_f32(u[i] >> 16) : bf16_bits_to_f32(u[i] >> 16);
        }
    } else {
        const uint8_t *blk = row + (g >> 2) * 34;
        const unsigned short *b16 = reinterpret_cast<const unsigned short *>(blk);
        const float d = f16_bits_to_f32(__ldg(b16));
        const int q0 = 1 + (g & 3) * 4;  // codes (g & 3) * 8 .. +7, two per 16-bit word
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w = __ldg(b16 + q0 + i);
            v[2 * i] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w & 0xFF)));
            v[2 * i + 1] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w >> 8)));
        }
    }
}

// Elements 4s .. 4s+3 of a row (hidden % 4 == 0; f32 rows 16-byte aligned,
// f16/bf16 rows 8-byte aligned; Q8_0 rows 2-byte aligned).
template <int DT>
__device__ __forceinline__ void row_elements4(const uint8_t *row, int s, float (&v)[4]) {
    if (DT == LHS_F32) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(row) + s);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if (DT == LHS_F16 || DT == LHS_BF16) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(row) + s);
        v[0] = DT == LHS_F16 ? f16_bits_to_f32(w.x & 0xFFFFu) : bf16_bits_to_f32(w.x & 0xFFFFu);
        v[1] = DT == LHS_F16 ? f16_bits_to_f32(w.x >> 16) : bf16_bits_to_f32(w.x >> 16);
        v[2] = DT == LHS_F16 ? f16_bits_to_f32(w.y & 0xFFFFu) : bf16_bits_to_f32(w.y & 0xFFFFu);
        v[3] = DT == LHS_F16 ? f16_bits_to_f32(w.y >> 16) : bf16_bits_to_f32(w.y >> 16);
    } else {
        const unsigned short *b16 = reinterpret_cast<const unsigned short *>(row + (s >> 3) * 34);
        const float d = f16_bits_to_f32(__ldg(b16));
        const int q0 = 1 + (s & 7) * 2;  // codes (s & 7) * 4 .. +3, two per 16-bit word
        const uint32_t w0 = __ldg(b16 + q0), w1 = __ldg(b16 + q0 + 1);
        v[0] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w0 & 0xFF)));
        v[1] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w0 >> 8)));
        v[2] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w1 & 0xFF)));
        v[3] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w1 >> 8)));
    }
}

// binary16 bits of x, round to nearest even; a finite x whose rounding
// overflows saturates to +-65504, inf stays inf, NaN becomes 0x7E00.
__device__ __forceinline__ uint32_t f16_sat_bits(float x) {
    if (x != x) return 0x7E00u;
    uint32_t b = __half_as_ushort(__float2half_rn(x));
    if ((b & 0x7FFFu) == 0x7C00u && isfinite(x)) b = (b & 0x8000u) | 0x7BFFu;
    return b;
}

// Eight binary16 values packed in a 16-byte word with f16_sat_bits' rules.
// When every value is finite and below 65504 in magnitude (no saturation,
// no inf/NaN), the conversion is two-at-a-time round-to-nearest-even.
__device__ __forceinline__ uint4 pack_f16x8(const float (&v)[8]) {
    bool plain = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) plain = plain && (fabsf(v[i]) < 65504.0f);  // false for NaN
    uint32_t w[4];
    if (plain) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = f16_sat_bits(v[2 * i]) | (f16_sat_bits(v[2 * i + 1]) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// i8 code of v: round half to even of the correctly rounded binary32
// quotient v / scale, clamped to [-127, 127]; 0 when scale is 0.  Returned
// as an int (its low byte is the code's two's-complement byte).
// rcp = __frcp_rn(scale).  The product t = RN(v * rcp) is within
// |v/scale| * 2^-23 of the exact quotient Q, and RN(Q) within |Q| * 2^-24
// of it; for |t| < 256 the two therefore differ by less than 2^-14.4, so
// unless t lies within 2^-12 of a half-integer (a rounding boundary of rint)
// both round to the same integer.  The test is on d = t - rint(t), exact
// (t and rint(t) are within a factor of two, or rint(t) = 0): |d| < 1/2 -
// 2^-12 means no boundary is near.  Near one — or when t is out of that
// range, e.g. a reciprocal that overflowed — the quotient is formed by the
// correctly rounded divide instead.
__device__ __forceinline__ int i8_code(float v, float scale, float rcp) {
    if (scale == 0.0f) return 0;
    const float t = __fmul_rn(v, rcp);
    float r = rintf(t);
    if (!(fabsf(t) < 256.0f && fabsf(t - r) < 0.5f - 0x1p-12f)) r = rintf(__fdiv_rn(v, scale));
    return __float2int_rn(fminf(fmaxf(r, -127.0f), 127.0f));
}

// The low bytes of four codes, first in the lowest byte.
__device__ __forceinline__ uint32_t pack_i8x4(int a, int b, int c, int d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// The codes of N values, the same as i8_code's, without conversion
// instructions on the common path: for |t| < 2^22, y = RN(t + 1.5 * 2^23)
// lies in [2^23, 2^24], where the spacing is 1, so y is t rounded half to
// even plus 1.5 * 2^23 — r = y - 1.5 * 2^23 (exact) is rint(t), and the
// bits of y are 0x4B400000 + rint(t).  When |t| < 127.5 and t is not within
// 2^-12 of a half-integer, rint(t) is the code (i8_code's argument), already
// in [-127, 127].  The other values, rare, take the correctly rounded divide
// in a loop over their bits that the compiler cannot turn into N divides for
// every call.  q[i]'s low byte is the code.
template <int N>
__device__ __forceinline__ void i8_codes(const float (&v)[N], float scale, float rcp, int (&q)[N]) {
    if (scale == 0.0f) {
#pragma unroll
        for (int i = 0; i < N; ++i) q[i] = 0;
        return;
    }
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    uint32_t slow = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float t = __fmul_rn(v[i], rcp);
        const float y = __fadd_rn(t, kMagic);
        const float r = __fsub_rn(y, kMagic);
        q[i] = static_cast<int>(__float_as_uint(y) - 0x4B400000u);
        if (!(fabsf(t) < 127.5f && fabsf(__fsub_rn(t, r)) < 0.5f - 0x1p-12f)) slow |= 1u << i;
    }
    while (slow) {
        const int i = __ffs(slow) - 1;
        slow &= slow - 1;
        float vi = v[0];
#pragma unroll
        for (int j = 1; j < N; ++j) vi = i == j ? v[j] : vi;
        const int qi = __float2int_rn(fminf(fmaxf(rintf(__fdiv_rn(vi, scale)), -127.0f), 127.0f));
#pragma unroll
        for (int j = 0; j < N; ++j) q[j] = i == j ? qi : q[j];
    }
}

// Eight codes as two little-endian words.
__device__ __forceinline__ uint2 i8_code8(const float (&v)[8], float scale, float rcp) {
    int q[8];
    i8_codes<8>(v, scale, rcp, q);
    return make_uint2(pack_i8x4(q[0], q[1], q[2], q[3]), pack_i8x4(q[4], q[5], q[6], q[7]));
}

// Four codes as one little-endian word.
__device__ __forceinline__ uint32_t i8_code4(const float (&v)[4], float scale, float rcp) {
    int q[4];
    i8_codes<4>(v, scale, rcp, q);
    return pack_i8x4(q[0], q[1], q[2], q[3]);
}

// Block-wide max of non-negative values and OR of a flag; every thread gets
// the result.  sm_m / sm_f hold one entry per warp.
__device__ __forceinline__ void block_max_or(float &m, int &flag, float *sm_m, int *sm_f) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        flag |= __shfl_xor_sync(0xFFFFFFFFu, flag, o);
    }
    if (lane == 0) {
        sm_m[warp] = m;
        sm_f[warp] = flag;
    }
    __syncthreads();
    m = sm_m[0];
    flag = sm_f[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) {
        m = fmaxf(m, sm_m[w]);
        flag |= sm_f[w];
    }
    __syncthreads();
}

// One i8 position by one warp, in two passes over its values: max|x| (and
// whether any value is inf/NaN), then scale = RN(m / 127) and the codes.
// load8(g, v) yields values 8g .. 8g+7 (ng groups); the second pass reads
// them again, from L1/L2.  pos: [scale f32][zero point f32 = 0][codes],
// 8-byte aligned.
template <typename Load8>
__device__ __forceinline__ void i8_position_warp(const Load8 &load8, int ng, uint8_t *pos, int lane,
                                                 int32_t *err) {
    float m = 0.0f;
    bool nonfinite = false;
#pragma unroll 4
    for (int g = lane; g < ng; g += 32) {
        float v[8];
        load8(g, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (!isfinite(v[i])) nonfinite = true;
            else m = fmaxf(m, fabsf(v[i]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    nonfinite = __any_sync(0xFFFFFFFFu, nonfinite);
    const float scale = nonfinite ? 0.0f : __fdiv_rn(m, 127.0f);
    const float rcp = __frcp_rn(scale);
    if (lane == 0) {
        *reinterpret_cast<uint2 *>(pos) = make_uint2(__float_as_uint(scale), 0u);
        if (nonfinite) set_err(err, LHS_ERRBIT_NONFINITE);
    }
    uint2 *codes = reinterpret_cast<uint2 *>(pos + 8);
#pragma unroll 2
    for (int g = lane; g < ng; g += 32) {
        float v[8];
        load8(g, v);
        codes[g] = i8_code8(v, scale, rcp);
    }
}

// One i8 position of at most 32 * kI8WarpSteps * 4 values by one warp, the
// values kept in registers between the two passes: load4(s, v) yields
// values 4s .. 4s+3 (n4 steps; lane l takes steps l, l + 32, ...; every load
// is issued before the first value is used).  Same results as
// i8_position_warp.  pos: [scale f32][zero point f32 = 0][codes], 4-byte
// aligned codes.
constexpr int kI8WarpSteps = 8;  // rows up to 1024 values
template <typename Load4>
__device__ __forceinline__ void i8_position_warp4(const Load4 &load4, int n4, uint8_t *pos, int lane,
                                                  int32_t *err) {
    float c[kI8WarpSteps][4];
#pragma unroll
    for (int k = 0; k < kI8WarpSteps; ++k)
        if (lane + 32 * k < n4) load4(lane + 32 * k, c[k]);
    // max|x| (fmaxf passes over NaN) and, in z, 0 * x summed: NaN exactly
    // when some x is inf or NaN
    float m = 0.0f, z = 0.0f;
#pragma unroll
    for (int k = 0; k < kI8WarpSteps; ++k)
        if (lane + 32 * k < n4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                m = fmaxf(m, fabsf(c[k][i]));
                z = __fmaf_rn(c[k][i], 0.0f, z);
            }
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const bool nonfinite = __any_sync(0xFFFFFFFFu, z != z);
    const float scale = nonfinite ? 0.0f : __fdiv_rn(m, 127.0f);
    const float rcp = __frcp_rn(scale);
    if (lane == 0) {
        *reinterpret_cast<uint2 *>(pos) = make_uint2(__float_as_uint(scale), 0u);
        if (nonfinite) set_err(err, LHS_ERRBIT_NONFINITE);
    }
    uint32_t *codes = reinterpret_cast<uint32_t *>(pos + 8);
#pragma unroll
    for (int k = 0; k < kI8WarpSteps; ++k)
        if (lane + 32 * k < n4) codes[lane + 32 * k] = i8_code4(c[k], scale, rcp);
}

// Warps per SM for the warp-per-position i8 kernels: as many as keep the
// positions' values (the second pass re-reads them) within about 192 KB of
// L1, between 8 and 48.
inline int i8_warps_per_sm(int64_t bytes_per_position) {
    int64_t w = (192 * 1024) / (bytes_per_position > 0 ? bytes_per_position : 1);
    if (w > 48) w = 48;
    if (w < 8) w = 8;
    return static_cast<int>(w);
}

// Grid of a warp-per-position kernel (4 warps per CTA) for n positions: at
// most `wps` warps per SM and no more CTAs than stay resident at once, so
// the grid is one wave and each warp walks its positions.
// (The occupancy query is made once per kernel and device.)
int resident_ctas_128(const void *kernel, int device);
template <typename K>
int warp_kernel_grid(K kernel, int64_t n, int wps, int num_sms, int device) {
    const int resident = resident_ctas_128(reinterpret_cast<const void *>(kernel), device);
    int per_sm = wps / 4 < resident ? wps / 4 : resident;
    if (per_sm < 1) per_sm = 1;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    const int64_t ctas = (n + 3) / 4;
    return static_cast<int>(ctas < 1 ? 1 : (ctas < cap ? ctas : cap));
}

__device__ __forceinline__ void write_wire_header(uint8_t *buf, uint32_t layer, uint32_t seq_len,
                                                  uint32_t flags, uint32_t top_k) {
    *reinterpret_cast<uint4 *>(buf) = make_uint4(layer, seq_len, flags, top_k);
}

// A message header as little-endian u32 words: the request's 4
// [layer][seq_len][flags][top_k] or the single-layer response's 3
// [layer][seq_len][latency_ms bits]; the payload follows at 4 * n bytes.
struct WireHdr {
    uint32_t w[4];
    int n;
};
__device__ __forceinline__ void write_hdr(uint8_t *buf, const WireHdr &h) {
    for (int i = 0; i < h.n; ++i) reinterpret_cast<uint32_t *>(buf)[i] = h.w[i];
}

// Load of data that the preceding kernel in the stream may have written
// (residuals, token ids, wire messages, intermediate buffers).  A kernel
// launched as a programmatic dependent starts before its predecessor has
// finished; a non-coherent read-only load (ld.global.nc, as __ldg or a
// const __restrict__ pointer produce) counts on its bytes staying fixed for
// the whole kernel, so it may be scheduled ahead of pdl_wait() and return
// the bytes from before the predecessor wrote them.  These loads take the
// coherent L2 path (ld.global.cg), which stays behind the wait.  Only the
// tables, which no kernel writes between calls, are read with __ldg.
template <typename T>
__device__ __forceinline__ T ld_dep(const T *p) {
    return __ldcg(p);
}

// Programmatic dependent launch.  pdl_wait(): block until the preceding
// kernel in the stream has completed and its memory is visible (a no-op when
// this kernel was not launched as a dependent).  pdl_trigger(): allow the
// next kernel in the stream to be scheduled now.  Every kernel here triggers
// at its start and calls pdl_wait() before it reads anything an earlier
// kernel may write and before it writes anything an earlier kernel may read.
// The wait covers the whole earlier kernel's completion, not its trigger, so
// the early trigger only lets the next kernel become resident and run its
// prologue (barrier setup, table prefetch) sooner.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier among `nthreads` threads (multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// constants
// ---------------------------------------------------------------------------
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s bound on any on-chip wait
constexpr int kMaxK = 128;                          // largest top-k served

// ---------------------------------------------------------------------------
// per-device facts (queried once per device)
// ---------------------------------------------------------------------------
struct DeviceInfo {
    int device;
    int num_sms;
    int max_smem_optin;
};
cudaError_t device_info(DeviceInfo *out);

// LHS_OK for cudaSuccess; otherwise records `e` for lhs_last_cuda_error()
// (per host thread) and returns LHS_ERR_CUDA.
int cuda_status(cudaError_t e);

// ---------------------------------------------------------------------------
// launchers (host side); each returns cudaSuccess or the launch error
// ---------------------------------------------------------------------------
cudaError_t launch_embed(const lhs_table &t, const int32_t *ids, int64_t n, float scale,
                         float *out, int32_t *err, cudaStream_t stream);

size_t unique_ids_workspace(int64_t vocab);
cudaError_t launch_unique_ids(int64_t vocab, const int32_t *ids, int64_t n, int32_t *unique, int32_t *inverse,
                              int32_t *count, void *ws, int32_t *err, cudaStream_t stream);
size_t embed_dedup_workspace(const lhs_table &t, int64_t n);
cudaError_t launch_embed_dedup(const lhs_table &t, const int32_t *ids, int64_t n, float scale, float *out,
                               void *ws, int32_t *err, cudaStream_t stream);
cudaError_t launch_embed_mixed(const void *data, int64_t data_bytes, const int64_t *row_offset,
                               const uint8_t *row_dtype, int64_t vocab, int32_t hidden, const int32_t *ids,
                               int64_t n, float scale, float *out, int32_t *err, cudaStream_t stream);
cudaError_t launch_embed_wire(const lhs_table &t, const int32_t *ids, int64_t n, float scale, int fmt,
                              const WireHdr &hdr, void *buf, int32_t *err, cudaStream_t stream);
// hdr.n words of header, then the payload (vector paths when the payload
// and x are 16-byte aligned, element-wise ones otherwise); decode reads the
// payload at buf + hoff
cudaError_t launch_wire_encode(int fmt, const void *x, int x_dtype, int32_t seq_len,
                               int32_t hidden, const WireHdr &hdr, void *buf, int32_t *err,
                               cudaStream_t stream);
cudaError_t launch_wire_decode(int fmt, const void *buf, int hoff, int32_t seq_len, int32_t hidden,
                               float *x, int32_t *err, cudaStream_t stream);

// lm_head: plan (workspace layout + kernel choice) and launch
struct LmHeadPlan {
    int path;          // 0 = tensor-core streaming GEMV (f16/bf16 table, batch <= 8 per pass)
                       // 1 = CUDA-core GEMV (any table dtype)
                       // 2 = tcgen05 GEMM (bf16 table, bf16 residuals, batch > 8)
                       // 3 = bulk-stream CUDA-core GEMV (f32, rows of 16..1024 bytes)
                       // 4 = Q8_0 tensor-core GEMV (hidden % 256 == 0, batch <= 8 per pass)
    int grid;          // CTAs of the projection kernel (= partial top-k lists)
    int batch_chunk;   // residuals per pass of the projection
    int kpad;          // hidden rounded up for the tensor-core operand
    size_t off_x;      // workspace offsets (bytes)
    size_t off_keys;   // partial lists (GEMM: candidate buffers)
    size_t off_ms;
    size_t off_sample, off_bound, off_sync;  // GEMM: first-tile sample, bounds, arrival counters
    int key_stride;    // entries between consecutive partial lists
    bool sample;       // GEMM: bound the candidates by a first-tile sample
    bool xres;         // tensor-core GEMV: residual operand resident in shared memory (no prep kernel)
    int nst;           // tensor-core GEMVs: TMA ring stages
    size_t bytes;      // total workspace
};
int plan_lm_head(const lhs_table &t, int32_t batch, int32_t k, int32_t resid_dtype,
                 const DeviceInfo &dev, LmHeadPlan *plan);
// Kernel launches one lhs_logits_topk (raw = false) or lhs_logits (raw =
// true) call with this plan enqueues.
int lm_head_launches(const LmHeadPlan &plan, int32_t batch, bool raw);
cudaError_t launch_lm_head(const lhs_table &t, const LmHeadPlan &plan, const void *resid,
                           int32_t resid_dtype, int32_t batch, int32_t k, float temperature,
                           int32_t *ids, float *logits_out, float *probs, float *raw_logits,
                           void *ws, int32_t *err, cudaStream_t stream);

cudaError_t launch_selftest_wait(int32_t *err, int64_t timeout_ns, cudaStream_t stream);

// 2-D TMA map over a row-major [rows x cols] 16-bit matrix with the given
// row pitch; box = box_cols x box_rows, 128-byte swizzle, zero fill outside.
bool make_tma_map_16bit(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                        uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, bool bf16);

// 2-D map over a row-major [rows x cols] matrix of 16-bit units (any bytes:
// the Q8_0 GEMV reads its rows' blocks through it) with the given row pitch;
// box = box_cols x box_rows, no swizzle, zero fill outside.
bool make_tma_map_u16_plain(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                            uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows);

// Q8_0 lm_head on the tensor cores (see gemv_q8.cu): ring stages that fit
// for passes of up to bc residuals (0: the kernel does not fit), and the
// projection passes of one call (partial lists per CTA, or raw logits).
int gemv_q8_stages(int K, int bc, int max_smem);
cudaError_t launch_gemv_q8(const lhs_table &t, int nst, const void *resid, int32_t resid_dtype, int32_t batch,
                           int32_t k, float invT, float *raw, uint64_t *part_keys, float2 *part_ms,
                           int32_t *err, int grid, const DeviceInfo &dev, cudaStream_t stream);

// Merge of per-CTA partial lists (stride entries apart, the first len of
// each used) into the sorted top-k per residual, with probabilities when
// `probs` is not null.
cudaError_t launch_merge(const uint64_t *part_keys, const float2 *part_ms, int G, int stride,
                         int len, int batch, int k, float invT, int32_t *ids, float *logits,
                         float *probs, const DeviceInfo &dev, cudaStream_t stream);

// Batched lm_head on tcgen05 (bf16 table, bf16 residuals): clusters of two
// CTAs; see gemm_tc.cu.
struct GemmBuffers {
    uint32_t *sample;        // [batch][clusters][16] first-tile group maxima, null: no sample
    uint32_t *bound;         // [batch] each residual's bound (order key)
    uint32_t *sync;          // two arrival counters, 128 bytes apart
    uint64_t *cand;          // [clusters][batch][cap]
    float2 *ms;              // [clusters][batch]
    int cap;
};
size_t gemm_lm_head_smem();
int gemm_lm_head_max_batch();
int gemm_lm_head_cap(int k);
int gemm_lm_head_sample_groups();
int gemm_lm_head_clusters(const DeviceInfo &dev);
cudaError_t launch_gemm_lm_head(const lhs_table &t, const void *resid, int batch, int k, float invT,
                                float *raw, const GemmBuffers &bufs, int32_t *err, int clusters,
                                const DeviceInfo &dev, cudaStream_t stream);

// Launch `kernel` as a programmatic dependent of the previous work in
// `stream` (its prologue may overlap the tail of the preceding kernel).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace lhs
