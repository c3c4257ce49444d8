// wire.cu — step 4: residual wire encode / decode.
//
// ADR-0009 "Wire Format Evolution: f16 Default + i8 Quantised Residuals",
// Wire Layout: a 16-byte header [layer u32][seq_len u32][flags u32][top_k u32]
// then the payload — binary32 (the unchanged format), binary16, or per
// position [scale f32][zero_point f32][hidden x int8] with symmetric
// quantisation scale = max|x|/127, x^ = q*scale.  Trade-offs: f16 overflow
// clamps to the largest finite value instead of producing inf/NaN.
//
// f32 / f16: one elementwise pass, 8 values per thread (16-byte accesses).
// i8: one warp per position for rows up to 1024 values; longer aligned rows
// staged in shared memory by a bulk copy while the CTA quantises the previous
// one; one CTA per position, element by element, for unaligned rows —
// max-reduce of |x|, one correctly rounded divide for the scale, then
// round-half-even of the binary32 quotient x/scale for every element.
// Positions start at 16 + p*(hidden+8): 8-byte aligned when hidden % 8 == 0,
// so the codes move as 8-byte words.
// The single-layer response (Wire Layout, "Single-layer response") has the
// 12-byte header [layer u32][seq_len u32][latency_ms f32] and the same
// payload: every kernel takes the header words and finds the payload after
// them; the vector paths run when the payload is 16-byte aligned, the
// element-wise ones otherwise.
#include <cuda_fp16.h>

#include <mutex>

#include "lhs_internal.cuh"

namespace lhs {
namespace {

constexpr int kEwThreads = 256;
constexpr int kI8Threads = 128;
constexpr int kI8Cache = 6;     // 8-value groups a thread keeps in registers (CTA path)
constexpr int kI8DecCache = 12;  // 4-code units a decoding thread loads with the header

template <int XDT>
__device__ __forceinline__ float load_x(const void *x, int64_t i) {
    if (XDT == LHS_F32) return ld_dep(static_cast<const float *>(x) + i);
    return __uint_as_float(static_cast<uint32_t>(ld_dep(static_cast<const unsigned short *>(x) + i))
                           << 16);
}

// 8 consecutive values starting at element 8*g (16-byte aligned source).
template <int XDT>
__device__ __forceinline__ void load_x8(const void *x, int64_t g, float (&v)[8]) {
    if (XDT == LHS_F32) {
        const float4 *p = static_cast<const float4 *>(x) + 2 * g;
        const float4 a = ld_dep(p), b = ld_dep(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 w = ld_dep(static_cast<const uint4 *>(x) + g);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(u[i] << 16);
            v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
        }
    }
}

// ---- f32 / f16 encode ------------------------------------------------------
template <int FMT, int XDT, bool VEC>
__global__ void __launch_bounds__(kEwThreads)
    encode_ew_kernel(const void *__restrict__ x, int64_t n, WireHdr hdr, uint8_t *__restrict__ buf) {
    pdl_trigger();
    pdl_wait();
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (tid == 0) write_hdr(buf, hdr);
    uint8_t *pay = buf + 4 * hdr.n;
    // f16: 8 values per step (a 16-byte store each); f32: 4 values per step
    // (a warp's stores are whole 32-byte sectors)
    const int per = FMT == LHS_WIRE_F16 ? 8 : 4;
    const int64_t ng = VEC ? n / per : 0;
    for (int64_t g = tid; g < ng; g += nth) {
        if (FMT == LHS_WIRE_F16) {
            float v[8];
            load_x8<XDT>(x, g, v);
            reinterpret_cast<uint4 *>(pay)[g] = pack_f16x8(v);
        } else if (XDT == LHS_F32) {
            reinterpret_cast<float4 *>(pay)[g] = ld_dep(static_cast<const float4 *>(x) + g);
        } else {
            const uint2 w = ld_dep(static_cast<const uint2 *>(x) + g);
            reinterpret_cast<float4 *>(pay)[g] =
                make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                            __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
        }
    }
    for (int64_t i = ng * per + tid; i < n; i += nth) {
        const float v = load_x<XDT>(x, i);
        if (FMT == LHS_WIRE_F16)
            reinterpret_cast<unsigned short *>(pay)[i] = static_cast<unsigned short>(f16_sat_bits(v));
        else
            reinterpret_cast<float *>(pay)[i] = v;
    }
}

// ---- f32 / f16 decode ------------------------------------------------------
template <int FMT, bool VEC>
__global__ void __launch_bounds__(kEwThreads)
    decode_ew_kernel(const uint8_t *__restrict__ buf, int hoff, int64_t n, uint32_t seq_len,
                     float *__restrict__ x, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint32_t hdr_seq = ld_dep(reinterpret_cast<const uint32_t *>(buf) + 1);
    if (hdr_seq != seq_len) {
        if (tid == 0) set_err(err, LHS_ERRBIT_MALFORMED);
        return;
    }
    const uint8_t *pay = buf + hoff;
    // 4 values per unit: a warp's unit loads and stores are contiguous (512
    // bytes written per instruction, whole 32-byte sectors); kDecUnroll units
    // per thread step, every load issued before the first store
    const int64_t ng = VEC ? n / 4 : 0;
    constexpr int kDecUnroll = 4;
    for (int64_t g0 = tid; g0 < ng; g0 += kDecUnroll * nth) {
        if (FMT == LHS_WIRE_F16) {
            uint2 w[kDecUnroll];
#pragma unroll
            for (int u = 0; u < kDecUnroll; ++u) {
                const int64_t g = g0 + u * nth;
                if (g < ng) w[u] = ld_dep(reinterpret_cast<const uint2 *>(pay) + g);
            }
#pragma unroll
            for (int u = 0; u < kDecUnroll; ++u) {
                const int64_t g = g0 + u * nth;
                if (g >= ng) break;
                const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w[u].x));
                const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w[u].y));
                reinterpret_cast<float4 *>(x)[g] = make_float4(a.x, a.y, b.x, b.y);
            }
        } else {
            float4 w[kDecUnroll];
#pragma unroll
            for (int u = 0; u < kDecUnroll; ++u) {
                const int64_t g = g0 + u * nth;
                if (g < ng) w[u] = ld_dep(reinterpret_cast<const float4 *>(pay) + g);
            }
#pragma unroll
            for (int u = 0; u < kDecUnroll; ++u) {
                const int64_t g = g0 + u * nth;
                if (g >= ng) break;
                reinterpret_cast<float4 *>(x)[g] = w[u];
            }
        }
    }
    for (int64_t i = ng * 4 + tid; i < n; i += nth) {
        if (FMT == LHS_WIRE_F16)
            x[i] = __half2float(__ushort_as_half(ld_dep(reinterpret_cast<const unsigned short *>(pay) + i)));
        else
            x[i] = ld_dep(reinterpret_cast<const float *>(pay) + i);
    }
}

// ---- i8 encode -------------------------------------------------------------
// i8 encode, any alignment or hidden: one CTA per position, element by element.
template <int XDT>
__global__ void __launch_bounds__(kI8Threads)
    encode_i8_kernel(const void *__restrict__ x, int32_t seq_len, int32_t hidden, WireHdr hdr,
                     uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sm_m[kI8Threads / 32];
    __shared__ int sm_f[kI8Threads / 32];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < seq_len; p += gridDim.x) {
        uint8_t *pos = buf + 4 * hdr.n + p * stride;
        const int64_t xrow = p * static_cast<int64_t>(hidden);
        float m = 0.0f;
        int nonfinite = 0;
        for (int j = threadIdx.x; j < hidden; j += kI8Threads) {
            const float v = load_x<XDT>(x, xrow + j);
            if (!isfinite(v)) nonfinite = 1;
            else m = fmaxf(m, fabsf(v));
        }
        block_max_or(m, nonfinite, sm_m, sm_f);
        const float scale = nonfinite ? 0.0f : __fdiv_rn(m, 127.0f);
        const float rcp = __frcp_rn(scale);
        if (threadIdx.x == 0) {
            const uint32_t sb = __float_as_uint(scale);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pos[i] = static_cast<uint8_t>(sb >> (8 * i));
                pos[4 + i] = 0;
            }
            if (nonfinite) set_err(err, LHS_ERRBIT_NONFINITE);
        }
        for (int j = threadIdx.x; j < hidden; j += kI8Threads)
            pos[8 + j] = static_cast<uint8_t>(i8_code(load_x<XDT>(x, xrow + j), scale, rcp));
    }
}

// i8 encode of long 16-byte-aligned rows (hidden % 8 == 0, hidden > 1024):
// one CTA per position, up to kI8Cache 8-value groups per thread held in
// registers between the block max-reduce and the quantisation.
template <int XDT>
__global__ void __launch_bounds__(kI8Threads)
    encode_i8_cta_kernel(const void *__restrict__ x, int32_t seq_len, int32_t hidden, WireHdr hdr,
                         uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sm_m[kI8Threads / 32];
    __shared__ int sm_f[kI8Threads / 32];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < seq_len; p += gridDim.x) {
        uint8_t *pos = buf + 4 * hdr.n + p * stride;
        const int64_t xrow = p * static_cast<int64_t>(hidden);
        float m = 0.0f;
        int nonfinite = 0;
        const int ng = hidden >> 3;
        const void *xp = XDT == LHS_F32
                             ? static_cast<const void *>(static_cast<const float *>(x) + xrow)
                             : static_cast<const void *>(static_cast<const unsigned short *>(x) + xrow);
        float cache[kI8Cache][8];
#pragma unroll
        for (int c = 0; c < kI8Cache; ++c) {
            const int g = threadIdx.x + c * kI8Threads;
            if (g < ng) {
                load_x8<XDT>(xp, g, cache[c]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (!isfinite(cache[c][i])) nonfinite = 1;
                    else m = fmaxf(m, fabsf(cache[c][i]));
                }
            }
        }
        for (int g = threadIdx.x + kI8Cache * kI8Threads; g < ng; g += kI8Threads) {
            float v[8];
            load_x8<XDT>(xp, g, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (!isfinite(v[i])) nonfinite = 1;
                else m = fmaxf(m, fabsf(v[i]));
            }
        }
        block_max_or(m, nonfinite, sm_m, sm_f);
        const float scale = nonfinite ? 0.0f : __fdiv_rn(m, 127.0f);
        const float rcp = __frcp_rn(scale);
        if (threadIdx.x == 0) {
            *reinterpret_cast<uint2 *>(pos) = make_uint2(__float_as_uint(scale), 0u);
            if (nonfinite) set_err(err, LHS_ERRBIT_NONFINITE);
        }
        uint2 *codes = reinterpret_cast<uint2 *>(pos + 8);
#pragma unroll
        for (int c = 0; c < kI8Cache; ++c) {
            const int g = threadIdx.x + c * kI8Threads;
            if (g < ng) {
                codes[g] = i8_code8(cache[c], scale, rcp);
            }
        }
        for (int g = threadIdx.x + kI8Cache * kI8Threads; g < ng; g += kI8Threads) {
            float v[8];
            load_x8<XDT>(xp, g, v);
            codes[g] = i8_code8(v, scale, rcp);
        }
    }
}

// i8 encode of long rows staged in shared memory: each CTA walks positions
// blockIdx.x, + gridDim.x, ...; one thread keeps the next kI8Bufs - 1
// positions' rows in flight (cp.async.bulk into a ring of kI8Bufs row
// buffers) while the CTA quantises the current one from shared memory —
// max|x| block-reduced, then 8 codes per thread step.  Two barriers per
// position: the one that makes the row visible to every thread (and frees
// the previous position's buffer for the next copy), and the max
// reduction's, whose per-warp slots alternate between two sets.  Rows of
// hidden values (f32 or bf16) at 16-byte aligned addresses, hidden % 8 == 0.
constexpr int kI8BulkThreads = 256;
constexpr int kI8Bufs = 2;
constexpr int64_t kI8BulkMaxSmem = 200 * 1024;  // kI8Bufs rows: f32 rows up to 25,600 values

template <int XDT>
__global__ void __launch_bounds__(kI8BulkThreads)
    encode_i8_bulk_kernel(const void *__restrict__ x, int32_t seq_len, int32_t hidden, WireHdr hdr,
                          uint8_t *__restrict__ buf, int32_t *err) {
    extern __shared__ __align__(128) uint8_t rows[];  // [kI8Bufs][row bytes]
    __shared__ uint64_t bar[kI8Bufs];
    __shared__ float sm_m[2][kI8BulkThreads / 32];
    __shared__ int sm_f[2][kI8BulkThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rb = static_cast<uint32_t>(hidden) * (XDT == LHS_F32 ? 4u : 2u);
    const uint8_t *xb = static_cast<const uint8_t *>(x);
    pdl_trigger();
    if (tid == 0) {
        for (int b = 0; b < kI8Bufs; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    if (blockIdx.x == 0 && tid == 0) write_hdr(buf, hdr);
    // thread 0: copy of the CTA's j-th position into buffer j % kI8Bufs
    int64_t issued = 0;
    auto issue = [&](int64_t j) {
        const int64_t p = blockIdx.x + j * gridDim.x;
        if (p >= seq_len) return;
        const int b = static_cast<int>(j % kI8Bufs);
        mbar_arrive_expect_tx(&bar[b], rb);
        bulk_load(rows + b * rb, xb + p * rb, rb, &bar[b]);
        issued = j + 1;
    };
    if (tid == 0)
        for (int j = 0; j < kI8Bufs - 1; ++j) issue(j);
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    const int n4 = hidden >> 2, ng = hidden >> 3;
    int64_t it = 0;
    for (int64_t p = blockIdx.x; p < seq_len; p += gridDim.x, ++it) {
        const int cur = static_cast<int>(it % kI8Bufs);
        const uint8_t *row = rows + cur * rb;
        const bool here = mbar_wait(&bar[cur], static_cast<uint32_t>(it / kI8Bufs) & 1, kWaitTimeoutNs);
        // every thread is past the previous position: its buffer takes the
        // copy kI8Bufs - 1 positions ahead
        if (!__syncthreads_and(here)) {
            if (tid == 0) set_err(err, LHS_ERRBIT_TIMEOUT);
            break;
        }
        if (tid == 0) issue(it + kI8Bufs - 1);
        // max|x| (fmaxf passes over NaN) and 0 * x summed: NaN exactly when
        // some x is inf or NaN
        float m = 0.0f, z = 0.0f;
        for (int i = tid; i < n4; i += kI8BulkThreads) {
            float v[4];
            if (XDT == LHS_F32) {
                const float4 f = reinterpret_cast<const float4 *>(row)[i];
                v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
            } else {
                const uint2 w = reinterpret_cast<const uint2 *>(row)[i];
                v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
                v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                m = fmaxf(m, fabsf(v[j]));
                z = __fmaf_rn(v[j], 0.0f, z);
            }
        }
        int nonfinite = z != z;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            nonfinite |= __shfl_xor_sync(0xFFFFFFFFu, nonfinite, o);
        }
        const int slot = static_cast<int>(it & 1);  // read by every thread before the next position's barrier
        if (lane == 0) {
            sm_m[slot][warp] = m;
            sm_f[slot][warp] = nonfinite;
        }
        __syncthreads();
#pragma unroll
        for (int w = 0; w < kI8BulkThreads / 32; ++w) {
            m = fmaxf(m, sm_m[slot][w]);
            nonfinite |= sm_f[slot][w];
        }
        const float scale = nonfinite ? 0.0f : __fdiv_rn(m, 127.0f);
        const float rcp = __frcp_rn(scale);
        uint8_t *pos = buf + 4 * hdr.n + p * stride;
        if (tid == 0) {
            *reinterpret_cast<uint2 *>(pos) = make_uint2(__float_as_uint(scale), 0u);
            if (nonfinite) set_err(err, LHS_ERRBIT_NONFINITE);
        }
        uint2 *codes = reinterpret_cast<uint2 *>(pos + 8);
        for (int g = tid; g < ng; g += kI8BulkThreads) {
            float v[8];
            if (XDT == LHS_F32) {
                const float4 a = reinterpret_cast<const float4 *>(row)[2 * g];
                const float4 b = reinterpret_cast<const float4 *>(row)[2 * g + 1];
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            } else {
                const uint4 w = reinterpret_cast<const uint4 *>(row)[g];
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[2 * j] = __uint_as_float(u[j] << 16);
                    v[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
                }
            }
            codes[g] = i8_code8(v, scale, rcp);
        }
    }
    // copies still headed for this CTA (after a timeout) land before it exits
    if (tid == 0)
        for (int64_t j = it; j < issued; ++j)
            if (!mbar_wait(&bar[j % kI8Bufs], static_cast<uint32_t>(j / kI8Bufs) & 1, kWaitTimeoutNs)) break;
}

// i8 encode with 16-byte-aligned rows (hidden % 8 == 0): one warp per
// position, two passes (i8_position_warp).
template <int XDT>
__global__ void __launch_bounds__(128)
    encode_i8_warp_kernel(const void *__restrict__ x, int32_t seq_len, int32_t hidden, WireHdr hdr,
                          uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    const int n4 = hidden >> 2;  // hidden <= 32 * kI8WarpSteps * 4
    for (int64_t p = w0; p < seq_len; p += nw) {
        const int64_t xrow = p * static_cast<int64_t>(hidden);
        i8_position_warp4(
            [&](int st, float (&v)[4]) {
                if (XDT == LHS_F32) {
                    const float4 a = ld_dep(reinterpret_cast<const float4 *>(static_cast<const float *>(x) + xrow) + st);
                    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                } else {
                    const uint2 w = ld_dep(reinterpret_cast<const uint2 *>(static_cast<const unsigned short *>(x) + xrow) + st);
                    v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
                    v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
                }
            },
            n4, buf + 4 * hdr.n + p * stride, lane, err);
    }
}

// ---- i8 decode -------------------------------------------------------------
template <bool VEC>
__global__ void __launch_bounds__(kI8Threads)
    decode_i8_kernel(const uint8_t *__restrict__ buf, int hoff, int32_t seq_len, int32_t hidden,
                     float *__restrict__ x, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    const uint32_t hdr_seq = ld_dep(reinterpret_cast<const uint32_t *>(buf) + 1);
    if (hdr_seq != static_cast<uint32_t>(seq_len)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_err(err, LHS_ERRBIT_MALFORMED);
        return;
    }
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < seq_len; p += gridDim.x) {
        const uint8_t *pos = buf + hoff + p * stride;
        float scale, zp;
        uint32_t pre[VEC ? kI8DecCache : 1];
        if (VEC) {
#pragma unroll
            for (int c = 0; c < kI8DecCache; ++c) {
                const int g = threadIdx.x + c * kI8Threads;
                if (g < (hidden >> 2)) pre[c] = ld_dep(reinterpret_cast<const uint32_t *>(pos + 8) + g);
            }
            const uint2 h = ld_dep(reinterpret_cast<const uint2 *>(pos));
            scale = __uint_as_float(h.x);
            zp = __uint_as_float(h.y);
        } else {
            uint32_t s = 0, z = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s |= static_cast<uint32_t>(ld_dep(pos + i)) << (8 * i);
                z |= static_cast<uint32_t>(ld_dep(pos + 4 + i)) << (8 * i);
            }
            scale = __uint_as_float(s);
            zp = __uint_as_float(z);
        }
        if (zp != 0.0f) {
            if (threadIdx.x == 0) set_err(err, LHS_ERRBIT_MALFORMED);
            continue;
        }
        float *xo = x + p * static_cast<int64_t>(hidden);
        if (VEC) {
            // 4 codes -> 4 values per unit: a warp's stores are 512
            // contiguous bytes (whole 32-byte sectors)
            const uint32_t *codes = reinterpret_cast<const uint32_t *>(pos + 8);
            float4 *o = reinterpret_cast<float4 *>(xo);
            const int ng = hidden >> 2;
            auto put = [&](int g, uint32_t w) {
                o[g] = make_float4(__fmul_rn(static_cast<float>(static_cast<int8_t>(w)), scale),
                                   __fmul_rn(static_cast<float>(static_cast<int8_t>(w >> 8)), scale),
                                   __fmul_rn(static_cast<float>(static_cast<int8_t>(w >> 16)), scale),
                                   __fmul_rn(static_cast<float>(static_cast<int8_t>(w >> 24)), scale));
            };
            // the first kI8DecCache units of this thread were loaded with
            // the header, before its scale is known
#pragma unroll
            for (int c = 0; c < kI8DecCache; ++c) {
                const int g = threadIdx.x + c * kI8Threads;
                if (g < ng) put(g, pre[c]);
            }
            for (int g = threadIdx.x + kI8DecCache * kI8Threads; g < ng; g += kI8Threads) put(g, ld_dep(codes + g));
        } else {
            for (int j = threadIdx.x; j < hidden; j += kI8Threads)
                xo[j] = __fmul_rn(static_cast<float>(static_cast<int8_t>(ld_dep(pos + 8 + j))), scale);
        }
    }
}

int ew_grid(int64_t work_items, int num_sms) {
    const int64_t need = (work_items + kEwThreads - 1) / kEwThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    const int64_t g = need < cap ? need : cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

// CTAs of 128 threads (no dynamic shared memory) of `kernel` resident on one
// SM, cached per kernel and device.
int resident_ctas_128(const void *kernel, int device) {
    struct Entry {
        const void *k;
        int device, n;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].k == kernel && cache[i].device == device) return cache[i].n;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 128, 0) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    if (used < 64) cache[used++] = Entry{kernel, device, n};
    return n;
}

cudaError_t launch_wire_encode(int fmt, const void *x, int x_dtype, int32_t seq_len,
                               int32_t hidden, const WireHdr &hdr, void *buf, int32_t *err,
                               cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    uint8_t *b = static_cast<uint8_t *>(buf);
    const int64_t n = static_cast<int64_t>(seq_len) * hidden;
    // the vector paths need the payload (and x) on 16-byte boundaries
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(b + 4 * hdr.n)) % 16) == 0;
    const int64_t i8_row = static_cast<int64_t>(hidden) * (x_dtype == LHS_F32 ? 4 : 2);
    if (fmt == LHS_WIRE_I8 && aligned && hidden % 8 == 0 && hidden > 1024 && kI8Bufs * i8_row <= kI8BulkMaxSmem) {
        // rows staged in shared memory, kI8Bufs per CTA; as many CTAs per SM
        // as the shared memory holds, at most 8
        const size_t smem = static_cast<size_t>(kI8Bufs * i8_row);
        auto kern = x_dtype == LHS_F32 ? encode_i8_bulk_kernel<LHS_F32> : encode_i8_bulk_kernel<LHS_BF16>;
        {
            // the largest size this kernel is launched with, once per device
            // and instantiation (static shared memory comes on top of it)
            static std::mutex mu;
            static bool done[2][64] = {};
            std::lock_guard<std::mutex> lock(mu);
            bool &d = done[x_dtype == LHS_F32 ? 0 : 1][dev.device];
            if (!d) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kI8BulkMaxSmem));
                if (e != cudaSuccess) return e;
                d = true;
            }
        }
        int64_t per_sm = (200 * 1024) / static_cast<int64_t>(smem + 1024);
        if (per_sm > 8) per_sm = 8;
        if (per_sm < 1) per_sm = 1;
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * per_sm;
        const int grid = static_cast<int>(seq_len < 1 ? 1 : (seq_len < cap ? seq_len : cap));
        return launch_pdl(kern, dim3(grid), dim3(kI8BulkThreads), smem, stream, x, seq_len, hidden, hdr, b, err);
    }
    if (fmt == LHS_WIRE_I8 && aligned && hidden % 8 == 0 && hidden > 1024) {
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
        const int grid = static_cast<int>(seq_len < 1 ? 1 : (seq_len < cap ? seq_len : cap));
        auto kern = x_dtype == LHS_F32 ? encode_i8_cta_kernel<LHS_F32> : encode_i8_cta_kernel<LHS_BF16>;
        return launch_pdl(kern, dim3(grid), dim3(kI8Threads), 0, stream, x, seq_len, hidden, hdr, b, err);
    }
    if (fmt == LHS_WIRE_I8 && aligned && hidden % 8 == 0) {
        const int wps = i8_warps_per_sm(static_cast<int64_t>(hidden) * (x_dtype == LHS_F32 ? 4 : 2));
        auto kern = x_dtype == LHS_F32 ? encode_i8_warp_kernel<LHS_F32> : encode_i8_warp_kernel<LHS_BF16>;
        const int grid = warp_kernel_grid(kern, seq_len, wps, dev.num_sms, dev.device);
        return launch_pdl(kern, dim3(grid), dim3(128), 0, stream, x, seq_len, hidden, hdr, b, err);
    }
    if (fmt == LHS_WIRE_I8) {
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
        int grid = static_cast<int>(seq_len < cap ? seq_len : cap);
        if (grid < 1) grid = 1;
        auto kern = x_dtype == LHS_F32 ? encode_i8_kernel<LHS_F32> : encode_i8_kernel<LHS_BF16>;
        return launch_pdl(kern, dim3(grid), dim3(kI8Threads), 0, stream, x, seq_len, hidden, hdr, b, err);
    }
    const bool vec = aligned;
    const int grid = ew_grid(vec ? (n + 7) / 8 : n, dev.num_sms);
    void (*kern)(const void *, int64_t, WireHdr, uint8_t *);
    if (fmt == LHS_WIRE_F16) {
        if (x_dtype == LHS_F32) kern = vec ? encode_ew_kernel<LHS_WIRE_F16, LHS_F32, true> : encode_ew_kernel<LHS_WIRE_F16, LHS_F32, false>;
        else kern = vec ? encode_ew_kernel<LHS_WIRE_F16, LHS_BF16, true> : encode_ew_kernel<LHS_WIRE_F16, LHS_BF16, false>;
    } else {
        if (x_dtype == LHS_F32) kern = vec ? encode_ew_kernel<LHS_WIRE_F32, LHS_F32, true> : encode_ew_kernel<LHS_WIRE_F32, LHS_F32, false>;
        else kern = vec ? encode_ew_kernel<LHS_WIRE_F32, LHS_BF16, true> : encode_ew_kernel<LHS_WIRE_F32, LHS_BF16, false>;
    }
    return launch_pdl(kern, dim3(grid), dim3(kEwThreads), 0, stream, x, n, hdr, b);
}

cudaError_t launch_wire_decode(int fmt, const void *buf, int hoff, int32_t seq_len, int32_t hidden,
                               float *x, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    const uint8_t *b = static_cast<const uint8_t *>(buf);
    const int64_t n = static_cast<int64_t>(seq_len) * hidden;
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(b + hoff)) % 16) == 0;
    if (fmt == LHS_WIRE_I8) {
        const bool vec = aligned && (hidden % 8 == 0);
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
        int grid = static_cast<int>(seq_len < cap ? seq_len : cap);
        if (grid < 1) grid = 1;
        return launch_pdl(vec ? decode_i8_kernel<true> : decode_i8_kernel<false>, dim3(grid),
                          dim3(kI8Threads), 0, stream, b, hoff, seq_len, hidden, x, err);
    }
    const int grid = ew_grid(aligned ? (n + 3) / 4 : n, dev.num_sms);
    const uint32_t s = static_cast<uint32_t>(seq_len);
    void (*kern)(const uint8_t *, int, int64_t, uint32_t, float *, int32_t *);
    if (fmt == LHS_WIRE_F16) kern = aligned ? decode_ew_kernel<LHS_WIRE_F16, true> : decode_ew_kernel<LHS_WIRE_F16, false>;
    else kern = aligned ? decode_ew_kernel<LHS_WIRE_F32, true> : decode_ew_kernel<LHS_WIRE_F32, false>;
    return launch_pdl(kern, dim3(grid), dim3(kEwThreads), 0, stream, b, hoff, n, s, x, err);
}

}  // namespace lhs
