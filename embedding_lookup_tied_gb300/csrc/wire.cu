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
// i8: one warp per position for rows up to 1024 values, one CTA per position
// for longer or unaligned rows —
// max-reduce of |x|, one correctly rounded divide for the scale, then
// round-half-even of the binary32 quotient x/scale for every element.
// Positions start at 16 + p*(hidden+8): 8-byte aligned when hidden % 8 == 0,
// so the codes move as 8-byte words.
#include <cuda_fp16.h>

#include "lhs_internal.cuh"

namespace lhs {
namespace {

constexpr int kEwThreads = 256;
constexpr int kI8Threads = 128;
constexpr int kI8Cache = 6;  // 8-value groups a thread keeps in registers (CTA path)

template <int XDT>
__device__ __forceinline__ float load_x(const void *x, int64_t i) {
    if (XDT == LHS_F32) return __ldg(static_cast<const float *>(x) + i);
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short *>(x) + i))
                           << 16);
}

// 8 consecutive values starting at element 8*g (16-byte aligned source).
template <int XDT>
__device__ __forceinline__ void load_x8(const void *x, int64_t g, float (&v)[8]) {
    if (XDT == LHS_F32) {
        const float4 *p = static_cast<const float4 *>(x) + 2 * g;
        const float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 w = __ldg(static_cast<const uint4 *>(x) + g);
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
    encode_ew_kernel(const void *__restrict__ x, int64_t n, uint32_t layer, uint32_t seq_len,
                     uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf) {
    pdl_trigger();
    pdl_wait();
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (tid == 0) write_wire_header(buf, layer, seq_len, flags, top_k);
    uint8_t *pay = buf + 16;
    const int64_t ng = VEC ? n / 8 : 0;
    for (int64_t g = tid; g < ng; g += nth) {
        float v[8];
        load_x8<XDT>(x, g, v);
        if (FMT == LHS_WIRE_F16) {
            reinterpret_cast<uint4 *>(pay)[g] = pack_f16x8(v);
        } else {
            float4 *p = reinterpret_cast<float4 *>(pay) + 2 * g;
            p[0] = make_float4(v[0], v[1], v[2], v[3]);
            p[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
    for (int64_t i = ng * 8 + tid; i < n; i += nth) {
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
    decode_ew_kernel(const uint8_t *__restrict__ buf, int64_t n, uint32_t seq_len,
                     float *__restrict__ x, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint32_t hdr_seq = __ldg(reinterpret_cast<const uint32_t *>(buf) + 1);
    if (hdr_seq != seq_len) {
        if (tid == 0) set_err(err, LHS_ERRBIT_MALFORMED);
        return;
    }
    const uint8_t *pay = buf + 16;
    const int64_t ng = VEC ? n / 8 : 0;
    for (int64_t g = tid; g < ng; g += nth) {
        float4 *o = reinterpret_cast<float4 *>(x) + 2 * g;
        if (FMT == LHS_WIRE_F16) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(pay) + g);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
            float v[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[i] & 0xFFFFu)));
                v[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(u[i] >> 16)));
            }
            o[0] = make_float4(v[0], v[1], v[2], v[3]);
            o[1] = make_float4(v[4], v[5], v[6], v[7]);
        } else {
            const float4 *p = reinterpret_cast<const float4 *>(pay) + 2 * g;
            o[0] = __ldg(p);
            o[1] = __ldg(p + 1);
        }
    }
    for (int64_t i = ng * 8 + tid; i < n; i += nth) {
        if (FMT == LHS_WIRE_F16)
            x[i] = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short *>(pay) + i)));
        else
            x[i] = __ldg(reinterpret_cast<const float *>(pay) + i);
    }
}

// ---- i8 encode -------------------------------------------------------------
// i8 encode, any alignment or hidden: one CTA per position, element by element.
template <int XDT>
__global__ void __launch_bounds__(kI8Threads)
    encode_i8_kernel(const void *__restrict__ x, int32_t seq_len, int32_t hidden, uint32_t layer,
                     uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sm_m[kI8Threads / 32];
    __shared__ int sm_f[kI8Threads / 32];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_wire_header(buf, layer, static_cast<uint32_t>(seq_len), flags, top_k);
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < seq_len; p += gridDim.x) {
        uint8_t *pos = buf + 16 + p * stride;
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
    encode_i8_cta_kernel(const void *__restrict__ x, int32_t seq_len, int32_t hidden, uint32_t layer,
                         uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sm_m[kI8Threads / 32];
    __shared__ int sm_f[kI8Threads / 32];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_wire_header(buf, layer, static_cast<uint32_t>(seq_len), flags, top_k);
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < seq_len; p += gridDim.x) {
        uint8_t *pos = buf + 16 + p * stride;
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
                uint32_t w0 = 0, w1 = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w0 |= (static_cast<uint32_t>(static_cast<uint8_t>(i8_code(cache[c][i], scale, rcp)))) << (8 * i);
                    w1 |= (static_cast<uint32_t>(static_cast<uint8_t>(i8_code(cache[c][i + 4], scale, rcp)))) << (8 * i);
                }
                codes[g] = make_uint2(w0, w1);
            }
        }
        for (int g = threadIdx.x + kI8Cache * kI8Threads; g < ng; g += kI8Threads) {
            float v[8];
            load_x8<XDT>(xp, g, v);
            uint32_t w0 = 0, w1 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w0 |= (static_cast<uint32_t>(static_cast<uint8_t>(i8_code(v[i], scale, rcp)))) << (8 * i);
                w1 |= (static_cast<uint32_t>(static_cast<uint8_t>(i8_code(v[i + 4], scale, rcp)))) << (8 * i);
            }
            codes[g] = make_uint2(w0, w1);
        }
    }
}

// i8 encode with 16-byte-aligned rows (hidden % 8 == 0): one warp per
// position, two passes (i8_position_warp).
template <int XDT>
__global__ void __launch_bounds__(128)
    encode_i8_warp_kernel(const void *__restrict__ x, int32_t seq_len, int32_t hidden, uint32_t layer,
                          uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_wire_header(buf, layer, static_cast<uint32_t>(seq_len), flags, top_k);
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    const int ng = hidden >> 3;
    for (int64_t p = w0; p < seq_len; p += nw) {
        const int64_t xrow = p * static_cast<int64_t>(hidden);
        const void *xp = XDT == LHS_F32 ? static_cast<const void *>(static_cast<const float *>(x) + xrow)
                                        : static_cast<const void *>(static_cast<const unsigned short *>(x) + xrow);
        i8_position_warp([&](int g, float (&v)[8]) { load_x8<XDT>(xp, g, v); }, ng, buf + 16 + p * stride,
                         lane, err);
    }
}

// ---- i8 decode -------------------------------------------------------------
template <bool VEC>
__global__ void __launch_bounds__(kI8Threads)
    decode_i8_kernel(const uint8_t *__restrict__ buf, int32_t seq_len, int32_t hidden,
                     float *__restrict__ x, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    const uint32_t hdr_seq = __ldg(reinterpret_cast<const uint32_t *>(buf) + 1);
    if (hdr_seq != static_cast<uint32_t>(seq_len)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_err(err, LHS_ERRBIT_MALFORMED);
        return;
    }
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < seq_len; p += gridDim.x) {
        const uint8_t *pos = buf + 16 + p * stride;
        float scale, zp;
        if (VEC) {
            const uint2 h = __ldg(reinterpret_cast<const uint2 *>(pos));
            scale = __uint_as_float(h.x);
            zp = __uint_as_float(h.y);
        } else {
            uint32_t s = 0, z = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s |= static_cast<uint32_t>(__ldg(pos + i)) << (8 * i);
                z |= static_cast<uint32_t>(__ldg(pos + 4 + i)) << (8 * i);
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
            const uint2 *codes = reinterpret_cast<const uint2 *>(pos + 8);
            float4 *o = reinterpret_cast<float4 *>(xo);
            for (int g = threadIdx.x; g < (hidden >> 3); g += kI8Threads) {
                const uint2 w = __ldg(codes + g);
                float v[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[i] = __fmul_rn(static_cast<float>(static_cast<int8_t>(w.x >> (8 * i))), scale);
                    v[4 + i] = __fmul_rn(static_cast<float>(static_cast<int8_t>(w.y >> (8 * i))), scale);
                }
                o[2 * g] = make_float4(v[0], v[1], v[2], v[3]);
                o[2 * g + 1] = make_float4(v[4], v[5], v[6], v[7]);
            }
        } else {
            for (int j = threadIdx.x; j < hidden; j += kI8Threads)
                xo[j] = __fmul_rn(static_cast<float>(static_cast<int8_t>(__ldg(pos + 8 + j))), scale);
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

cudaError_t launch_wire_encode(int fmt, const void *x, int x_dtype, int32_t seq_len,
                               int32_t hidden, uint32_t layer, uint32_t flags, uint32_t top_k,
                               void *buf, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    uint8_t *b = static_cast<uint8_t *>(buf);
    const int64_t n = static_cast<int64_t>(seq_len) * hidden;
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(buf)) % 16) == 0;
    const uint32_t s = static_cast<uint32_t>(seq_len);
    if (fmt == LHS_WIRE_I8 && aligned && hidden % 8 == 0 && hidden > 1024) {
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
        const int grid = static_cast<int>(seq_len < 1 ? 1 : (seq_len < cap ? seq_len : cap));
        auto kern = x_dtype == LHS_F32 ? encode_i8_cta_kernel<LHS_F32> : encode_i8_cta_kernel<LHS_BF16>;
        return launch_pdl(kern, dim3(grid), dim3(kI8Threads), 0, stream, x, seq_len, hidden, layer, flags, top_k,
                          b, err);
    }
    if (fmt == LHS_WIRE_I8 && aligned && hidden % 8 == 0) {
        const int wps = i8_warps_per_sm(static_cast<int64_t>(hidden) * (x_dtype == LHS_F32 ? 4 : 2));
        const int64_t warps = seq_len < static_cast<int64_t>(dev.num_sms) * wps ? seq_len
                                                                                  : static_cast<int64_t>(dev.num_sms) * wps;
        const int grid = static_cast<int>(warps < 4 ? 1 : (warps + 3) / 4);
        auto kern = x_dtype == LHS_F32 ? encode_i8_warp_kernel<LHS_F32> : encode_i8_warp_kernel<LHS_BF16>;
        return launch_pdl(kern, dim3(grid), dim3(128), 0, stream, x, seq_len, hidden, layer, flags, top_k, b,
                          err);
    }
    if (fmt == LHS_WIRE_I8) {
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
        int grid = static_cast<int>(seq_len < cap ? seq_len : cap);
        if (grid < 1) grid = 1;
        auto kern = x_dtype == LHS_F32 ? encode_i8_kernel<LHS_F32> : encode_i8_kernel<LHS_BF16>;
        return launch_pdl(kern, dim3(grid), dim3(kI8Threads), 0, stream, x, seq_len, hidden, layer,
                          flags, top_k, b, err);
    }
    const bool vec = aligned;
    const int grid = ew_grid(vec ? (n + 7) / 8 : n, dev.num_sms);
void (*kern)(const void *, int64_t, uint32_t, uint32_t, uint32_t, uint32_t, uint8_t *);
    if (fmt == LHS_WIRE_F16) {
        if (x_dtype == LHS_F32) kern = vec ? encode_ew_kernel<LHS_WIRE_F16, LHS_F32, true> : encode_ew_kernel<LHS_WIRE_F16, LHS_F32, false>;
        else kern = vec ? encode_ew_kernel<LHS_WIRE_F16, LHS_BF16, true> : encode_ew_kernel<LHS_WIRE_F16, LHS_BF16, false>;
    } else {
        if (x_dtype == LHS_F32) kern = vec ? encode_ew_kernel<LHS_WIRE_F32, LHS_F32, true> : encode_ew_kernel<LHS_WIRE_F32, LHS_F32, false>;
        else kern = vec ? encode_ew_kernel<LHS_WIRE_F32, LHS_BF16, true> : encode_ew_kernel<LHS_WIRE_F32, LHS_BF16, false>;
    }
    return launch_pdl(kern, dim3(grid), dim3(kEwThreads), 0, stream, x, n, layer, s, flags, top_k, b);
}

cudaError_t launch_wire_decode(int fmt, const void *buf, int32_t seq_len, int32_t hidden,
                               float *x, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    const uint8_t *b = static_cast<const uint8_t *>(buf);
    const int64_t n = static_cast<int64_t>(seq_len) * hidden;
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(buf)) % 16) == 0;
    if (fmt == LHS_WIRE_I8) {
        const bool vec = aligned && (hidden % 8 == 0);
        const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
        int grid = static_cast<int>(seq_len < cap ? seq_len : cap);
        if (grid < 1) grid = 1;
        return launch_pdl(vec ? decode_i8_kernel<true> : decode_i8_kernel<false>, dim3(grid),
                          dim3(kI8Threads), 0, stream, b, seq_len, hidden, x, err);
    }
    const int grid = ew_grid(aligned ? (n + 7) / 8 : n, dev.num_sms);
    const uint32_t s = static_cast<uint32_t>(seq_len);
    void (*kern)(const uint8_t *, int64_t, uint32_t, float *, int32_t *);
    if (fmt == LHS_WIRE_F16) kern = aligned ? decode_ew_kernel<LHS_WIRE_F16, true> : decode_ew_kernel<LHS_WIRE_F16, false>;
    else kern = aligned ? decode_ew_kernel<LHS_WIRE_F32, true> : decode_ew_kernel<LHS_WIRE_F32, false>;
    return launch_pdl(kern, dim3(grid), dim3(kEwThreads), 0, stream, b, n, s, x, err);
}

}  // namespace lhs
