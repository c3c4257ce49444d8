// embed_wire.cu — the embed lookup written straight into a wire message.
//
// ADR-0008 "Remote Embeddings and lm_head Service", POST /v1/embed: the
// response carries the looked-up rows in "the same codec as FFN grid";
// ADR-0009 "Wire Format Evolution", Wire Layout: a 16-byte header, then an
// f32, f16 or per-position i8 payload.  lhs_embed_wire produces, byte for
// byte, lhs_wire_encode(fmt, lhs_embed(ids, scale)) without the binary32
// intermediate: the gather's cost is its output write, which the f16 payload
// halves and the i8 payload cuts to (hidden + 8) / (4 hidden).
//
// f32 / f16: one warp per token, 8 elements per lane step (16-byte loads and
// stores).  i8: one warp per token — max|x| of the scaled row, then the
// codes (the same steps, in the same binary32 operations, as the i8
// encoder); rows up to 1024 values stay in registers between the two,
// longer rows are read a second time.
#include "lhs_internal.cuh"

namespace lhs {
namespace {

constexpr int kWarps = 8;
constexpr int kI8Threads = 128;

__device__ __forceinline__ bool bad_id(int32_t id, int64_t vocab) {
    return id < 0 || static_cast<int64_t>(id) >= vocab;
}

template <int DT, int FMT, bool VEC>
__global__ void __launch_bounds__(kWarps * 32)
    embed_wire_ew_kernel(const uint8_t *__restrict__ table, int64_t vocab, int hidden, int64_t row_bytes,
                         const int32_t *__restrict__ ids, int64_t n, float scale, uint32_t layer,
                         uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_wire_header(buf, layer, static_cast<uint32_t>(n), flags, top_k);
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    uint8_t *pay = buf + 16;
    for (int64_t t = warp0; t < n; t += nwarps) {
        const int32_t id = ld_dep(ids + t);
        const bool bad = bad_id(id, vocab);
        if (bad && lane == 0) set_err(err, LHS_ERRBIT_BAD_TOKEN);
        const uint8_t *row = table + static_cast<int64_t>(bad ? 0 : id) * row_bytes;
        if (VEC && FMT == LHS_WIRE_F32) {
            // 4 values per lane step: a warp's stores are whole 32-byte sectors
            const int n4 = hidden >> 2;
            for (int s4 = lane; s4 < n4; s4 += 32) {
                float v[4];
                if (bad) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = 0.0f;
                } else {
                    row_elements4<DT>(row, s4, v);
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = __fmul_rn(v[i], scale);
                }
                reinterpret_cast<float4 *>(pay)[t * n4 + s4] = make_float4(v[0], v[1], v[2], v[3]);
            }
        } else if (VEC) {
            const int ng = hidden >> 3;
            for (int g = lane; g < ng; g += 32) {
                float v[8];
                if (bad) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = 0.0f;
                } else {
                    row_elements8<DT>(row, g, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], scale);
                }
                reinterpret_cast<uint4 *>(pay)[t * ng + g] = pack_f16x8(v);
            }
        } else {
            for (int j = lane; j < hidden; j += 32) {
                const float v = bad ? 0.0f : __fmul_rn(row_element<DT>(row, j), scale);
                const int64_t o = t * hidden + j;
                if (FMT == LHS_WIRE_F32) reinterpret_cast<float *>(pay)[o] = v;
                else reinterpret_cast<unsigned short *>(pay)[o] = static_cast<unsigned short>(f16_sat_bits(v));
            }
        }
    }
}

// i8, any hidden or row alignment: one CTA per token, element by element.
template <int DT>
__global__ void __launch_bounds__(kI8Threads)
    embed_wire_i8_kernel(const uint8_t *__restrict__ table, int64_t vocab, int hidden, int64_t row_bytes,
                         const int32_t *__restrict__ ids, int64_t n, float scale, uint32_t layer,
                         uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sm_m[kI8Threads / 32];
    __shared__ int sm_f[kI8Threads / 32];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_wire_header(buf, layer, static_cast<uint32_t>(n), flags, top_k);
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < n; p += gridDim.x) {
        const int32_t id = ld_dep(ids + p);
        const bool bad = bad_id(id, vocab);  // uniform over the block
        if (bad && threadIdx.x == 0) set_err(err, LHS_ERRBIT_BAD_TOKEN);
        const uint8_t *row = table + static_cast<int64_t>(bad ? 0 : id) * row_bytes;
        uint8_t *pos = buf + 16 + p * stride;
        auto value = [&](int j) { return bad ? 0.0f : __fmul_rn(row_element<DT>(row, j), scale); };
        float m = 0.0f;
        int nonfinite = 0;
        for (int j = threadIdx.x; j < hidden; j += kI8Threads) {
            const float v = value(j);
            if (!isfinite(v)) nonfinite = 1;
            else m = fmaxf(m, fabsf(v));
        }
        block_max_or(m, nonfinite, sm_m, sm_f);
        const float qs = nonfinite ? 0.0f : __fdiv_rn(m, 127.0f);
        const float rcp = __frcp_rn(qs);
        if (threadIdx.x == 0) {
            const uint32_t sb = __float_as_uint(qs);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pos[i] = static_cast<uint8_t>(sb >> (8 * i));
                pos[4 + i] = 0;
            }
            if (nonfinite) set_err(err, LHS_ERRBIT_NONFINITE);
        }
        for (int j = threadIdx.x; j < hidden; j += kI8Threads)
            pos[8 + j] = static_cast<uint8_t>(i8_code(value(j), qs, rcp));
    }
}

// i8 with 8-element steps: one warp per token, two passes over the row.
template <int DT>
__global__ void __launch_bounds__(128)
    embed_wire_i8_warp_kernel(const uint8_t *__restrict__ table, int64_t vocab, int hidden, int64_t row_bytes,
                              const int32_t *__restrict__ ids, int64_t n, float scale, uint32_t layer,
                              uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_wire_header(buf, layer, static_cast<uint32_t>(n), flags, top_k);
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    const int ng = hidden >> 3;
    for (int64_t p = w0; p < n; p += nw) {
        const int32_t id = ld_dep(ids + p);
        const bool bad = bad_id(id, vocab);
        if (bad && lane == 0) set_err(err, LHS_ERRBIT_BAD_TOKEN);
        const uint8_t *row = table + static_cast<int64_t>(bad ? 0 : id) * row_bytes;
        i8_position_warp(
            [&](int g, float (&v)[8]) {
                if (bad) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = 0.0f;
                } else {
                    row_elements8<DT>(row, g, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], scale);
                }
            },
            ng, buf + 16 + p * stride, lane, err);
    }
}

// i8 with rows of at most 1024 values: one warp per token, the scaled row in
// registers between the max and the codes.
template <int DT>
__global__ void __launch_bounds__(128)
    embed_wire_i8_warp4_kernel(const uint8_t *__restrict__ table, int64_t vocab, int hidden, int64_t row_bytes,
                               const int32_t *__restrict__ ids, int64_t n, float scale, uint32_t layer,
                               uint32_t flags, uint32_t top_k, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_wire_header(buf, layer, static_cast<uint32_t>(n), flags, top_k);
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    const int n4 = hidden >> 2;
    for (int64_t p = w0; p < n; p += nw) {
        const int32_t id = ld_dep(ids + p);
        const bool bad = bad_id(id, vocab);
        if (bad && lane == 0) set_err(err, LHS_ERRBIT_BAD_TOKEN);
        const uint8_t *row = table + static_cast<int64_t>(bad ? 0 : id) * row_bytes;
        i8_position_warp4(
            [&](int st, float (&v)[4]) {
                if (bad) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = 0.0f;
                } else {
                    row_elements4<DT>(row, st, v);
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = __fmul_rn(v[i], scale);
                }
            },
            n4, buf + 16 + p * stride, lane, err);
    }
}

template <int DT>
cudaError_t launch_dt(const lhs_table &t, const int32_t *ids, int64_t n, float scale, int fmt,
                      uint32_t layer, uint32_t flags, uint32_t top_k, uint8_t *buf, int32_t *err,
                      cudaStream_t stream, int num_sms, int device) {
    const uint8_t *tb = static_cast<const uint8_t *>(t.data);
    // 8-element steps: rows 16-byte aligned (Q8_0: 2-byte) and hidden % 8 == 0
    bool vec = t.hidden % 8 == 0;
    if (DT != LHS_Q8_0) vec = vec && (reinterpret_cast<uintptr_t>(t.data) % 16 == 0) && (t.row_bytes % 16 == 0);
    if (fmt == LHS_WIRE_I8 && vec && t.hidden <= 32 * kI8WarpSteps * 4) {
        const int wps = i8_warps_per_sm(t.row_bytes);
        const int grid = warp_kernel_grid(embed_wire_i8_warp4_kernel<DT>, n, wps, num_sms, device);
        return launch_pdl(embed_wire_i8_warp4_kernel<DT>, dim3(grid), dim3(128), 0, stream, tb, t.vocab, t.hidden,
                          t.row_bytes, ids, n, scale, layer, flags, top_k, buf, err);
    }
    if (fmt == LHS_WIRE_I8 && vec) {
        const int wps = i8_warps_per_sm(t.row_bytes);
        const int grid = warp_kernel_grid(embed_wire_i8_warp_kernel<DT>, n, wps, num_sms, device);
        return launch_pdl(embed_wire_i8_warp_kernel<DT>, dim3(grid), dim3(128), 0, stream, tb, t.vocab, t.hidden,
                          t.row_bytes, ids, n, scale, layer, flags, top_k, buf, err);
    }
    if (fmt == LHS_WIRE_I8) {
        const int64_t cap = static_cast<int64_t>(num_sms) * 16;
        const int grid = static_cast<int>(n < 1 ? 1 : (n < cap ? n : cap));
        return launch_pdl(embed_wire_i8_kernel<DT>, dim3(grid),
                          dim3(kI8Threads), 0, stream, tb, t.vocab, t.hidden, t.row_bytes, ids, n, scale,
                          layer, flags, top_k, buf, err);
    }
    const int64_t blocks_needed = (n + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(num_sms) * 32;
    const int grid = static_cast<int>(blocks_needed < 1 ? 1 : (blocks_needed < cap ? blocks_needed : cap));
    auto k = fmt == LHS_WIRE_F16
                 ? (vec ? embed_wire_ew_kernel<DT, LHS_WIRE_F16, true> : embed_wire_ew_kernel<DT, LHS_WIRE_F16, false>)
                 : (vec ? embed_wire_ew_kernel<DT, LHS_WIRE_F32, true> : embed_wire_ew_kernel<DT, LHS_WIRE_F32, false>);
    return launch_pdl(k, dim3(grid), dim3(kWarps * 32), 0, stream, tb, t.vocab, t.hidden, t.row_bytes, ids,
                      n, scale, layer, flags, top_k, buf, err);
}

}  // namespace

cudaError_t launch_embed_wire(const lhs_table &t, const int32_t *ids, int64_t n, float scale, int fmt,
                              uint32_t layer, uint32_t flags, uint32_t top_k, void *buf, int32_t *err,
                              cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    uint8_t *b = static_cast<uint8_t *>(buf);
    switch (t.dtype) {
    case LHS_F32: return launch_dt<LHS_F32>(t, ids, n, scale, fmt, layer, flags, top_k, b, err, stream,
                                                   dev.num_sms, dev.device);
    case LHS_F16: return launch_dt<LHS_F16>(t, ids, n, scale, fmt, layer, flags, top_k, b, err, stream,
                                                   dev.num_sms, dev.device);
    case LHS_BF16: return launch_dt<LHS_BF16>(t, ids, n, scale, fmt, layer, flags, top_k, b, err, stream,
                                                   dev.num_sms, dev.device);
    default: return launch_dt<LHS_Q8_0>(t, ids, n, scale, fmt, layer, flags, top_k, b, err, stream,
                                                   dev.num_sms, dev.device);
    }
}

}  // namespace lhs
