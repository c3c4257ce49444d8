// mixed.cu — gather from a table whose rows carry their own precision.
//
// HELIX "Columnar Embedding", §3: the row-aligned store needs a sidecar
// (embed-rows.idx) only when rows are heterogeneous — mixed precision per row
// (common tokens in fp16, the long Unicode tail in fp8) or quantised rows with
// their dequantisation header inline.  The sidecar gives, per row, its byte
// offset in the data and its element type: f32, f16, bf16, Q8_0 (inline d per
// 32 values) or OCP FP8 E4M3.
//
// One warp per token; the row type is uniform over the warp.  Element values
// widen exactly to binary32, then one multiply by the scale, as the
// homogeneous gather does.
#include "lhs_internal.cuh"

namespace lhs {
namespace {

// OCP FP8 E4M3 (bias 7, no infinities, S.1111.111 = NaN) -> binary32, exact:
// normal codes map to exponent e - 7 + 127 and fraction m << 20; subnormal
// codes are m * 2^-9.
__device__ __forceinline__ float fp8_e4m3_to_f32(uint32_t c) {
    const uint32_t s = (c & 0x80u) << 24, e = (c >> 3) & 0xFu, m = c & 0x7u;
    if (e == 0xFu && m == 0x7u) return __uint_as_float(s | 0x7FC00000u);
    if (e == 0u) return __uint_as_float(s | __float_as_uint(__fmul_rn(static_cast<float>(m), 0x1p-9f)));
    return __uint_as_float(s | ((e + 120u) << 23) | (m << 20));
}

__device__ __forceinline__ float mixed_element(const uint8_t *row, int dt, int j) {
    switch (dt) {
    case LHS_F32: return row_element<LHS_F32>(row, j);
    case LHS_F16: return row_element<LHS_F16>(row, j);
    case LHS_BF16: return row_element<LHS_BF16>(row, j);
    case LHS_Q8_0: return row_element<LHS_Q8_0>(row, j);
    default: return fp8_e4m3_to_f32(__ldg(row + j));
    }
}

// Bytes of a row of type dt, or -1 when dt is not a row type for this hidden.
__device__ __forceinline__ int64_t mixed_row_bytes(int dt, int hidden) {
    switch (dt) {
    case LHS_F32: return 4ll * hidden;
    case LHS_F16:
    case LHS_BF16: return 2ll * hidden;
    case LHS_Q8_0: return hidden % 32 == 0 ? static_cast<int64_t>(hidden / 32) * 34 : -1;
    case LHS_FP8_E4M3: return hidden;
    default: return -1;
    }
}

// A row is read only when its type is known, it is aligned for its element
// loads (4 bytes for f32, 2 for the 16-bit types and Q8_0) and it lies
// inside the data.
__device__ __forceinline__ bool row_ok(int dt, int hidden, int64_t off, int64_t data_bytes) {
    const int64_t rb = mixed_row_bytes(dt, hidden);
    if (rb < 0 || off < 0 || off > data_bytes - rb) return false;
    const int64_t align = dt == LHS_F32 ? 4 : (dt == LHS_FP8_E4M3 ? 1 : 2);
    return off % align == 0;
}

__global__ void __launch_bounds__(256)
    embed_mixed_kernel(const uint8_t *__restrict__ data, int64_t data_bytes, const int64_t *__restrict__ row_offset,
                       const uint8_t *__restrict__ row_dtype, int64_t vocab, int hidden,
                       const int32_t *__restrict__ ids, int64_t n, float scale, float *__restrict__ out,
                       int32_t *err) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = w0; t < n; t += nw) {
        const int32_t id = ld_dep(ids + t);
        float *o = out + t * hidden;
        if (id < 0 || static_cast<int64_t>(id) >= vocab) {
            for (int j = lane; j < hidden; j += 32) o[j] = 0.0f;
            if (lane == 0) set_err(err, LHS_ERRBIT_BAD_TOKEN);
            continue;
        }
        const int dt = __ldg(row_dtype + id);
        const int64_t off = __ldg(row_offset + id);
        if (!row_ok(dt, hidden, off, data_bytes)) {
            for (int j = lane; j < hidden; j += 32) o[j] = 0.0f;
            if (lane == 0) set_err(err, LHS_ERRBIT_MALFORMED);
            continue;
        }
        const uint8_t *row = data + off;
        for (int j = lane; j < hidden; j += 32) o[j] = __fmul_rn(mixed_element(row, dt, j), scale);
    }
}

}  // namespace

cudaError_t launch_embed_mixed(const void *data, int64_t data_bytes, const int64_t *row_offset, const uint8_t *row_dtype,
                               int64_t vocab, int32_t hidden, const int32_t *ids, int64_t n, float scale,
                               float *out, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    const int64_t need = (n + 7) / 8;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
    const int grid = static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
    return launch_pdl(embed_mixed_kernel, dim3(grid), dim3(256), 0, stream, static_cast<const uint8_t *>(data),
                      data_bytes, row_offset, row_dtype, vocab, hidden, ids, n, scale, out, err);
}

}  // namespace lhs
