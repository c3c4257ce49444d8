// gather.cu — step 1: embed row gather + dequant + scale.
//
// ADR-0008 "Remote Embeddings and lm_head Service", POST /v1/embed: one row
// lookup per token id, a prefill of n tokens is n independent lookups
// (Open Question 2).  HELIX "Columnar Embedding", §3: row i lives at byte
// offset i*row_bytes.  Port Specification, Tensor inventory / Forward graph:
// Q8_0 token_embd is row-gathered and dequantised, x = token_embd[ids]*sqrt(768).
//
// out[t][j] = f32(element(row ids[t], j) * scale): the stored element widened
// exactly to f32 (Q8_0: d*q, exact), then one round-to-nearest multiply.
//
// One warp per output row, grid-stride over rows.  The work is a pure stream:
// 16-byte read-only loads of the row, 16-byte stores of the f32 output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lhs_internal.cuh"

namespace lhs {
namespace {

constexpr int kWarps = 8;


__device__ __forceinline__ float4 scale4(float a, float b, float c, float d, float s) {
    return make_float4(__fmul_rn(a, s), __fmul_rn(b, s), __fmul_rn(c, s), __fmul_rn(d, s));
}


template <int DT, bool VEC>
__global__ void __launch_bounds__(kWarps * 32)
    embed_kernel(const uint8_t *__restrict__ table, int64_t vocab, int hidden, int64_t row_bytes,
                 const int32_t *__restrict__ ids, int64_t n, float scale, float *__restrict__ out,
                 int32_t *err) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = warp0; t < n; t += nwarps) {
        const int32_t id = ld_dep(ids + t);
        float *o = out + t * hidden;
        if (id < 0 || static_cast<int64_t>(id) >= vocab) {
            if (VEC) {
                float4 *o4 = reinterpret_cast<float4 *>(o);
                for (int c = lane; c < hidden / 4; c += 32) o4[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                for (int j = lane; j < hidden; j += 32) o[j] = 0.0f;
            }
            if (lane == 0) set_err(err, LHS_ERRBIT_BAD_TOKEN);
            continue;
        }
        const uint8_t *row = table + static_cast<int64_t>(id) * row_bytes;
        if (!VEC) {
            for (int j = lane; j < hidden; j += 32) o[j] = __fmul_rn(row_element<DT>(row, j), scale);
            continue;
        }
        float4 *o4 = reinterpret_cast<float4 *>(o);
        if (DT == LHS_F32) {
            const float4 *r4 = reinterpret_cast<const float4 *>(row);
            const int nv = hidden >> 2;
#pragma unroll 4
            for (int c = lane; c < nv; c += 32) {
                const float4 v = __ldg(r4 + c);
                o4[c] = scale4(v.x, v.y, v.z, v.w, scale);
            }
        } else if (DT == LHS_F16 || DT == LHS_BF16) {
            // four values per lane step: a warp's 16-byte stores are 512
            // contiguous bytes (whole 32-byte sectors)
            const uint2 *r2 = reinterpret_cast<const uint2 *>(row);
            const int nv = hidden >> 2;
#pragma unroll 4
            for (int c = lane; c < nv; c += 32) {
                const uint2 v = __ldg(r2 + c);
                float e[4];
                if (DT == LHS_F16) {
                    e[0] = f16_bits_to_f32(v.x & 0xFFFFu);
                    e[1] = f16_bits_to_f32(v.x >> 16);
                    e[2] = f16_bits_to_f32(v.y & 0xFFFFu);
                    e[3] = f16_bits_to_f32(v.y >> 16);
                } else {
                    e[0] = bf16_bits_to_f32(v.x & 0xFFFFu);
                    e[1] = bf16_bits_to_f32(v.x >> 16);
                    e[2] = bf16_bits_to_f32(v.y & 0xFFFFu);
                    e[3] = bf16_bits_to_f32(v.y >> 16);
                }
                o4[c] = scale4(e[0], e[1], e[2], e[3], scale);
            }
        } else {
            // Q8_0: four outputs j..j+3 (same block) per step; the block's
            // d and the four codes are 2-byte aligned (34-byte blocks).
            const int nv = hidden >> 2;
#pragma unroll 2
            for (int c = lane; c < nv; c += 32) {
                const int j = c << 2;
                const uint8_t *blk = row + (j >> 5) * 34;
                const unsigned short *b16 = reinterpret_cast<const unsigned short *>(blk);
                const float d = f16_bits_to_f32(__ldg(b16));
                const uint32_t q01 = __ldg(b16 + 1 + ((j & 31) >> 1));
                const uint32_t q23 = __ldg(b16 + 2 + ((j & 31) >> 1));
                const float q0 = static_cast<float>(static_cast<int8_t>(q01 & 0xFF));
                const float q1 = static_cast<float>(static_cast<int8_t>(q01 >> 8));
                const float q2 = static_cast<float>(static_cast<int8_t>(q23 & 0xFF));
                const float q3 = static_cast<float>(static_cast<int8_t>(q23 >> 8));
                o4[c] = scale4(__fmul_rn(d, q0), __fmul_rn(d, q1), __fmul_rn(d, q2),
                               __fmul_rn(d, q3), scale);
            }
        }
    }
}

template <int DT>
cudaError_t launch_dt(const lhs_table &t, const int32_t *ids, int64_t n, float scale, float *out,
                      int32_t *err, cudaStream_t stream, int num_sms) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(t.data) | reinterpret_cast<uintptr_t>(out);
    bool vec = (a % 16) == 0;
    if (DT == LHS_F32) vec = vec && (t.hidden % 4 == 0);
    if (DT == LHS_F16 || DT == LHS_BF16) vec = vec && (t.hidden % 8 == 0);
    if (DT == LHS_Q8_0) vec = vec && (t.hidden % 4 == 0);
    const int64_t blocks_needed = (n + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(num_sms) * 32;
    const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
    const uint8_t *tb = static_cast<const uint8_t *>(t.data);
    return launch_pdl(vec ? embed_kernel<DT, true> : embed_kernel<DT, false>, dim3(grid),
                      dim3(kWarps * 32), 0, stream, tb, t.vocab, t.hidden, t.row_bytes, ids, n,
                      scale, out, err);
}

}  // namespace

cudaError_t launch_embed(const lhs_table &t, const int32_t *ids, int64_t n, float scale,
                         float *out, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    switch (t.dtype) {
    case LHS_F32: return launch_dt<LHS_F32>(t, ids, n, scale, out, err, stream, dev.num_sms);
    case LHS_F16: return launch_dt<LHS_F16>(t, ids, n, scale, out, err, stream, dev.num_sms);
    case LHS_BF16: return launch_dt<LHS_BF16>(t, ids, n, scale, out, err, stream, dev.num_sms);
    default: return launch_dt<LHS_Q8_0>(t, ids, n, scale, out, err, stream, dev.num_sms);
    }
}

}  // namespace lhs
