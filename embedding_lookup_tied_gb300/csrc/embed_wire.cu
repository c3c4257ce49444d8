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
// The message is either the request (16-byte header) or the single-layer
// response (12-byte header [layer][seq_len][latency_ms]; ADR-0009 Wire
// Layout): the kernels take the header words and write the payload after
// them, with the vector paths when the payload is 16-byte aligned.
//
// f32 / f16: one warp per token, 8 elements per lane step (16-byte loads and
// stores).  i8: one warp per token — max|x| of the scaled row, then the
// codes (the same steps, in the same binary32 operations, as the i8
// encoder); rows up to 1024 values stay in registers between the two,
// longer rows are read a second time.  Q8_0 rows that are 16-byte multiples
// are first staged whole in a per-warp ring of shared memory, several tokens
// ahead, so that the row reads of many tokens are in flight at once.
#include <mutex>

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
                         const int32_t *__restrict__ ids, int64_t n, float scale, WireHdr hdr, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    uint8_t *pay = buf + 4 * hdr.n;
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
                         const int32_t *__restrict__ ids, int64_t n, float scale, WireHdr hdr, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sm_m[kI8Threads / 32];
    __shared__ int sm_f[kI8Threads / 32];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    for (int64_t p = blockIdx.x; p < n; p += gridDim.x) {
        const int32_t id = ld_dep(ids + p);
        const bool bad = bad_id(id, vocab);  // uniform over the block
        if (bad && threadIdx.x == 0) set_err(err, LHS_ERRBIT_BAD_TOKEN);
        const uint8_t *row = table + static_cast<int64_t>(bad ? 0 : id) * row_bytes;
        uint8_t *pos = buf + 4 * hdr.n + p * stride;
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
                              const int32_t *__restrict__ ids, int64_t n, float scale, WireHdr hdr, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
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
            ng, buf + 4 * hdr.n + p * stride, lane, err);
    }
}

// i8 with rows of at most 1024 values: one warp per token, the scaled row in
// registers between the max and the codes.
template <int DT>
__global__ void __launch_bounds__(128)
    embed_wire_i8_warp4_kernel(const uint8_t *__restrict__ table, int64_t vocab, int hidden, int64_t row_bytes,
                               const int32_t *__restrict__ ids, int64_t n, float scale, WireHdr hdr, uint8_t *__restrict__ buf, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
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
            n4, buf + 4 * hdr.n + p * stride, lane, err);
    }
}

// i8 with rows staged in shared memory: each warp keeps a ring of S whole
// rows (16-byte cp.async copies, issued S - 1 tokens ahead) so that several
// rows per warp are in flight while it quantises the current one; the token
// ids are read 32 at a time (one per lane) and passed round by shuffles.
// The quantiser is the encoder's (i8_position_warp4), fed from the staged row.
constexpr int kRingWarps = 4;
constexpr int kRingBytesPerWarp = 8192;  // S * row_bytes <= this

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// values 4s .. 4s+3 of a row held in shared memory
template <int DT>
__device__ __forceinline__ void staged_elements4(const uint8_t *row, int s, float (&v)[4]) {
    if (DT == LHS_F32) {
        const float4 a = *reinterpret_cast<const float4 *>(row + 16 * s);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if (DT == LHS_F16 || DT == LHS_BF16) {
        const uint2 w = *reinterpret_cast<const uint2 *>(row + 8 * s);
        v[0] = DT == LHS_F16 ? f16_bits_to_f32(w.x & 0xFFFFu) : bf16_bits_to_f32(w.x & 0xFFFFu);
        v[1] = DT == LHS_F16 ? f16_bits_to_f32(w.x >> 16) : bf16_bits_to_f32(w.x >> 16);
        v[2] = DT == LHS_F16 ? f16_bits_to_f32(w.y & 0xFFFFu) : bf16_bits_to_f32(w.y & 0xFFFFu);
        v[3] = DT == LHS_F16 ? f16_bits_to_f32(w.y >> 16) : bf16_bits_to_f32(w.y >> 16);
    } else {  // Q8_0: block s / 8, its codes 4 (s % 8) .. +3 (2-byte aligned)
        const unsigned short *b16 = reinterpret_cast<const unsigned short *>(row + (s >> 3) * 34);
        const float d = f16_bits_to_f32(b16[0]);
        const int q0 = 1 + (s & 7) * 2;
        const uint32_t w = static_cast<uint32_t>(b16[q0]) | (static_cast<uint32_t>(b16[q0 + 1]) << 16);
        // int8 -> binary32 without a conversion instruction: with u = q + 128
        // (the code's bits, top bit flipped), 0x4B000000 | u is the float
        // 2^23 + u, and subtracting 2^23 + 128 leaves q exactly
        const uint32_t u = w ^ 0x80808080u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float q = __int_as_float(static_cast<int>(__byte_perm(u, 0x4B000000u, 0x7440 + i))) - 8388736.0f;
            v[i] = __fmul_rn(d, q);
        }
    }
}

// Four codes of one position, packed little-endian: q = clamp(rne(v /
// scale), -127, 127) with the division correctly rounded.  Fast path: t = v
// * rcp; adding 1.5 * 2^23 rounds it to an integer held in the sum's low
// bits (its low byte is the code's two's-complement byte), which is the
// division's result unless |t| reaches 127.5 or t lies within 2^-12 of a
// half-integer (far beyond the product's error of a few ulp); those values
// take the exact division.
__device__ __forceinline__ uint32_t i8_quant4(const float (&v)[4], float scale, float rcp) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    uint32_t yb[4];
    uint32_t slow = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float t = __fmul_rn(v[i], rcp);
        const float y = __fadd_rn(t, kMagic);
        const float r = __fsub_rn(y, kMagic);
        yb[i] = __float_as_uint(y);
        if (!(fabsf(t) < 127.5f && fabsf(__fsub_rn(t, r)) < 0.5f - 0x1p-12f)) slow |= 1u << i;
    }
    uint32_t w = __byte_perm(__byte_perm(yb[0], yb[1], 0x0040), __byte_perm(yb[2], yb[3], 0x0040), 0x5410);
    while (slow) {
        const int i = __ffs(slow) - 1;
        slow &= slow - 1;
        float vi = v[0];
#pragma unroll
        for (int j = 1; j < 4; ++j) vi = i == j ? v[j] : vi;
        const int qi = __float2int_rn(fminf(fmaxf(rintf(__fdiv_rn(vi, scale)), -127.0f), 127.0f));
        const uint32_t sh = 8u * static_cast<uint32_t>(i);
        w = (w & ~(0xFFu << sh)) | ((static_cast<uint32_t>(qi) & 0xFFu) << sh);
    }
    return w;
}

// i8_quant4 for a row whose every |v| is at most its max m (scale = m / 127,
// so |v / scale| <= 127 and no clamp is reached): one predicate per four
// values chooses the exact divisions, for t within 2^-12 of a half-integer.
__device__ __forceinline__ uint32_t i8_quant4_bounded(const float (&v)[4], float scale, float rcp) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    uint32_t yb[4];
    bool fast = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float t = __fmul_rn(v[i], rcp);
        const float y = __fadd_rn(t, kMagic);
        yb[i] = __float_as_uint(y);
        fast &= fabsf(__fsub_rn(t, __fsub_rn(y, kMagic))) < 0.5f - 0x1p-12f;
    }
    if (fast) return __byte_perm(__byte_perm(yb[0], yb[1], 0x0040), __byte_perm(yb[2], yb[3], 0x0040), 0x5410);
    return i8_quant4(v, scale, rcp);
}

// S: ring slots per warp (2, 4 or 8); KS: value steps (4 values each) per
// lane, n4 <= 32 * KS; FULL: n4 == 32 * KS (no step is out of the row).
// Shared memory: kRingWarps rings of S rows, one zero row (read for a bad
// id, which gives the all-zero position the format asks for), then
// kRingWarps x S token ids.
template <int DT, int KS, bool FULL>
__global__ void __launch_bounds__(kRingWarps * 32)
    embed_wire_i8_ring_kernel(const uint8_t *__restrict__ table, int64_t vocab, int hidden, int64_t row_bytes,
                              const int32_t *__restrict__ ids, int64_t n, float scale, WireHdr hdr, uint8_t *__restrict__ buf, int32_t *err, int S) {
    extern __shared__ __align__(16) uint8_t ring_smem[];
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        write_hdr(buf, hdr);
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kRingWarps + wib;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * kRingWarps;
    uint8_t *ring = ring_smem + static_cast<size_t>(wib) * S * row_bytes;
    uint8_t *zero_row = ring_smem + static_cast<size_t>(kRingWarps) * S * row_bytes;
    int32_t *slot_id = reinterpret_cast<int32_t *>(zero_row + row_bytes) + wib * S;
    for (int c = threadIdx.x; c < static_cast<int>(row_bytes >> 4); c += kRingWarps * 32)
        reinterpret_cast<uint4 *>(zero_row)[c] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const int64_t stride = static_cast<int64_t>(hidden) + 8;
    const int n4 = hidden >> 2, nc = static_cast<int>(row_bytes >> 4);
    const int64_t mine = w < n ? (n - 1 - w) / nw + 1 : 0;  // tokens of this warp: w, w + nw, ...
    // ids of this warp's tokens i .. i+31, lane l holding token i + l; read
    // in increasing i by the copies, which leave each id in its slot
    int32_t idbuf = 0;
    int64_t idbase = -64;
    auto id_of = [&](int64_t i) {  // warp-uniform, non-decreasing i
        if (i >= idbase + 32) {
            idbase = i;
            const int64_t t = w + (i + lane) * nw;
            idbuf = i + lane < mine ? ld_dep(ids + t) : 0;
        }
        return __shfl_sync(0xFFFFFFFFu, idbuf, static_cast<int>(i - idbase));
    };
    // S is 2, 4 or 8: a token's slot is its index's low bits (a 64-bit
    // remainder by a run-time S would cost a division routine per use)
    const int64_t smask = S - 1;
    auto issue = [&](int64_t i) {  // copy token i's row into slot i & (S - 1) (one group per token)
        if (i < mine) {
            const int32_t id = id_of(i);
            const int slot = static_cast<int>(i & smask);
            if (lane == 0) slot_id[slot] = id;
            if (id >= 0 && static_cast<int64_t>(id) < vocab) {
                const uint8_t *src = table + static_cast<int64_t>(id) * row_bytes;
                uint8_t *dst = ring + static_cast<size_t>(slot) * row_bytes;
                for (int c = lane; c < nc; c += 32) cp_async16(dst + 16 * c, src + 16 * c);
            }
        }
        cp_async_commit();
    };
    // Q8_0: the byte offsets, in step 0, of its block's d and of the aligned
    // words around its four codes (2-byte aligned), and the byte selector.
    // Step k (values 4 (lane + 32 k) ..) lies 4 k blocks further on, 136 k
    // bytes, at the same place in its block: one selector for every step.
    int q8_d0 = 0, q8_w0 = 0;
    uint32_t q8_sel = 0x3210u;
    if constexpr (DT == LHS_Q8_0) {
        const int o = (lane >> 3) * 34 + 2 + (lane & 7) * 4;
        q8_d0 = (lane >> 3) * 34;
        q8_w0 = o & ~3;
        q8_sel = (o & 3) ? 0x5432u : 0x3210u;
    }
    for (int64_t i = 0; i < S - 1; ++i) issue(i);
    for (int64_t i = 0; i < mine; ++i) {
        issue(i + S - 1);
        // token i's group is done once at most S - 1 newer ones are pending
        if (S == 8) cp_async_wait<7>();
        else if (S == 4) cp_async_wait<3>();
        else cp_async_wait<1>();
        __syncwarp();
        const int slot = static_cast<int>(i & smask);
        const int32_t id = slot_id[slot];
        const bool bad = id < 0 || static_cast<int64_t>(id) >= vocab;
        const uint8_t *row = bad ? zero_row : ring + static_cast<size_t>(slot) * row_bytes;
        // the scaled row in registers; max |x| as the largest magnitude bit
        // pattern (inf and NaN lie above every finite one).  Q8_0: a value is
        // non-finite only through its block's d (inf / NaN) or an overflow to
        // inf, so the float max plus a test of each d is enough.
        float c[KS][4];
        uint32_t mb = 0u;
        if constexpr (DT == LHS_Q8_0) {
            float mf = 0.0f;
            bool dbad = false;
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                if (FULL || lane + 32 * k < n4) {
                    const float d = f16_bits_to_f32(*reinterpret_cast<const unsigned short *>(row + q8_d0 + 136 * k));
                    dbad = dbad || !(fabsf(d) <= 3.402823466e38f);
                    const uint32_t w0 = *reinterpret_cast<const uint32_t *>(row + q8_w0 + 136 * k);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t *>(row + q8_w0 + 136 * k + 4);
                    const uint32_t u = __byte_perm(w0, w1, q8_sel) ^ 0x80808080u;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float qv = __int_as_float(static_cast<int>(__byte_perm(u, 0x4B000000u, 0x7440 + q))) - 8388736.0f;
                        c[k][q] = __fmul_rn(__fmul_rn(d, qv), scale);
                        mf = fmaxf(mf, fabsf(c[k][q]));
                    }
                }
            }
            mb = dbad ? 0x7F800000u : __float_as_uint(mf);
        } else {
#pragma unroll
            for (int k = 0; k < KS; ++k) {
                const int st = lane + 32 * k;
                if (FULL || st < n4) {
                    staged_elements4<DT>(row, st, c[k]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        c[k][q] = __fmul_rn(c[k][q], scale);
                        mb = max(mb, __float_as_uint(c[k][q]) & 0x7FFFFFFFu);
                    }
                }
            }
        }
        __syncwarp();  // every lane has read the slot before it is refilled
        mb = __reduce_max_sync(0xFFFFFFFFu, mb);
        const bool nonfinite = mb >= 0x7F800000u;
        const float qs = nonfinite ? 0.0f : __fdiv_rn(__uint_as_float(mb), 127.0f);
        const float rcp = __frcp_rn(qs);
        uint8_t *pos = buf + 4 * hdr.n + (w + i * nw) * stride;
        if (lane == 0) {
            *reinterpret_cast<uint2 *>(pos) = make_uint2(__float_as_uint(qs), 0u);
            if (bad) set_err(err, LHS_ERRBIT_BAD_TOKEN);
            if (nonfinite) set_err(err, LHS_ERRBIT_NONFINITE);
        }
        uint32_t *codes = reinterpret_cast<uint32_t *>(pos + 8);
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            const int st = lane + 32 * k;
            if (FULL || st < n4) codes[st] = qs == 0.0f ? 0u : i8_quant4_bounded(c[k], qs, rcp);
        }
    }
    cp_async_wait<0>();
}

template <int DT>
cudaError_t launch_dt(const lhs_table &t, const int32_t *ids, int64_t n, float scale, int fmt,
                      const WireHdr &hdr, uint8_t *buf, int32_t *err,
                      cudaStream_t stream, int num_sms, int device) {
    const uint8_t *tb = static_cast<const uint8_t *>(t.data);
    // 8-element steps: rows 16-byte aligned (Q8_0: 2-byte), hidden % 8 == 0,
    // and the payload after the header on a 16-byte boundary
    bool vec = t.hidden % 8 == 0 && reinterpret_cast<uintptr_t>(buf + 4 * hdr.n) % 16 == 0;
    if (DT != LHS_Q8_0) vec = vec && (reinterpret_cast<uintptr_t>(t.data) % 16 == 0) && (t.row_bytes % 16 == 0);
    // Q8_0 rows staged whole by 16-byte copies (16-byte multiples at 16-byte
    // aligned addresses): the 2-byte-aligned blocks are then read from shared
    // memory.  Rows of the other types are read straight from global memory
    // by aligned vector loads, which staging does not speed up.
    const bool stage = DT == LHS_Q8_0 && t.row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(t.data) % 16 == 0 &&
                       t.row_bytes * 2 <= kRingBytesPerWarp;
    if (fmt == LHS_WIRE_I8 && vec && stage && t.hidden <= 32 * kI8WarpSteps * 4) {
        const int S = t.row_bytes * 8 <= kRingBytesPerWarp ? 8 : (t.row_bytes * 4 <= kRingBytesPerWarp ? 4 : 2);
        const int ks = (t.hidden / 4 + 31) / 32;  // 1 .. 8, rounded up to even below
        using Kern = void (*)(const uint8_t *, int64_t, int, int64_t, const int32_t *, int64_t, float, WireHdr,
                              uint8_t *, int32_t *, int);
        static const Kern kTable[2][4] = {
            {embed_wire_i8_ring_kernel<DT, 2, false>, embed_wire_i8_ring_kernel<DT, 4, false>,
             embed_wire_i8_ring_kernel<DT, 6, false>, embed_wire_i8_ring_kernel<DT, 8, false>},
            {embed_wire_i8_ring_kernel<DT, 2, true>, embed_wire_i8_ring_kernel<DT, 4, true>,
             embed_wire_i8_ring_kernel<DT, 6, true>, embed_wire_i8_ring_kernel<DT, 8, true>}};
        const int kidx = (ks + 1) / 2 - 1;
        const bool full = t.hidden / 4 == 32 * 2 * (kidx + 1);
        const Kern kern = kTable[full][kidx];
        const int which = full * 4 + kidx;
        const size_t smem = static_cast<size_t>(kRingWarps) * S * (t.row_bytes + 4) + t.row_bytes;
        {
            static std::mutex mu;
            static bool attr_done[8][64] = {};
            std::lock_guard<std::mutex> lock(mu);
            if (!attr_done[which][device]) {
                const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           static_cast<int>(kRingWarps * kRingBytesPerWarp + 8192));
                if (e != cudaSuccess) return e;
                attr_done[which][device] = true;
            }
        }
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRingWarps * 32, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
        const int64_t want = (n + kRingWarps * 4 - 1) / (kRingWarps * 4);  // >= 4 tokens per warp
        const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
        const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
        return launch_pdl(kern, dim3(grid), dim3(kRingWarps * 32), smem, stream, tb, t.vocab, t.hidden,
                          t.row_bytes, ids, n, scale, hdr, buf, err, S);
    }
    if (fmt == LHS_WIRE_I8 && vec && t.hidden <= 32 * kI8WarpSteps * 4) {
        const int wps = i8_warps_per_sm(t.row_bytes);
        const int grid = warp_kernel_grid(embed_wire_i8_warp4_kernel<DT>, n, wps, num_sms, device);
        return launch_pdl(embed_wire_i8_warp4_kernel<DT>, dim3(grid), dim3(128), 0, stream, tb, t.vocab, t.hidden,
                          t.row_bytes, ids, n, scale, hdr, buf, err);
    }
    if (fmt == LHS_WIRE_I8 && vec) {
        const int wps = i8_warps_per_sm(t.row_bytes);
        const int grid = warp_kernel_grid(embed_wire_i8_warp_kernel<DT>, n, wps, num_sms, device);
        return launch_pdl(embed_wire_i8_warp_kernel<DT>, dim3(grid), dim3(128), 0, stream, tb, t.vocab, t.hidden,
                          t.row_bytes, ids, n, scale, hdr, buf, err);
    }
    if (fmt == LHS_WIRE_I8) {
        const int64_t cap = static_cast<int64_t>(num_sms) * 16;
        const int grid = static_cast<int>(n < 1 ? 1 : (n < cap ? n : cap));
        return launch_pdl(embed_wire_i8_kernel<DT>, dim3(grid),
                          dim3(kI8Threads), 0, stream, tb, t.vocab, t.hidden, t.row_bytes, ids, n, scale,
                          hdr, buf, err);
    }
    const int64_t blocks_needed = (n + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(num_sms) * 32;
    const int grid = static_cast<int>(blocks_needed < 1 ? 1 : (blocks_needed < cap ? blocks_needed : cap));
    auto k = fmt == LHS_WIRE_F16
                 ? (vec ? embed_wire_ew_kernel<DT, LHS_WIRE_F16, true> : embed_wire_ew_kernel<DT, LHS_WIRE_F16, false>)
                 : (vec ? embed_wire_ew_kernel<DT, LHS_WIRE_F32, true> : embed_wire_ew_kernel<DT, LHS_WIRE_F32, false>);
    return launch_pdl(k, dim3(grid), dim3(kWarps * 32), 0, stream, tb, t.vocab, t.hidden, t.row_bytes, ids,
                      n, scale, hdr, buf, err);
}

}  // namespace

cudaError_t launch_embed_wire(const lhs_table &t, const int32_t *ids, int64_t n, float scale, int fmt,
                              const WireHdr &hdr, void *buf, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    uint8_t *b = static_cast<uint8_t *>(buf);
    switch (t.dtype) {
    case LHS_F32: return launch_dt<LHS_F32>(t, ids, n, scale, fmt, hdr, b, err, stream,
                                                   dev.num_sms, dev.device);
    case LHS_F16: return launch_dt<LHS_F16>(t, ids, n, scale, fmt, hdr, b, err, stream,
                                                   dev.num_sms, dev.device);
    case LHS_BF16: return launch_dt<LHS_BF16>(t, ids, n, scale, fmt, hdr, b, err, stream,
                                                   dev.num_sms, dev.device);
    default: return launch_dt<LHS_Q8_0>(t, ids, n, scale, fmt, hdr, b, err, stream,
                                                   dev.num_sms, dev.device);
    }
}

}  // namespace lhs
