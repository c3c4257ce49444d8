// dedup.cu — distinct ids of a batch, and the gather through them.
//
// HELIX "Columnar Embedding", Appendix B: the honest prefetch is "tokenize,
// dedupe, issue range fetches in parallel before the embed lookup" — the ids
// are known before the lookup, so the distinct rows are fetched once each.
// On a device-resident table the same plan reads and decodes every distinct
// row once and copies it to each position that names it.
//
// Distinct ids without a sort: ids are bounded by the vocabulary, so a
// per-vocab-row flag array, an exclusive scan of it (tile sums, a scan of
// the sums, then each tile's local scan) and one pass over the ids give the
// ascending distinct ids and every position's index into them.
#include "lhs_internal.cuh"

namespace lhs {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kTile = kScanThreads;  // flags per scan tile

__global__ void __launch_bounds__(256) zero_u32_kernel(uint32_t *p, int64_t n) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = 0u;
}

__global__ void __launch_bounds__(256)
    mark_kernel(const int32_t *__restrict__ ids, int64_t n, int64_t vocab, uint32_t *flags, int32_t *err) {
    pdl_trigger();
    pdl_wait();
    bool bad = false;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t id = ld_dep(ids + i);
        if (id < 0 || static_cast<int64_t>(id) >= vocab) bad = true;
        else flags[id] = 1u;  // every writer stores the same value
    }
    if (bad) set_err(err, LHS_ERRBIT_BAD_TOKEN);
}

// Block-wide exclusive scan of one value per thread; returns the block total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t &excl, uint32_t *warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0u;
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += t;
        }
        warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    excl = warp_sums[warp] + incl - v;
    const uint32_t total = warp_sums[32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kScanThreads)
    tile_sum_kernel(const uint32_t *__restrict__ flags, int64_t vocab, uint32_t *tile_sums) {
    pdl_trigger();
    pdl_wait();
    __shared__ uint32_t ws[33];
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kTile + threadIdx.x;
    uint32_t excl;
    const uint32_t total = block_exclusive_scan(i < vocab ? ld_dep(flags + i) : 0u, excl, ws);
    if (threadIdx.x == 0) tile_sums[blockIdx.x] = total;
}

// One block: exclusive scan of the tile sums in place (any number of tiles),
// and the distinct count.
__global__ void __launch_bounds__(kScanThreads)
    scan_sums_kernel(uint32_t *tile_sums, int64_t ntiles, int32_t *count) {
    pdl_trigger();
    pdl_wait();
    __shared__ uint32_t ws[33];
    uint32_t carry = 0;
    for (int64_t base = 0; base < ntiles; base += kScanThreads) {
        const int64_t i = base + threadIdx.x;
        const uint32_t v = i < ntiles ? tile_sums[i] : 0u;
        uint32_t excl;
        const uint32_t total = block_exclusive_scan(v, excl, ws);
        if (i < ntiles) tile_sums[i] = carry + excl;
        carry += total;
    }
    if (threadIdx.x == 0) *count = static_cast<int32_t>(carry);
}

// rank[v] = number of distinct ids below v (for flagged v); unique[rank] = v.
__global__ void __launch_bounds__(kScanThreads)
    rank_kernel(uint32_t *flags, int64_t vocab, const uint32_t *__restrict__ tile_offs, int32_t *unique) {
    pdl_trigger();
    pdl_wait();
    __shared__ uint32_t ws[33];
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kTile + threadIdx.x;
    const uint32_t f = i < vocab ? flags[i] : 0u;
    uint32_t excl;
    block_exclusive_scan(f, excl, ws);
    if (f) {
        const uint32_t r = ld_dep(tile_offs + blockIdx.x) + excl;
        flags[i] = r;  // the flag array becomes the rank array
        unique[r] = static_cast<int32_t>(i);
    }
}

__global__ void __launch_bounds__(256)
    inverse_kernel(const int32_t *__restrict__ ids, int64_t n, int64_t vocab, const uint32_t *__restrict__ rank,
                   int32_t *inverse) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t id = ld_dep(ids + i);
        inverse[i] = (id < 0 || static_cast<int64_t>(id) >= vocab) ? -1 : static_cast<int32_t>(ld_dep(rank + id));
    }
}

// Distinct rows, decoded and scaled once: rows[u] for u < *count.
template <int DT>
__global__ void __launch_bounds__(256)
    gather_unique_kernel(const uint8_t *__restrict__ table, int hidden, int64_t row_bytes,
                         const int32_t *__restrict__ unique, const int32_t *__restrict__ count, float scale,
                         float *__restrict__ rows) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nu = ld_dep(count);
    for (int64_t u = w0; u < nu; u += nw) {
        const uint8_t *row = table + static_cast<int64_t>(ld_dep(unique + u)) * row_bytes;
        float *o = rows + u * hidden;
        for (int j = lane; j < hidden; j += 32) o[j] = __fmul_rn(row_element<DT>(row, j), scale);
    }
}

// out[i] = rows[inverse[i]], or zeros for a bad id.
__global__ void __launch_bounds__(256)
    scatter_rows_kernel(const int32_t *__restrict__ inverse, int64_t n, int hidden, const float *__restrict__ rows,
                        float *__restrict__ out, bool vec) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t i = w0; i < n; i += nw) {
        const int32_t u = ld_dep(inverse + i);
        float *o = out + i * hidden;
        if (vec) {
            float4 *o4 = reinterpret_cast<float4 *>(o);
            const float4 *r4 = reinterpret_cast<const float4 *>(rows + static_cast<int64_t>(u < 0 ? 0 : u) * hidden);
            for (int c = lane; c < hidden / 4; c += 32) o4[c] = u < 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : ld_dep(r4 + c);
        } else {
            const float *r = rows + static_cast<int64_t>(u < 0 ? 0 : u) * hidden;
            for (int j = lane; j < hidden; j += 32) o[j] = u < 0 ? 0.0f : ld_dep(r + j);
        }
    }
}

int grid_for(int64_t items, int per_block, int num_sms, int per_sm) {
    const int64_t need = (items + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    const int64_t g = need < cap ? need : cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

size_t unique_ids_workspace(int64_t vocab) {
    const int64_t ntiles = (vocab + kTile - 1) / kTile;
    return align256(static_cast<size_t>(vocab) * 4) + align256(static_cast<size_t>(ntiles) * 4);
}

cudaError_t launch_unique_ids(int64_t vocab, const int32_t *ids, int64_t n, int32_t *unique, int32_t *inverse,
                              int32_t *count, void *ws, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *flags = reinterpret_cast<uint32_t *>(w);
    uint32_t *tile_sums = reinterpret_cast<uint32_t *>(w + align256(static_cast<size_t>(vocab) * 4));
    const int64_t ntiles = (vocab + kTile - 1) / kTile;
    if ((e = launch_pdl(zero_u32_kernel, dim3(grid_for(vocab, 256, dev.num_sms, 8)), dim3(256), 0, stream, flags,
                        vocab)) != cudaSuccess)
        return e;
    if (n > 0 && (e = launch_pdl(mark_kernel, dim3(grid_for(n, 256, dev.num_sms, 8)), dim3(256), 0, stream, ids, n,
                                 vocab, flags, err)) != cudaSuccess)
        return e;
    if ((e = launch_pdl(tile_sum_kernel, dim3(static_cast<unsigned>(ntiles)), dim3(kScanThreads), 0, stream,
                        static_cast<const uint32_t *>(flags), vocab, tile_sums)) != cudaSuccess)
        return e;
    if ((e = launch_pdl(scan_sums_kernel, dim3(1), dim3(kScanThreads), 0, stream, tile_sums, ntiles, count)) !=
        cudaSuccess)
        return e;
    if ((e = launch_pdl(rank_kernel, dim3(static_cast<unsigned>(ntiles)), dim3(kScanThreads), 0, stream, flags,
                        vocab, static_cast<const uint32_t *>(tile_sums), unique)) != cudaSuccess)
        return e;
    if (n > 0)
        e = launch_pdl(inverse_kernel, dim3(grid_for(n, 256, dev.num_sms, 8)), dim3(256), 0, stream, ids, n, vocab,
                       static_cast<const uint32_t *>(flags), inverse);
    return e;
}

size_t embed_dedup_workspace(const lhs_table &t, int64_t n) {
    const int64_t nu = n < t.vocab ? n : t.vocab;
    return unique_ids_workspace(t.vocab) + align256(static_cast<size_t>(nu) * 4) +
           align256(static_cast<size_t>(n) * 4) + 256 + align256(static_cast<size_t>(nu) * t.hidden * 4);
}

cudaError_t launch_embed_dedup(const lhs_table &t, const int32_t *ids, int64_t n, float scale, float *out,
                               void *ws, int32_t *err, cudaStream_t stream) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    const int64_t nu = n < t.vocab ? n : t.vocab;
    uint8_t *w = static_cast<uint8_t *>(ws);
    size_t off = unique_ids_workspace(t.vocab);
    int32_t *unique = reinterpret_cast<int32_t *>(w + off);
    off += align256(static_cast<size_t>(nu) * 4);
    int32_t *inverse = reinterpret_cast<int32_t *>(w + off);
    off += align256(static_cast<size_t>(n) * 4);
    int32_t *count = reinterpret_cast<int32_t *>(w + off);
    off += 256;
    float *rows = reinterpret_cast<float *>(w + off);
    if ((e = launch_unique_ids(t.vocab, ids, n, unique, inverse, count, ws, err, stream)) != cudaSuccess) return e;
    const uint8_t *tb = static_cast<const uint8_t *>(t.data);
    const int grid = grid_for(nu * 32, 256, dev.num_sms, 8);
    switch (t.dtype) {
    case LHS_F32: e = launch_pdl(gather_unique_kernel<LHS_F32>, dim3(grid), dim3(256), 0, stream, tb, t.hidden, t.row_bytes, static_cast<const int32_t *>(unique), static_cast<const int32_t *>(count), scale, rows); break;
    case LHS_F16: e = launch_pdl(gather_unique_kernel<LHS_F16>, dim3(grid), dim3(256), 0, stream, tb, t.hidden, t.row_bytes, static_cast<const int32_t *>(unique), static_cast<const int32_t *>(count), scale, rows); break;
    case LHS_BF16: e = launch_pdl(gather_unique_kernel<LHS_BF16>, dim3(grid), dim3(256), 0, stream, tb, t.hidden, t.row_bytes, static_cast<const int32_t *>(unique), static_cast<const int32_t *>(count), scale, rows); break;
    default: e = launch_pdl(gather_unique_kernel<LHS_Q8_0>, dim3(grid), dim3(256), 0, stream, tb, t.hidden, t.row_bytes, static_cast<const int32_t *>(unique), static_cast<const int32_t *>(count), scale, rows); break;
    }
    if (e != cudaSuccess) return e;
    const bool vec = t.hidden % 4 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
    return launch_pdl(scatter_rows_kernel, dim3(grid_for(n * 32, 256, dev.num_sms, 8)), dim3(256), 0, stream,
                      static_cast<const int32_t *>(inverse), n, t.hidden, static_cast<const float *>(rows), out,
                      vec);
}

}  // namespace lhs
