// lhs_abi.cu — the C-ABI boundary: argument checks, workspace sizing and
// dispatch to the kernels.  Every entry point is declared in include/lhs.h.
// Host-detectable errors return a status and enqueue nothing; data-dependent
// errors are reported by the kernels through the caller's error word.
#include <cmath>
#include <mutex>

#include <cstring>

#include "lhs_internal.cuh"

namespace lhs {

static thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return LHS_OK;
    g_last_cuda_error = static_cast<int>(e);
    return LHS_ERR_CUDA;
}

cudaError_t device_info(DeviceInfo *out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d{};
        d.device = dev;
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cache[dev] = d;
        have[dev] = true;
    }
    *out = cache[dev];
    return cudaSuccess;
}

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static int64_t row_bytes_of(int32_t dtype, int32_t hidden) {
    switch (dtype) {
    case LHS_F32: return static_cast<int64_t>(hidden) * 4;
    case LHS_F16:
    case LHS_BF16: return static_cast<int64_t>(hidden) * 2;
    case LHS_Q8_0: return hidden % 32 ? -1 : static_cast<int64_t>(hidden / 32) * 34;
    default: return -1;
    }
}

static int check_table(const lhs_table *t) {
    if (!t || !t->data || !aligned(t->data, 16)) return LHS_ERR_INVALID_ARG;
    if (t->vocab < 1 || t->vocab > 0x7FFFFFFFll || t->hidden < 1) return LHS_ERR_INVALID_ARG;
    const int64_t rb = row_bytes_of(t->dtype, t->hidden);
    if (rb < 0 || rb != t->row_bytes) return LHS_ERR_INVALID_ARG;
    return LHS_OK;
}

static int check_lm_head_args(const lhs_table *t, const void *resid, int32_t resid_dtype,
                              int32_t batch, int32_t k) {
    int rc = check_table(t);
    if (rc) return rc;
    if (!resid || !aligned(resid, 16)) return LHS_ERR_INVALID_ARG;
    if (resid_dtype != LHS_F32 && resid_dtype != LHS_BF16) return LHS_ERR_INVALID_ARG;
    if (batch < 1) return LHS_ERR_INVALID_ARG;
    if (k < 0 || k > kMaxK || k > t->vocab) return LHS_ERR_INVALID_ARG;
    return LHS_OK;
}

}  // namespace lhs

using namespace lhs;

extern "C" {

int lhs_table_init(lhs_table *t, const void *d_table, int64_t vocab, int32_t hidden, int32_t dtype) {
    if (!t) return LHS_ERR_INVALID_ARG;
    lhs_table tmp;
    tmp.data = d_table;
    tmp.vocab = vocab;
    tmp.hidden = hidden;
    tmp.dtype = dtype;
    tmp.row_bytes = row_bytes_of(dtype, hidden);
    const int rc = check_table(&tmp);
    if (rc) return rc;
    *t = tmp;
    return LHS_OK;
}

int lhs_table_info(const lhs_table *t, int64_t *vocab, int32_t *hidden, int64_t *row_bytes,
                   int64_t *total_bytes) {
    const int rc = check_table(t);
    if (rc) return rc;
    if (vocab) *vocab = t->vocab;
    if (hidden) *hidden = t->hidden;
    if (row_bytes) *row_bytes = t->row_bytes;
    if (total_bytes) *total_bytes = t->vocab * t->row_bytes;
    return LHS_OK;
}

int lhs_embed(const lhs_table *t, const int32_t *d_ids, int64_t n, float scale, float *d_out,
              int32_t *d_err, void *stream) {
    int rc = check_table(t);
    if (rc) return rc;
    if (n < 0 || !std::isfinite(scale)) return LHS_ERR_INVALID_ARG;
    if (n == 0) return LHS_OK;
    if (!d_ids || !d_out || !d_err || !aligned(d_ids, 4) || !aligned(d_out, 16) || !aligned(d_err, 4))
        return LHS_ERR_INVALID_ARG;
    return cuda_status(launch_embed(*t, d_ids, n, scale, d_out, d_err, static_cast<cudaStream_t>(stream)));
}

int lhs_embed_wire(const lhs_table *t, const int32_t *d_ids, int64_t n, float scale, int32_t fmt,
                   uint32_t layer, uint32_t flags, uint32_t top_k, void *d_buf, size_t buf_bytes,
                   int32_t *d_err, void *stream) {
    int rc = check_table(t);
    if (rc) return rc;
    if (n < 0 || n > INT32_MAX || !std::isfinite(scale)) return LHS_ERR_INVALID_ARG;
    const int64_t need = lhs_wire_bytes(fmt, static_cast<int32_t>(n), t->hidden);
    if (need < 0) return LHS_ERR_INVALID_ARG;
    if (!d_buf || !d_err || !aligned(d_buf, 16) || !aligned(d_err, 4)) return LHS_ERR_INVALID_ARG;
    if (n > 0 && (!d_ids || !aligned(d_ids, 4))) return LHS_ERR_INVALID_ARG;
    if (buf_bytes < static_cast<size_t>(need)) return LHS_ERR_BUFFER_TOO_SMALL;
    const WireHdr hdr = {{layer, static_cast<uint32_t>(n), flags, top_k}, 4};
    return cuda_status(launch_embed_wire(*t, d_ids, n, scale, fmt, hdr, d_buf, d_err,
                                         static_cast<cudaStream_t>(stream)));
}

int lhs_embed_wire_response(const lhs_table *t, const int32_t *d_ids, int64_t n, float scale, int32_t fmt,
                            uint32_t layer, float latency_ms, void *d_buf, size_t buf_bytes, int32_t *d_err,
                            void *stream) {
    int rc = check_table(t);
    if (rc) return rc;
    if (n < 0 || n > INT32_MAX || !std::isfinite(scale)) return LHS_ERR_INVALID_ARG;
    const int64_t need = lhs_wire_response_bytes(fmt, static_cast<int32_t>(n), t->hidden);
    if (need < 0) return LHS_ERR_INVALID_ARG;
    if (!d_buf || !d_err || !aligned(d_buf, 4) || !aligned(d_err, 4)) return LHS_ERR_INVALID_ARG;
    if (n > 0 && (!d_ids || !aligned(d_ids, 4))) return LHS_ERR_INVALID_ARG;
    if (buf_bytes < static_cast<size_t>(need)) return LHS_ERR_BUFFER_TOO_SMALL;
    uint32_t lat;
    memcpy(&lat, &latency_ms, 4);
    const WireHdr hdr = {{layer, static_cast<uint32_t>(n), lat, 0u}, 3};
    return cuda_status(launch_embed_wire(*t, d_ids, n, scale, fmt, hdr, d_buf, d_err,
                                         static_cast<cudaStream_t>(stream)));
}

int64_t lhs_unique_ids_workspace(int64_t vocab) {
    if (vocab < 1 || vocab > INT32_MAX) return -1;
    return static_cast<int64_t>(unique_ids_workspace(vocab));
}

int lhs_unique_ids(int64_t vocab, const int32_t *d_ids, int64_t n, int32_t *d_unique, int32_t *d_inverse,
                   int32_t *d_count, void *d_ws, size_t ws_bytes, int32_t *d_err, void *stream) {
    if (vocab < 1 || vocab > INT32_MAX || n < 0) return LHS_ERR_INVALID_ARG;
    if (!d_count || !d_ws || !d_err || !aligned(d_count, 4) || !aligned(d_ws, 16) || !aligned(d_err, 4))
        return LHS_ERR_INVALID_ARG;
    if (n > 0 && (!d_ids || !d_unique || !d_inverse || !aligned(d_ids, 4) || !aligned(d_unique, 4) ||
                  !aligned(d_inverse, 4)))
        return LHS_ERR_INVALID_ARG;
    if (ws_bytes < unique_ids_workspace(vocab)) return LHS_ERR_BUFFER_TOO_SMALL;
    return cuda_status(launch_unique_ids(vocab, d_ids, n, d_unique, d_inverse, d_count, d_ws, d_err,
                                         static_cast<cudaStream_t>(stream)));
}

int64_t lhs_embed_dedup_workspace(const lhs_table *t, int64_t n) {
    if (check_table(t) || n < 0) return -1;
    return static_cast<int64_t>(embed_dedup_workspace(*t, n));
}

int lhs_embed_dedup(const lhs_table *t, const int32_t *d_ids, int64_t n, float scale, float *d_out, void *d_ws,
                    size_t ws_bytes, int32_t *d_err, void *stream) {
    int rc = check_table(t);
    if (rc) return rc;
    if (n < 0 || !std::isfinite(scale)) return LHS_ERR_INVALID_ARG;
    if (n == 0) return LHS_OK;
    if (!d_ids || !d_out || !d_ws || !d_err || !aligned(d_ids, 4) || !aligned(d_out, 16) || !aligned(d_ws, 16) ||
        !aligned(d_err, 4))
        return LHS_ERR_INVALID_ARG;
    if (ws_bytes < embed_dedup_workspace(*t, n)) return LHS_ERR_BUFFER_TOO_SMALL;
    return cuda_status(launch_embed_dedup(*t, d_ids, n, scale, d_out, d_ws, d_err, static_cast<cudaStream_t>(stream)));
}

int lhs_embed_mixed(const void *d_data, int64_t data_bytes, const int64_t *d_row_offset, const uint8_t *d_row_dtype,
                    int64_t vocab, int32_t hidden, const int32_t *d_ids, int64_t n, float scale, float *d_out,
                    int32_t *d_err, void *stream) {
    if (!d_data || !aligned(d_data, 16) || data_bytes < 0 || !d_row_offset || !aligned(d_row_offset, 8) ||
        !d_row_dtype)
        return LHS_ERR_INVALID_ARG;
    if (vocab < 1 || vocab > INT32_MAX || hidden < 1 || n < 0 || !std::isfinite(scale)) return LHS_ERR_INVALID_ARG;
    if (n == 0) return LHS_OK;
    if (!d_ids || !d_out || !d_err || !aligned(d_ids, 4) || !aligned(d_out, 16) || !aligned(d_err, 4))
        return LHS_ERR_INVALID_ARG;
    return cuda_status(launch_embed_mixed(d_data, data_bytes, d_row_offset, d_row_dtype, vocab, hidden, d_ids, n,
                                          scale, d_out, d_err, static_cast<cudaStream_t>(stream)));
}

int lhs_logits_topk_workspace(const lhs_table *t, int32_t batch, int32_t k, int32_t resid_dtype,
                              size_t *bytes) {
    if (!bytes) return LHS_ERR_INVALID_ARG;
    int rc = check_table(t);
    if (rc) return rc;
    if (resid_dtype != LHS_F32 && resid_dtype != LHS_BF16) return LHS_ERR_INVALID_ARG;
    if (batch < 1 || k < 0 || k > kMaxK || k > t->vocab) return LHS_ERR_INVALID_ARG;
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    LmHeadPlan plan;
    rc = plan_lm_head(*t, batch, k, resid_dtype, dev, &plan);
    if (rc) return rc;
    *bytes = plan.bytes;
    return LHS_OK;
}

int lhs_logits_topk_launches(const lhs_table *t, int32_t batch, int32_t k, int32_t resid_dtype,
                             int32_t *launches) {
    if (!launches) return LHS_ERR_INVALID_ARG;
    int rc = check_table(t);
    if (rc) return rc;
    if (resid_dtype != LHS_F32 && resid_dtype != LHS_BF16) return LHS_ERR_INVALID_ARG;
    if (batch < 1 || k < 0 || k > kMaxK || k > t->vocab) return LHS_ERR_INVALID_ARG;
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    LmHeadPlan plan;
    rc = plan_lm_head(*t, batch, k, resid_dtype, dev, &plan);
    if (rc) return rc;
    *launches = lm_head_launches(plan, batch, k == 0);
    return LHS_OK;
}

int lhs_logits_topk(const lhs_table *t, const void *d_resid, int32_t resid_dtype, int32_t batch,
                    int32_t k, float temperature, int32_t *d_ids, float *d_logits, float *d_probs,
                    void *d_ws, size_t ws_bytes, int32_t *d_err, void *stream) {
    int rc = check_lm_head_args(t, d_resid, resid_dtype, batch, k);
    if (rc) return rc;
    if (k < 1 || !std::isfinite(temperature) || !(temperature > 0.0f)) return LHS_ERR_INVALID_ARG;
    if (!d_ids || !d_logits || !d_ws || !d_err || !aligned(d_ids, 4) || !aligned(d_logits, 4) ||
        !aligned(d_ws, 16) || !aligned(d_err, 4) || (d_probs && !aligned(d_probs, 4)))
        return LHS_ERR_INVALID_ARG;
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    LmHeadPlan plan;
    rc = plan_lm_head(*t, batch, k, resid_dtype, dev, &plan);
    if (rc) return rc;
    if (ws_bytes < plan.bytes) return LHS_ERR_BUFFER_TOO_SMALL;
    return cuda_status(launch_lm_head(*t, plan, d_resid, resid_dtype, batch, k, temperature, d_ids,
                                      d_logits, d_probs, nullptr, d_ws, d_err,
                                      static_cast<cudaStream_t>(stream)));
}

int lhs_logits(const lhs_table *t, const void *d_resid, int32_t resid_dtype, int32_t batch,
               float *d_logits, void *d_ws, size_t ws_bytes, int32_t *d_err, void *stream) {
    int rc = check_lm_head_args(t, d_resid, resid_dtype, batch, 0);
    if (rc) return rc;
    if (!d_logits || !d_ws || !d_err || !aligned(d_logits, 4) || !aligned(d_ws, 16) || !aligned(d_err, 4))
        return LHS_ERR_INVALID_ARG;
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    LmHeadPlan plan;
    rc = plan_lm_head(*t, batch, 0, resid_dtype, dev, &plan);
    if (rc) return rc;
    if (ws_bytes < plan.bytes) return LHS_ERR_BUFFER_TOO_SMALL;
    return cuda_status(launch_lm_head(*t, plan, d_resid, resid_dtype, batch, 0, 1.0f, nullptr,
                                      nullptr, nullptr, d_logits, d_ws, d_err,
                                      static_cast<cudaStream_t>(stream)));
}

int64_t lhs_wire_bytes(int32_t fmt, int32_t seq_len, int32_t hidden) {
    if (seq_len < 0 || hidden < 1) return -1;
    const int64_t s = seq_len, h = hidden;
    switch (fmt) {
    case LHS_WIRE_F32: return 16 + s * h * 4;
    case LHS_WIRE_F16: return 16 + s * h * 2;
    case LHS_WIRE_I8: return 16 + s * (h + 8);
    default: return -1;
    }
}

int lhs_wire_encode(int32_t fmt, const void *d_x, int32_t x_dtype, int32_t seq_len, int32_t hidden,
                    uint32_t layer, uint32_t flags, uint32_t top_k, void *d_buf, size_t buf_bytes,
                    int32_t *d_err, void *stream) {
    const int64_t need = lhs_wire_bytes(fmt, seq_len, hidden);
    if (need < 0) return LHS_ERR_INVALID_ARG;
    if (x_dtype != LHS_F32 && x_dtype != LHS_BF16) return LHS_ERR_INVALID_ARG;
    if (!d_buf || !d_err || !aligned(d_buf, 16) || !aligned(d_err, 4)) return LHS_ERR_INVALID_ARG;
    if (seq_len > 0 && (!d_x || !aligned(d_x, 16))) return LHS_ERR_INVALID_ARG;
    if (buf_bytes < static_cast<size_t>(need)) return LHS_ERR_BUFFER_TOO_SMALL;
    const WireHdr hdr = {{layer, static_cast<uint32_t>(seq_len), flags, top_k}, 4};
    return cuda_status(launch_wire_encode(fmt, d_x, x_dtype, seq_len, hidden, hdr, d_buf, d_err,
                                          static_cast<cudaStream_t>(stream)));
}

int lhs_wire_decode(int32_t fmt, const void *d_buf, size_t buf_bytes, int32_t seq_len, int32_t hidden,
                    float *d_x, int32_t *d_err, void *stream) {
    const int64_t need = lhs_wire_bytes(fmt, seq_len, hidden);
    if (need < 0) return LHS_ERR_INVALID_ARG;
    if (!d_buf || !d_err || !aligned(d_buf, 16) || !aligned(d_err, 4)) return LHS_ERR_INVALID_ARG;
    if (seq_len > 0 && (!d_x || !aligned(d_x, 16))) return LHS_ERR_INVALID_ARG;
    if (buf_bytes < static_cast<size_t>(need)) return LHS_ERR_BUFFER_TOO_SMALL;
    return cuda_status(launch_wire_decode(fmt, d_buf, 16, seq_len, hidden, d_x, d_err,
                                          static_cast<cudaStream_t>(stream)));
}

int64_t lhs_wire_response_bytes(int32_t fmt, int32_t seq_len, int32_t hidden) {
    const int64_t request = lhs_wire_bytes(fmt, seq_len, hidden);
    return request < 0 ? -1 : request - 16 + 12;  // a 12-byte header instead of 16
}

int lhs_wire_encode_response(int32_t fmt, const void *d_x, int32_t x_dtype, int32_t seq_len, int32_t hidden,
                             uint32_t layer, float latency_ms, void *d_buf, size_t buf_bytes, int32_t *d_err,
                             void *stream) {
    const int64_t need = lhs_wire_response_bytes(fmt, seq_len, hidden);
    if (need < 0) return LHS_ERR_INVALID_ARG;
    if (x_dtype != LHS_F32 && x_dtype != LHS_BF16) return LHS_ERR_INVALID_ARG;
    if (!d_buf || !d_err || !aligned(d_buf, 4) || !aligned(d_err, 4)) return LHS_ERR_INVALID_ARG;
    if (seq_len > 0 && (!d_x || !aligned(d_x, 16))) return LHS_ERR_INVALID_ARG;
    if (buf_bytes < static_cast<size_t>(need)) return LHS_ERR_BUFFER_TOO_SMALL;
    uint32_t lat;
    memcpy(&lat, &latency_ms, 4);
    const WireHdr hdr = {{layer, static_cast<uint32_t>(seq_len), lat, 0u}, 3};
    return cuda_status(launch_wire_encode(fmt, d_x, x_dtype, seq_len, hidden, hdr, d_buf, d_err,
                                          static_cast<cudaStream_t>(stream)));
}

int lhs_wire_decode_response(int32_t fmt, const void *d_buf, size_t buf_bytes, int32_t seq_len, int32_t hidden,
                             float *d_x, int32_t *d_err, void *stream) {
    const int64_t need = lhs_wire_response_bytes(fmt, seq_len, hidden);
    if (need < 0) return LHS_ERR_INVALID_ARG;
    if (!d_buf || !d_err || !aligned(d_buf, 4) || !aligned(d_err, 4)) return LHS_ERR_INVALID_ARG;
    if (seq_len > 0 && (!d_x || !aligned(d_x, 16))) return LHS_ERR_INVALID_ARG;
    if (buf_bytes < static_cast<size_t>(need)) return LHS_ERR_BUFFER_TOO_SMALL;
    return cuda_status(launch_wire_decode(fmt, d_buf, 12, seq_len, hidden, d_x, d_err,
                                          static_cast<cudaStream_t>(stream)));
}

int lhs_selftest_bounded_wait(int32_t *d_err, int64_t timeout_ns, void *stream) {
    if (!d_err || !aligned(d_err, 4) || timeout_ns < 0 || timeout_ns > 10000000000ll)
        return LHS_ERR_INVALID_ARG;
    return cuda_status(launch_selftest_wait(d_err, timeout_ns, static_cast<cudaStream_t>(stream)));
}

const char *lhs_strerror(int status) {
    switch (status) {
    case LHS_OK: return "ok";
    case LHS_ERR_INVALID_ARG: return "invalid argument";
    case LHS_ERR_BUFFER_TOO_SMALL: return "buffer too small";
    case LHS_ERR_UNSUPPORTED: return "unsupported request";
    case LHS_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
    }
}

int lhs_last_cuda_error(void) { return g_last_cuda_error; }

const char *lhs_version(void) { return "lhs 0.1.0 (sm_103a)"; }

}  // extern "C"
