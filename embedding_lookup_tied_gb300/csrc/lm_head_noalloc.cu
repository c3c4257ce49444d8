// lm_head_noalloc.cu — lhs_logits_topk_noalloc: the lm_head + top-k call
// for callers that cannot hand the library a workspace.
//
// Some callers cannot allocate device memory at the moment they need top-k
// tokens: a plugin running inside a host application that owns the whole
// device memory budget through its own pool and exposes no allocator; or a
// latency-critical loop where a cudaMalloc / cudaFree — which may
// synchronise the device — would stall every other stream.  For them this
// entry point takes its scratch from a fixed array compiled into the
// library instead of from the caller.  The caller still passes the inputs
// and the outputs; nothing here allocates.
#include <mutex>

#include "lhs_internal.cuh"

namespace lhs {
namespace {

// The scratch.  Every GPU that loads this library keeps these bytes
// reserved until the process exits.  Every call shares them and they keep
// the last call's contents; nothing in them has to start at zero, because
// each call writes every scratch byte before it reads it.  Calls that
// overlap on the GPU (different streams, or several host threads without
// ordering) race on this array and corrupt each other's results.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LHS_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_ptr[64] = {};

// Device address of the scratch on the current device.  In host code the
// array's name stands for a host-side shadow, not a device address, so the
// address is looked up once per device (with that device current) and
// cached.
cudaError_t scratch_address(int device, void **out) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[device]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return cudaSuccess;
}

}  // namespace
}  // namespace lhs

extern "C" {

LHS_API int lhs_logits_topk_noalloc(const lhs_table *t, const void *d_resid, int32_t resid_dtype,
                                    int32_t batch, int32_t k, float temperature, int32_t *d_ids,
                                    float *d_logits, float *d_probs, int32_t *d_err, void *stream) {
    size_t need = 0;
    const int rc = lhs_logits_topk_workspace(t, batch, k, resid_dtype, &need);
    if (rc != LHS_OK) return rc;
    if (need > static_cast<size_t>(LHS_NOALLOC_SCRATCH_BYTES)) return LHS_ERR_BUFFER_TOO_SMALL;
    lhs::DeviceInfo dev;
    cudaError_t e = lhs::device_info(&dev);
    void *scratch = nullptr;
    if (e == cudaSuccess) e = lhs::scratch_address(dev.device, &scratch);
    if (e != cudaSuccess) return LHS_ERR_CUDA;
    return lhs_logits_topk(t, d_resid, resid_dtype, batch, k, temperature, d_ids, d_logits, d_probs,
                           scratch, static_cast<size_t>(LHS_NOALLOC_SCRATCH_BYTES), d_err, stream);
}

}  // extern "C"
