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

// The array's device address is a property of a CUDA context: after a
// cudaDeviceReset the device's next (primary) context places the array
// anew.  So the cached address is keyed by the current context's
// process-unique id (cuCtxGetId), read through driver entry points that the
// runtime hands out (the library does not link the driver library itself).
// Without those entry points every call looks the address up again.
struct ScratchSlot {
    void *ptr;
    unsigned long long ctx_id;
    bool have_id;
};
ScratchSlot g_slot[64] = {};

typedef int (*CtxGetCurrentFn)(void **);
typedef int (*CtxGetIdFn)(void *, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_entry_once;

void load_entry_points() {
    void *f = nullptr, *g = nullptr;
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &g, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess && f && g) {
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(g);
    }
    (void)cudaGetLastError();
}

// Id of the calling thread's current context; false when there is none yet
// or the driver entry points are unavailable.
bool current_ctx_id(unsigned long long *id) {
    if (!g_ctx_get_current || !g_ctx_get_id) return false;
    void *ctx = nullptr;
    if (g_ctx_get_current(&ctx) != 0 || !ctx) return false;
    return g_ctx_get_id(ctx, id) == 0;
}

// Device address of the scratch in the current context of `device` (the
// current device).  In host code the array's name stands for a host-side
// shadow, not a device address: the address comes from
// cudaGetSymbolAddress, made with the device current, once per context.
cudaError_t scratch_address(int device, void **out) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::call_once(g_entry_once, load_entry_points);
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchSlot &s = g_slot[device];
    unsigned long long id = 0;
    if (s.ptr && s.have_id && current_ctx_id(&id) && id == s.ctx_id) {
        *out = s.ptr;
        return cudaSuccess;
    }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    // the lookup made the device's primary context current if none was
    s.ptr = p;
    s.have_id = current_ctx_id(&s.ctx_id);
    *out = p;
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
    if (e != cudaSuccess) return lhs::cuda_status(e);
    return lhs_logits_topk(t, d_resid, resid_dtype, batch, k, temperature, d_ids, d_logits, d_probs,
                           scratch, static_cast<size_t>(LHS_NOALLOC_SCRATCH_BYTES), d_err, stream);
}

}  // extern "C"
