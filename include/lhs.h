/*
 * lhs.h — C-ABI of the GB300 embed / tied lm_head service hot path.
 *
 * The library implements the compute behind the embed service described in
 * "ADR-0008 — Remote Embeddings and lm_head Service" (POST /v1/embed,
 * POST /v1/logits, error contract) over the row-addressed table of
 * "HELIX Columnar Embedding — Design Proposal" (§3), with the Q8_0 table and
 * sqrt(hidden) input scale of "embedding-inference — Port Specification"
 * (Tensor inventory, Forward graph), and the residual wire codecs of
 * "ADR-0009 — Wire Format Evolution: f16 Default + i8 Quantised Residuals"
 * (Wire Layout).
 *
 * Conventions shared by every call:
 *  - Pointers named d_* are DEVICE pointers owned by the caller and only
 *    borrowed for the call.  The library allocates no device memory, keeps
 *    no state between calls (beyond per-device kernel attributes set on first
 *    use) and never synchronises: work is enqueued on `stream`
 *    (a cudaStream_t; NULL = the legacy default stream) and the call returns.
 *  - Alignment: tables, embed outputs, residuals, workspaces, wire buffers
 *    and decoded residuals must be 16-byte aligned; id arrays, top-k outputs
 *    and d_err 4-byte aligned.  Violations return LHS_ERR_INVALID_ARG.
 *  - Return value: LHS_OK or a negative LHS_ERR_* for problems detectable on
 *    the host (bad arguments, sizes, unsupported shapes, a failed launch).
 *    Nothing is enqueued when a call returns an error.
 *  - d_err: a device int32 the caller zeroes before the request; kernels
 *    OR LHS_ERRBIT_* bits into it in stream order for data-dependent errors.
 *    Any nonzero bit means the request failed as a whole (the single error
 *    envelope of ADR-0008's error contract).
 *  - Calls are thread-safe; calls on different streams may run concurrently
 *    when they use disjoint outputs and workspaces.
 */
#ifndef LHS_H_
#define LHS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LHS_API __attribute__((visibility("default")))
#else
#define LHS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (host-detectable errors) ----------------------------- */
#define LHS_OK 0
#define LHS_ERR_INVALID_ARG (-1)      /* null pointer, bad size/enum, misalignment */
#define LHS_ERR_BUFFER_TOO_SMALL (-2) /* workspace or wire buffer below the size query */
#define LHS_ERR_UNSUPPORTED (-3)      /* valid request this build does not serve */
#define LHS_ERR_CUDA (-4)             /* a CUDA runtime call or launch failed */

/* ---- data-dependent error bits OR-ed into *d_err ----------------------- */
#define LHS_ERRBIT_BAD_TOKEN 1  /* a token id < 0 or >= vocab; its row is zero */
#define LHS_ERRBIT_MALFORMED 2  /* wire message header / zero_point mismatch */
#define LHS_ERRBIT_NONFINITE 4  /* i8 encode of a non-finite value; f16-table
                                   lm_head residual outside the f16 range */
#define LHS_ERRBIT_TIMEOUT 8    /* a bounded on-device wait gave up */

/* ---- table element types and wire formats ------------------------------ */
typedef enum {
    LHS_F32 = 0,   /* IEEE binary32, little-endian */
    LHS_F16 = 1,   /* IEEE binary16 ("f16 store", ADR-0008 memory footprint) */
    LHS_BF16 = 2,  /* bfloat16 */
    LHS_Q8_0 = 3,  /* blocks of 32: [f16 d (LE)][32 x int8 q], value d*q (Port Spec) */
    LHS_FP8_E4M3 = 4 /* OCP FP8 E4M3: a row type of mixed-precision tables only
                        (lhs_embed_mixed); lhs_table_init rejects it */
} lhs_dtype;

typedef enum {
    LHS_WIRE_F32 = 0, /* application/x-larql-ffn     : binary32 payload      */
    LHS_WIRE_F16 = 1, /* application/x-larql-ffn-f16 : binary16 payload      */
    LHS_WIRE_I8 = 2   /* application/x-larql-ffn-i8  : per position
                         [scale f32][zero_point f32][hidden x int8]          */
} lhs_wire;

/* A static vocab x hidden table, row-major: row i occupies bytes
 * [i*row_bytes, (i+1)*row_bytes) of `data` (HELIX §3; no framing, no
 * index).  row_bytes = hidden*itemsize, or hidden/32*34 for Q8_0.
 * Tied lm_head (ADR-0008, Open Question 1): the same table serves the
 * embedding lookup and the output projection. */
typedef struct {
    const void *data;  /* device pointer, 16-byte aligned, caller-owned */
    int64_t vocab;     /* rows; 1 <= vocab <= 2^31-1 (token ids are int32) */
    int32_t hidden;    /* elements per row; >= 1; multiple of 32 for Q8_0 */
    int32_t dtype;     /* lhs_dtype */
    int64_t row_bytes; /* filled by lhs_table_init */
} lhs_table;

/* Fill *t after checking the arguments.  Does not touch device memory.
 * Errors: LHS_ERR_INVALID_ARG for a null/misaligned pointer, vocab or
 * hidden out of range, unknown dtype, or Q8_0 with hidden % 32 != 0. */
LHS_API int lhs_table_init(lhs_table *t, const void *d_table, int64_t vocab, int32_t hidden,
                   int32_t dtype);

/* The /v1/stats figures of ADR-0008: vocab, hidden, row bytes and table
 * bytes (vocab * row_bytes).  Any output pointer may be NULL. */
LHS_API int lhs_table_info(const lhs_table *t, int64_t *vocab, int32_t *hidden,
                   int64_t *row_bytes, int64_t *total_bytes);

/* Step 1 — embed gather (ADR-0008 POST /v1/embed: one row lookup per token;
 * a prefill of n tokens is n independent lookups, Open Question 2;
 * Port Spec forward graph: x = token_embd[ids] * sqrt(768)).
 *   d_out[t*hidden + j] = f32(element(row ids[t], j) * scale)
 * element() is the exact f32 value stored (f16/bf16 widened; Q8_0 = d*q,
 * exact), then ONE binary32 multiply by `scale` (pass sqrt(hidden) rounded
 * to binary32 for the Gemma profile, 1.0f for an unscaled lookup).
 *   d_ids : int32 [n]            d_out : f32 [n x hidden], row-major
 * An id outside [0, vocab) yields a zero row and LHS_ERRBIT_BAD_TOKEN.
 * n == 0 enqueues nothing.  Errors: LHS_ERR_INVALID_ARG (n < 0, null or
 * misaligned pointers, non-finite scale). */
LHS_API int lhs_embed(const lhs_table *t, const int32_t *d_ids, int64_t n, float scale,
              float *d_out, int32_t *d_err, void *stream);

/* Steps 1+4 fused — the embed lookup written straight into a wire message
 * (ADR-0008 POST /v1/embed: the looked-up rows travel in the same codec as
 * the FFN grid; ADR-0009 Wire Layout).  d_buf receives, byte for byte, what
 * lhs_wire_encode(fmt, x, LHS_F32, n, hidden, layer, flags, top_k, ...)
 * writes for the rows x = lhs_embed(t, d_ids, n, scale): the 16-byte header
 * [layer][n][flags][top_k], then the f32, f16 or per-position i8 payload.
 * The binary32 rows are never materialised.  An id outside [0, vocab) gives
 * a zero row and LHS_ERRBIT_BAD_TOKEN; an i8 position holding inf/NaN is
 * written as scale 0, codes 0 with LHS_ERRBIT_NONFINITE.
 *   0 <= n <= INT32_MAX (n == 0 writes the header only); scale finite;
 *   d_buf 16-byte aligned, buf_bytes >= lhs_wire_bytes(fmt, n, hidden).
 * Errors: LHS_ERR_INVALID_ARG, LHS_ERR_BUFFER_TOO_SMALL, LHS_ERR_CUDA. */
LHS_API int lhs_embed_wire(const lhs_table *t, const int32_t *d_ids, int64_t n, float scale,
                   int32_t fmt, uint32_t layer, uint32_t flags, uint32_t top_k, void *d_buf,
                   size_t buf_bytes, int32_t *d_err, void *stream);

/* lhs_embed_wire writing the single-layer response message instead (the
 * embed service's reply in the FFN grid's codec; ADR-0009 Wire Layout,
 * "Single-layer response"): byte for byte what lhs_wire_encode_response(fmt,
 * x, LHS_F32, n, hidden, layer, latency_ms, ...) writes for the rows
 * x = lhs_embed(t, d_ids, n, scale) — the 12-byte header
 * [layer][n][latency_ms], then the same payload.  d_buf needs 4-byte
 * alignment; one 4 bytes past a 16-byte boundary puts the payload on one
 * and takes the vectorised kernels.  buf_bytes >=
 * lhs_wire_response_bytes(fmt, n, hidden).  Otherwise as lhs_embed_wire. */
LHS_API int lhs_embed_wire_response(const lhs_table *t, const int32_t *d_ids, int64_t n,
                                    float scale, int32_t fmt, uint32_t layer, float latency_ms,
                                    void *d_buf, size_t buf_bytes, int32_t *d_err, void *stream);

/* Dedup (HELIX Columnar Embedding, Appendix B: tokenize, dedupe, then fetch
 * the distinct rows).  For ids d_ids[0..n) and a vocabulary of `vocab` rows:
 *   d_unique  int32 [min(n, vocab)]: the distinct ids in [0, vocab), ascending;
 *             entries past *d_count are left as they were
 *   d_inverse int32 [n]: position of d_ids[i] in d_unique, or -1 for an id
 *             outside [0, vocab) (and LHS_ERRBIT_BAD_TOKEN)
 *   d_count   int32 [1]: number of distinct ids
 * Scratch: lhs_unique_ids_workspace(vocab) bytes (a flag per vocabulary row
 * and per-1024-row sums).  n >= 0.  Errors: LHS_ERR_INVALID_ARG,
 * LHS_ERR_BUFFER_TOO_SMALL, LHS_ERR_CUDA.  No counterpart as a call on the
 * pages: the distinct-id plan the pages describe, as a device step. */
LHS_API int64_t lhs_unique_ids_workspace(int64_t vocab);
LHS_API int lhs_unique_ids(int64_t vocab, const int32_t *d_ids, int64_t n, int32_t *d_unique,
                   int32_t *d_inverse, int32_t *d_count, void *d_ws, size_t ws_bytes,
                   int32_t *d_err, void *stream);

/* lhs_embed through the distinct ids: every distinct row is read, decoded
 * and scaled once (into scratch), then copied to each position that names
 * it.  d_out [n x hidden] f32 equals lhs_embed's output bit for bit, and the
 * error bits are the same.  Scratch: lhs_embed_dedup_workspace(t, n) bytes,
 * 16-byte aligned.  Errors as lhs_embed, plus LHS_ERR_BUFFER_TOO_SMALL. */
LHS_API int64_t lhs_embed_dedup_workspace(const lhs_table *t, int64_t n);
LHS_API int lhs_embed_dedup(const lhs_table *t, const int32_t *d_ids, int64_t n, float scale,
                    float *d_out, void *d_ws, size_t ws_bytes, int32_t *d_err, void *stream);

/* Gather from a mixed-precision table (HELIX Columnar Embedding, §3: the
 * optional sidecar for heterogeneous rows — mixed precision per row, e.g.
 * fp16 for common tokens and fp8 for the long tail, or quantised rows with an
 * inline dequantisation header).  Row r's bytes start at
 * d_data + d_row_offset[r] and hold hidden elements of type d_row_dtype[r]:
 * LHS_F32, LHS_F16, LHS_BF16, LHS_Q8_0 (hidden % 32 == 0) or LHS_FP8_E4M3.
 *   d_out[t*hidden + j] = f32(element(row ids[t], j) * scale)
 * An id outside [0, vocab) gives a zero row and LHS_ERRBIT_BAD_TOKEN; a row
 * with an unknown type, an offset that is not a multiple of its element size
 * (4 for f32, 2 for f16 / bf16 / Q8_0) or bytes outside [0, data_bytes) gives
 * a zero row and LHS_ERRBIT_MALFORMED (nothing outside the data is read).
 * d_data 16-byte aligned; d_out 16-byte aligned.  Errors: LHS_ERR_INVALID_ARG,
 * LHS_ERR_CUDA. */
LHS_API int lhs_embed_mixed(const void *d_data, int64_t data_bytes, const int64_t *d_row_offset,
                    const uint8_t *d_row_dtype, int64_t vocab, int32_t hidden,
                    const int32_t *d_ids, int64_t n, float scale, float *d_out,
                    int32_t *d_err, void *stream);

/* Workspace bytes lhs_logits_topk / lhs_logits need for this table, batch,
 * k (0 for the raw-logits call) and residual dtype.  Depends on the current
 * device's SM count.  Errors as for lhs_logits_topk. */
LHS_API int lhs_logits_topk_workspace(const lhs_table *t, int32_t batch, int32_t k,
                              int32_t resid_dtype, size_t *bytes);

/* Kernel launches one lhs_logits_topk call (k >= 1) or lhs_logits call
 * (k == 0) with these arguments enqueues on the current device: the
 * projection's passes over the table (with the residual-operand prep kernel
 * where one runs, and the batched GEMM's one-thread counter reset) plus,
 * where it runs as a kernel of its own, the cross-CTA merge.  For launch
 * accounting and CUDA-graph sizing; no
 * counterpart in the source pages.  Errors as for
 * lhs_logits_topk_workspace. */
LHS_API int lhs_logits_topk_launches(const lhs_table *t, int32_t batch, int32_t k,
                             int32_t resid_dtype, int32_t *launches);

/* Steps 2+3 — tied lm_head projection with fused top-k (ADR-0008
 * POST /v1/logits: residual @ lm_head.T over every vocab row, top_k entries
 * {token_id, prob}; HELIX §5: the projection needs all vocab rows).
 *   logit[b][v] = sum_j element(row v, j) * x[b][j], f32 accumulation
 *   d_resid : [batch x hidden] of resid_dtype (LHS_F32 or LHS_BF16)
 *   d_ids   : int32 [batch x k]  token ids, logit descending, equal logits by
 *             id ascending (a NaN logit ranks above every number)
 *   d_logits: f32 [batch x k]    the selected logits
 *   d_probs : f32 [batch x k] or NULL: softmax(logit / temperature) over the
 *             FULL vocabulary, evaluated for the selected ids
 * The full logits vector is never written.  1 <= k <= min(128, vocab);
 * temperature finite and > 0; batch >= 1.  d_ws/ws_bytes: caller-owned
 * scratch of at least lhs_logits_topk_workspace() bytes; its contents on
 * entry do not matter and are overwritten.  Errors: LHS_ERR_INVALID_ARG,
 * LHS_ERR_BUFFER_TOO_SMALL, LHS_ERR_UNSUPPORTED (table dtype / residual
 * dtype pair not served), LHS_ERR_CUDA.  An f16 table with a residual whose
 * magnitude reaches 65504 sets LHS_ERRBIT_NONFINITE.  A bf16 table with
 * more than 8 bf16 residuals runs one kernel of one CTA per SM whose CTAs
 * exchange a top-k bound: kernels holding SMs on other streams hold that
 * exchange back (for at most 2 s, after which it goes on without the bound,
 * with the same results). */
LHS_API int lhs_logits_topk(const lhs_table *t, const void *d_resid, int32_t resid_dtype,
                    int32_t batch, int32_t k, float temperature, int32_t *d_ids,
                    float *d_logits, float *d_probs, void *d_ws, size_t ws_bytes,
                    int32_t *d_err, void *stream);

/* Raw-logits mode (ADR-0008 POST /v1/logits, "raw logits mode for beam
 * search / sampling"): d_logits f32 [batch x vocab].  Computed by the same
 * kernels and in the same summation order as lhs_logits_topk, so the top-k
 * of these logits equals the fused call's result bit for bit.  Workspace:
 * lhs_logits_topk_workspace(t, batch, 0, resid_dtype, ...). */
LHS_API int lhs_logits(const lhs_table *t, const void *d_resid, int32_t resid_dtype,
               int32_t batch, float *d_logits, void *d_ws, size_t ws_bytes,
               int32_t *d_err, void *stream);

/* Bytes of the fixed scratch array lhs_logits_topk_noalloc uses (4 MiB). */
#define LHS_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)

/* lhs_logits_topk for callers that cannot allocate device memory where they
 * need top-k tokens — a plugin inside an application that owns the whole
 * device memory budget through its own pool, or a latency-critical loop in
 * which cudaMalloc/cudaFree (which may synchronise the device) is not
 * acceptable.  No counterpart in the source pages (the paper): this is an
 * interface convenience, not part of the method.
 * Same arguments, results and errors as lhs_logits_topk minus the
 * workspace: the scratch is an array of LHS_NOALLOC_SCRATCH_BYTES compiled
 * into the library (each GPU that loads the library holds it until exit).
 * A request whose lhs_logits_topk_workspace() size exceeds that limit
 * returns LHS_ERR_BUFFER_TOO_SMALL and enqueues nothing (with 152 SMs, every
 * batch <= 8 with k <= 128 and hidden <= 65536 fits, and so does a batched
 * bf16 call of up to 50 residuals with k <= 96, or 26 with a larger k).  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress, with that
 * device current), and so does the first call after the device's context
 * has changed (cudaDeviceReset): make those first calls before any stream
 * capture.  Allocates nothing.  All calls share the one array and it keeps
 * the last call's contents (no part of it needs to start at zero); calls
 * that overlap on the GPU — different streams or unordered host threads —
 * race on it: serialise them. */
LHS_API int lhs_logits_topk_noalloc(const lhs_table *t, const void *d_resid,
                                    int32_t resid_dtype, int32_t batch, int32_t k,
                                    float temperature, int32_t *d_ids, float *d_logits,
                                    float *d_probs, int32_t *d_err, void *stream);

/* Step 4 — residual wire codecs (ADR-0009 Wire Layout).
 * Message = 16-byte header [layer u32][seq_len u32][flags u32][top_k u32]
 * (little-endian) followed by the payload:
 *   LHS_WIRE_F32: binary32[seq_len*hidden]
 *   LHS_WIRE_F16: binary16[seq_len*hidden]; round to nearest even; a finite
 *                 value beyond the f16 range saturates to +-65504
 *                 (ADR-0009 Trade-offs, clamp-to-max); inf stays inf; NaN
 *                 becomes 0x7E00
 *   LHS_WIRE_I8 : per position [scale f32][zero_point f32 = 0][int8 x hidden],
 *                 scale = f32(max|x| / 127), q = clamp(rne(f32(x / scale)),
 *                 -127, 127); decode x^ = f32(q * scale).  An all-zero
 *                 position has scale 0.  A position with a non-finite value
 *                 sets LHS_ERRBIT_NONFINITE and is written as scale 0, q 0.
 * lhs_wire_bytes returns the message size, or -1 for bad arguments. */
LHS_API int64_t lhs_wire_bytes(int32_t fmt, int32_t seq_len, int32_t hidden);

/* Encode d_x [seq_len x hidden] of x_dtype (LHS_F32 or LHS_BF16) into d_buf
 * (buf_bytes >= lhs_wire_bytes).  Errors: LHS_ERR_INVALID_ARG,
 * LHS_ERR_BUFFER_TOO_SMALL, LHS_ERR_CUDA. */
LHS_API int lhs_wire_encode(int32_t fmt, const void *d_x, int32_t x_dtype, int32_t seq_len,
                    int32_t hidden, uint32_t layer, uint32_t flags, uint32_t top_k,
                    void *d_buf, size_t buf_bytes, int32_t *d_err, void *stream);

/* Decode d_buf into d_x f32 [seq_len x hidden].  If the header's seq_len
 * differs from `seq_len`, LHS_ERRBIT_MALFORMED is set and d_x is not
 * written.  For i8, a position whose zero_point is not 0 is flagged
 * LHS_ERRBIT_MALFORMED and left unwritten.  Errors: LHS_ERR_INVALID_ARG,
 * LHS_ERR_BUFFER_TOO_SMALL (buf_bytes < lhs_wire_bytes), LHS_ERR_CUDA. */
LHS_API int lhs_wire_decode(int32_t fmt, const void *d_buf, size_t buf_bytes, int32_t seq_len,
                    int32_t hidden, float *d_x, int32_t *d_err, void *stream);

/* Step 4, response side — the single-layer response message ("ADR-0009 —
 * Wire Format Evolution", Wire Layout, "Single-layer response"): a 12-byte
 * header [layer u32][seq_len u32][latency_ms f32] (little-endian) followed
 * by the same payload as the request message of the same format (binary32,
 * binary16, or the i8 positions, with the same rounding, saturation and
 * error rules).  lhs_wire_response_bytes returns 12 + the payload bytes, or
 * -1 for bad arguments. */
LHS_API int64_t lhs_wire_response_bytes(int32_t fmt, int32_t seq_len, int32_t hidden);

/* Encode d_x [seq_len x hidden] of x_dtype (LHS_F32 or LHS_BF16) as a
 * response message in d_buf (buf_bytes >= lhs_wire_response_bytes).  d_buf
 * needs 4-byte alignment only; the payload starts 12 bytes in, so a buffer
 * that starts 4 bytes past a 16-byte boundary puts it on one and takes the
 * vectorised kernels (any other 4-byte-aligned buffer takes element-wise
 * ones, with the same bytes).  d_x must be 16-byte aligned.  Errors as for
 * lhs_wire_encode. */
LHS_API int lhs_wire_encode_response(int32_t fmt, const void *d_x, int32_t x_dtype,
                                     int32_t seq_len, int32_t hidden, uint32_t layer,
                                     float latency_ms, void *d_buf, size_t buf_bytes,
                                     int32_t *d_err, void *stream);

/* Decode a response message (d_buf 4-byte aligned, d_x 16-byte aligned)
 * into d_x f32 [seq_len x hidden], with lhs_wire_decode's checks: a header
 * seq_len other than `seq_len` sets LHS_ERRBIT_MALFORMED and leaves d_x
 * unwritten; an i8 position whose zero_point is not 0 is flagged and left
 * unwritten.  Errors as for lhs_wire_decode (against
 * lhs_wire_response_bytes). */
LHS_API int lhs_wire_decode_response(int32_t fmt, const void *d_buf, size_t buf_bytes,
                                     int32_t seq_len, int32_t hidden, float *d_x,
                                     int32_t *d_err, void *stream);

/* Diagnostic: launch one tiny kernel whose wait on an on-chip barrier is
 * never satisfied, bounded by timeout_ns; the kernel gives up, sets
 * LHS_ERRBIT_TIMEOUT in *d_err and exits normally.  This exercises the same
 * bounded-wait routine the lm_head pipeline uses, without a hang. */
LHS_API int lhs_selftest_bounded_wait(int32_t *d_err, int64_t timeout_ns, void *stream);

/* Message for a status code; never NULL. */
LHS_API const char *lhs_strerror(int status);

/* The cudaError_t of the last LHS_ERR_CUDA returned on this host thread. */
LHS_API int lhs_last_cuda_error(void);

/* Library version string. */
LHS_API const char *lhs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LHS_H_ */
