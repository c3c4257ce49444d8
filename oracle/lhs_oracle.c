/*
 * lhs_oracle.c — the ORACLE for the embed / tied lm_head service hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it and shares no code,
 * header, table or constant with it.
 *
 * Plain, slow, obviously correct C.  Floating-point results that the service
 * must reproduce bit-for-bit (gather, dequant, wire codecs, top-k order) are
 * computed with single IEEE-754 binary32 operations written out exactly as the
 * definitions state; the lm_head projection is accumulated in binary64.
 * Compile with -O2 -ffp-contract=off and without fast-math so that every f32
 * operation below is one correctly rounded IEEE operation.
 *
 * Sources (page title, section):
 *   [ADR-0008] "ADR-0008 — Remote Embeddings and lm_head Service":
 *              POST /v1/embed, POST /v1/logits, Error contract,
 *              Open Questions 1 (tied weights) and 2 (batch embed).
 *   [HELIX]    "HELIX Columnar Embedding — Design Proposal":
 *              §3 Architecture (row-aligned file, row i at i*row_bytes),
 *              §5 Handling lm_head.
 *   [PORT]     "embedding-inference — Port Specification":
 *              Tensor inventory (Q8_0 token_embd, row-gather + dequant) and
 *              Forward graph (x = token_embd[ids] * sqrt(768)).
 *   [ADR-0009] "ADR-0009 — Wire Format Evolution: f16 Default + i8 Quantised
 *              Residuals": Wire Layout (f16, i8 symmetric), Trade-offs
 *              (f16 clamp-to-max on overflow).
 *
 * Readings where the pages leave a step open are listed next to the code that
 * takes them; every reading is also listed in the design notes.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

/* Table element types (the oracle's own numbering; the public header uses
 * the same values because both follow the same documented enumeration). */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_Q8_0 = 3, ORC_FP8_E4M3 = 4 };
/* Wire formats: [ADR-0009] Decision table — f32, f16, i8. */
enum { ORC_WIRE_F32 = 0, ORC_WIRE_F16 = 1, ORC_WIRE_I8 = 2 };
/* Data-dependent error bits ([ADR-0008] Error contract: bad token ids,
 * malformed binary payloads). */
enum { ORC_ERR_BAD_TOKEN = 1, ORC_ERR_MALFORMED = 2, ORC_ERR_NONFINITE = 4 };

/* Q8_0 block: 32 signed 8-bit codes sharing one f16 scale d ([PORT] Tensor
 * inventory).  Reading: the block is 34 bytes, d (little-endian f16) first,
 * then q[0..31]; element value = d * q. */
#define ORC_Q8_BLOCK 32
#define ORC_Q8_BLOCK_BYTES 34

/* ------------------------------------------------------------------------- */
/* IEEE 754 binary16 / bfloat16 decoding                                     */
/* ------------------------------------------------------------------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Returns the exact value as a double (every binary16 value is exact in
 * binary64). */
double orc_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of a binary32 pattern. */
float orc_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static float orc_f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t orc_bits_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* Round a non-negative double holding an exact value to the nearest integer,
 * ties to even. */
static double orc_round_half_even(double n)
{
    double fl = floor(n);
    double d = n - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* f32 -> binary16 for the f16 wire ([ADR-0009] Wire Layout, f16; Trade-offs).
 * Round to nearest, ties to even.  Reading of "clamp-to-max behaviour of f16
 * overflow (not NaN for normal finite values)": a finite input whose rounded
 * magnitude would overflow (|x| >= 65520) becomes +-65504; infinities stay
 * infinities; any NaN becomes the quiet NaN 0x7E00. */
uint16_t orc_f16_from_f32_sat(float x)
{
    uint16_t sign;
    double a, quantum, n;
    int E;
    if (isnan(x)) return 0x7E00;
    sign = signbit(x) ? 0x8000 : 0;
    if (isinf(x)) return sign | 0x7C00;
    a = fabs((double)x);
    if (a >= 65520.0) return sign | 0x7BFF;      /* saturate to 65504 */
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: spacing 2^-24, field = round(a / 2^-24); a result
         * of 1024 is exactly the smallest normal 0x0400. */
        n = orc_round_half_even(a / ldexp(1.0, -24));
        return sign | (uint16_t)n;
    }
    frexp(a, &E);                                /* a = f * 2^E, f in [0.5,1) */
    quantum = ldexp(1.0, (E - 1) - 10);          /* 10 fraction bits */
    n = orc_round_half_even(a / quantum);        /* in [1024, 2048] */
    {
        int expo = (E - 1) + 15;
        int mant = (int)n;
        if (mant == 2048) { mant = 1024; expo += 1; }
        return sign | (uint16_t)((expo << 10) | (mant - 1024));
    }
}

/* ------------------------------------------------------------------------- */
/* Table layout: [HELIX] §3 — row i occupies bytes [i*row_bytes,            */
/* (i+1)*row_bytes), row_bytes = hidden * itemsize, no framing, no index.    */
/* ------------------------------------------------------------------------- */

int64_t orc_row_bytes(int dtype, int32_t hidden)
{
    switch (dtype) {
    case ORC_F32: return (int64_t)hidden * 4;
    case ORC_F16:
    case ORC_BF16: return (int64_t)hidden * 2;
    case ORC_Q8_0:
        if (hidden % ORC_Q8_BLOCK) return -1;
        return (int64_t)(hidden / ORC_Q8_BLOCK) * ORC_Q8_BLOCK_BYTES;
    default: return -1;
    }
}

static uint16_t orc_load_u16le(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

static uint32_t orc_load_u32le(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

static void orc_store_u32le(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)(v & 0xff);
    p[1] = (uint8_t)((v >> 8) & 0xff);
    p[2] = (uint8_t)((v >> 16) & 0xff);
    p[3] = (uint8_t)((v >> 24) & 0xff);
}

/* Element j of a table row, as the f32 value the row stores ([ADR-0008]
 * f16-at-rest store decoded per lookup; [PORT] q8_0 row dequant).
 * Q8_0: d * q is exact in binary32 (11-bit by 8-bit significands). */
static float orc_row_element(const uint8_t *row, int dtype, int32_t j)
{
    switch (dtype) {
    case ORC_F32: return orc_f32_from_bits(orc_load_u32le(row + 4 * (size_t)j));
    case ORC_F16: return (float)orc_f16_value(orc_load_u16le(row + 2 * (size_t)j));
    case ORC_BF16: return orc_bf16_value(orc_load_u16le(row + 2 * (size_t)j));
    case ORC_Q8_0: {
        const uint8_t *blk = row + (size_t)(j / ORC_Q8_BLOCK) * ORC_Q8_BLOCK_BYTES;
        double d = orc_f16_value(orc_load_u16le(blk));
        int q = (int)(int8_t)blk[2 + (j % ORC_Q8_BLOCK)];
        return (float)(d * (double)q);
    }
    default: return NAN;
    }
}

/* ------------------------------------------------------------------------- */
/* Step 1 — embed gather + dequant + scale                                   */
/* [ADR-0008] POST /v1/embed: one row lookup per token id, N lookups for a   */
/* prefill of N tokens (Open Question 2); the per-lookup cost is a copy plus */
/* a scalar multiply (Measured Performance, embed lookup).                   */
/* [PORT] Forward graph: x = token_embd[ids] * sqrt(768).                    */
/* out[t][j] = f32(element(T[ids[t]], j) * scale).  A token id outside      */
/* [0, vocab) is an error ([ADR-0008] Error contract): its output row is    */
/* zero and the BAD_TOKEN bit is set.                                        */
/* ------------------------------------------------------------------------- */

int orc_embed(const uint8_t *table, int dtype, int64_t vocab, int32_t hidden,
              int64_t row_bytes, const int32_t *ids, int64_t n, float scale,
              float *out, int32_t *err_bits)
{
    int64_t t;
    int32_t j;
    if (orc_row_bytes(dtype, hidden) < 0 || row_bytes != orc_row_bytes(dtype, hidden))
        return -1;
    for (t = 0; t < n; ++t) {
        int64_t id = ids[t];
        float *o = out + t * (int64_t)hidden;
        if (id < 0 || id >= vocab) {
            for (j = 0; j < hidden; ++j) o[j] = 0.0f;
            *err_bits |= ORC_ERR_BAD_TOKEN;
            continue;
        }
        {
            const uint8_t *row = table + id * row_bytes;
            for (j = 0; j < hidden; ++j) {
                float e = orc_row_element(row, dtype, j);
                o[j] = e * scale;                 /* one binary32 multiply */
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Mixed-precision rows ([HELIX] §3, optional sidecar embed-rows.idx: rows   */
/* of one table stored at different precisions, e.g. fp16 for common tokens */
/* and fp8 for the long tail, or quantised rows with their dequantisation    */
/* header inline).  Reading: the sidecar gives, per row, its byte offset in  */
/* the data and its element type; "fp8" is the OCP 8-bit E4M3 format.        */
/* ------------------------------------------------------------------------- */

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 * infinities; exponent and fraction all ones is NaN.  Exact in binary64. */
double orc_fp8_e4m3_value(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int m = c & 0x7;
    double v;
    if (e == 15 && m == 7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -9);                /* subnormal: (m/8) * 2^-6 */
    } else {
        v = ldexp((double)(8 + m), e - 10);      /* (1 + m/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

int64_t orc_mixed_row_bytes(int dtype, int32_t hidden)
{
    if (dtype == ORC_FP8_E4M3) return hidden > 0 ? (int64_t)hidden : -1;
    return orc_row_bytes(dtype, hidden);
}

/* out[t][j] = f32(element(row ids[t], j) * scale) where row r is decoded
 * with its own type row_dtype[r] from data + row_offset[r].  A bad id gives a
 * zero row and BAD_TOKEN; a row whose type code is not a row type gives a
 * zero row and MALFORMED. */
void orc_embed_mixed(const uint8_t *data, int64_t data_bytes, const int64_t *row_offset,
                     const uint8_t *row_dtype, int64_t vocab, int32_t hidden, const int32_t *ids,
                     int64_t n, float scale, float *out, int32_t *err_bits)
{
    int64_t t;
    int32_t j;
    for (t = 0; t < n; ++t) {
        int64_t id = ids[t];
        float *o = out + t * (int64_t)hidden;
        int dt;
        const uint8_t *row;
        if (id < 0 || id >= vocab) {
            for (j = 0; j < hidden; ++j) o[j] = 0.0f;
            *err_bits |= ORC_ERR_BAD_TOKEN;
            continue;
        }
        dt = row_dtype[id];
        /* Reading: a row whose type is unknown, whose offset is not a
         * multiple of its element size (4 bytes f32, 2 bytes f16 / bf16 /
         * Q8_0) or whose bytes fall outside the data is malformed. */
        if (dt < ORC_F32 || dt > ORC_FP8_E4M3 || orc_mixed_row_bytes(dt, hidden) < 0 ||
            row_offset[id] < 0 || row_offset[id] > data_bytes - orc_mixed_row_bytes(dt, hidden) ||
            row_offset[id] % (dt == ORC_F32 ? 4 : (dt == ORC_FP8_E4M3 ? 1 : 2)) != 0) {
            for (j = 0; j < hidden; ++j) o[j] = 0.0f;
            *err_bits |= ORC_ERR_MALFORMED;
            continue;
        }
        row = data + row_offset[id];
        for (j = 0; j < hidden; ++j) {
            float e = dt == ORC_FP8_E4M3 ? (float)orc_fp8_e4m3_value(row[j]) : orc_row_element(row, dt, j);
            o[j] = e * scale;                     /* one binary32 multiply */
        }
    }
}

/* Decode whole tables / residual arrays to f32 (test convenience). */
void orc_decode_rows(const uint8_t *table, int dtype, int32_t hidden,
                     int64_t row_bytes, int64_t row0, int64_t nrows, float *out)
{
    int64_t r;
    int32_t j;
    for (r = 0; r < nrows; ++r) {
        const uint8_t *row = table + (row0 + r) * row_bytes;
        for (j = 0; j < hidden; ++j)
            out[r * hidden + j] = orc_row_element(row, dtype, j);
    }
}

void orc_decode_bf16_array(const uint16_t *src, int64_t n, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_bf16_value(src[i]);
}

void orc_decode_f16_array(const uint16_t *src, int64_t n, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = (float)orc_f16_value(src[i]);
}

/* ------------------------------------------------------------------------- */
/* Step 2 — tied lm_head projection                                          */
/* [ADR-0008] POST /v1/logits: residual @ lm_head.T over every vocab row;    */
/* Open Question 1: the tied lm_head is the embedding table itself.         */
/* [HELIX] §5: logits = hidden @ lm_head.T needs all vocab rows.             */
/* logit[b][v] = sum_j T[v][j] * x[b][j], accumulated in binary64 (each      */
/* product of two binary32 values is exact in binary64).  The optional     */
/* sumabs[b][v] = sum_j |T[v][j] * x[b][j]| is the scale of the rounding    */
/* error any summation order can make, used for tolerances.                  */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint8_t *table;
    int dtype;
    int32_t hidden;
    int64_t row_bytes;
    const float *x;
    int32_t batch;
    double *out;
    double *sumabs;
    int64_t base, ld;  /* output row (v0 of the call) and row stride */
    int64_t v0, v1;    /* this worker's rows */
} orc_logits_job;

static void *orc_logits_worker(void *arg)
{
    orc_logits_job *jb = (orc_logits_job *)arg;
    float *rowf = (float *)malloc(sizeof(float) * (size_t)jb->hidden);
    int64_t v;
    int32_t b, j;
    if (!rowf) return (void *)1;
    for (v = jb->v0; v < jb->v1; ++v) {
        const uint8_t *row = jb->table + v * jb->row_bytes;
        for (j = 0; j < jb->hidden; ++j) rowf[j] = orc_row_element(row, jb->dtype, j);
        for (b = 0; b < jb->batch; ++b) {
            const float *xb = jb->x + (int64_t)b * jb->hidden;
            double acc = 0.0, aacc = 0.0;
            for (j = 0; j < jb->hidden; ++j) {
                double p = (double)rowf[j] * (double)xb[j];
                acc += p;
                aacc += fabs(p);
            }
            jb->out[(int64_t)b * jb->ld + (v - jb->base)] = acc;
            if (jb->sumabs) jb->sumabs[(int64_t)b * jb->ld + (v - jb->base)] = aacc;
        }
    }
    free(rowf);
    return NULL;
}

/* Rows [v0, v1) of the logits, written to out[b*(v1-v0) + (v-v0)];
 * nthreads splits the rows into contiguous ranges (a plain partition,
 * results do not depend on it). */
int orc_logits(const uint8_t *table, int dtype, int64_t vocab, int32_t hidden,
               int64_t row_bytes, const float *x, int32_t batch, int64_t v0,
               int64_t v1, double *out, double *sumabs, int nthreads)
{
    orc_logits_job jobs[256];
    pthread_t th[256];
    int t, rc = 0;
    int64_t span;
    if (row_bytes != orc_row_bytes(dtype, hidden)) return -1;
    if (v0 < 0 || v1 > vocab || v0 > v1) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    span = (v1 - v0 + nthreads - 1) / nthreads;
    for (t = 0; t < nthreads; ++t) {
        jobs[t].table = table;
        jobs[t].dtype = dtype;
        jobs[t].hidden = hidden;
        jobs[t].row_bytes = row_bytes;
        jobs[t].x = x;
        jobs[t].batch = batch;
        jobs[t].out = out;
        jobs[t].sumabs = sumabs;
        jobs[t].base = v0;
        jobs[t].ld = v1 - v0;
        jobs[t].v0 = v0 + t * span;
        jobs[t].v1 = v0 + (t + 1) * span;
        if (jobs[t].v0 > v1) jobs[t].v0 = v1;
        if (jobs[t].v1 > v1) jobs[t].v1 = v1;
    }
    if (nthreads == 1) return orc_logits_worker(&jobs[0]) ? -2 : 0;
    for (t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, orc_logits_worker, &jobs[t])) return -2;
    for (t = 0; t < nthreads; ++t) {
        void *r = NULL;
        pthread_join(th[t], &r);
        if (r) rc = -2;
    }
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Step 3 — top-k selection ([ADR-0008] POST /v1/logits: top_k entries of    */
/* {token_id, prob}).  Reading: entries are ordered by logit descending,     */
/* equal logits by token id ascending; +0 and -0 are equal; a NaN logit      */
/* ranks above every number.  Brute force: k passes of "best remaining".    */
/* ------------------------------------------------------------------------- */

static int orc_ranks_before_f64(double a, int64_t ia, double b, int64_t ib)
{
    int an = isnan(a), bn = isnan(b);
    if (an || bn) {
        if (an && bn) return ia < ib;
        return an;
    }
    if (a > b) return 1;
    if (a < b) return 0;
    return ia < ib;
}

static int orc_topk_generic(const float *lf, const double *ld, int64_t V,
                            int32_t k, int32_t *ids, double *vals)
{
    unsigned char *taken;
    int32_t r;
    int64_t v;
    if (k < 0 || k > V) return -1;
    taken = (unsigned char *)calloc((size_t)(V > 0 ? V : 1), 1);
    if (!taken) return -2;
    for (r = 0; r < k; ++r) {
        int64_t best = -1;
        double bv = 0.0;
        for (v = 0; v < V; ++v) {
            double cv;
            if (taken[v]) continue;
            cv = lf ? (double)lf[v] : ld[v];
            if (best < 0 || orc_ranks_before_f64(cv, v, bv, best)) {
                best = v;
                bv = cv;
            }
        }
        taken[best] = 1;
        ids[r] = (int32_t)best;
        vals[r] = bv;
    }
    free(taken);
    return 0;
}

int orc_topk_f32(const float *logits, int64_t V, int32_t k, int32_t *ids, float *vals)
{
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    int32_t i;
    int rc;
    if (!tmp) return -2;
    rc = orc_topk_generic(logits, NULL, V, k, ids, tmp);
    for (i = 0; rc == 0 && i < k; ++i) vals[i] = (float)tmp[i];
    free(tmp);
    return rc;
}

int orc_topk_f64(const double *logits, int64_t V, int32_t k, int32_t *ids, double *vals)
{
    return orc_topk_generic(NULL, logits, V, k, ids, vals);
}

/* prob of the selected tokens ([ADR-0008] POST /v1/logits: prob, temperature).
 * Reading: prob = softmax(logit / temperature) over the FULL vocabulary:
 * prob(id) = exp((L_id - M)/T) / sum_v exp((L_v - M)/T), M = max_v L_v,
 * evaluated in binary64. */
int orc_softmax_probs(const float *logits, int64_t V, double temperature,
                      const int32_t *ids, int32_t k, double *probs)
{
    double M = -INFINITY, S = 0.0;
    int64_t v;
    int32_t i;
    if (!(temperature > 0.0) || V <= 0) return -1;
    for (v = 0; v < V; ++v)
        if ((double)logits[v] > M) M = (double)logits[v];
    for (v = 0; v < V; ++v) S += exp(((double)logits[v] - M) / temperature);
    for (i = 0; i < k; ++i)
        probs[i] = exp(((double)logits[ids[i]] - M) / temperature) / S;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Step 4 — residual wire codecs ([ADR-0009] Wire Layout).                   */
/* Request message: [layer u32][seq_len u32][flags u32][top_k u32] (LE),    */
/* then the payload:                                                         */
/*   f32: seq_len*hidden binary32 LE (the unchanged format)                  */
/*   f16: seq_len*hidden binary16 LE                                         */
/*   i8 : per position [scale f32 LE][zero_point f32 LE][hidden x int8]     */
/* i8 quantisation: symmetric, zero_point = 0, scale = max|x| / 127,         */
/* dequantise x^ = q * scale.                                                */
/* ------------------------------------------------------------------------- */

#define ORC_WIRE_HEADER 16

int64_t orc_wire_bytes(int fmt, int32_t seq_len, int32_t hidden)
{
    int64_t s = seq_len, h = hidden;
    if (seq_len < 0 || hidden <= 0) return -1;
    switch (fmt) {
    case ORC_WIRE_F32: return ORC_WIRE_HEADER + s * h * 4;
    case ORC_WIRE_F16: return ORC_WIRE_HEADER + s * h * 2;
    case ORC_WIRE_I8: return ORC_WIRE_HEADER + s * (8 + h);
    default: return -1;
    }
}

/* Round a binary32 value to the nearest integer, ties to even.  |y| <= 2^23
 * here, so y - floor(y) is exact. */
static float orc_rne_f32(float y)
{
    float fl = floorf(y);
    float d = y - fl;
    if (d > 0.5f) return fl + 1.0f;
    if (d < 0.5f) return fl;
    return (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

/* One position of the i8 codec.  Readings: q = round-half-even of the
 * binary32 quotient x / scale (scale as stored), clamped to [-127, 127];
 * an all-zero position has scale 0 and codes 0; a position holding a
 * non-finite value sets NONFINITE and is written as scale 0, codes 0. */
static void orc_i8_encode_position(const float *x, int32_t hidden, uint8_t *dst,
                                   int32_t *err_bits)
{
    float m = 0.0f, scale;
    int32_t j;
    int nonfinite = 0;
    for (j = 0; j < hidden; ++j) {
        float a = fabsf(x[j]);
        if (!isfinite(x[j])) nonfinite = 1;
        else if (a > m) m = a;
    }
    if (nonfinite) {
        *err_bits |= ORC_ERR_NONFINITE;
        scale = 0.0f;
    } else {
        scale = m / 127.0f;                        /* binary32 division */
    }
    orc_store_u32le(dst, orc_bits_from_f32(scale));
    orc_store_u32le(dst + 4, orc_bits_from_f32(0.0f)); /* zero_point */
    for (j = 0; j < hidden; ++j) {
        int q = 0;
        if (scale != 0.0f) {
            float y = x[j] / scale;                /* binary32 division */
            float r = orc_rne_f32(y);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q = (int)r;
        }
        dst[8 + j] = (uint8_t)(int8_t)q;
    }
}

int orc_wire_encode(int fmt, const float *x, int32_t seq_len, int32_t hidden,
                    uint32_t layer, uint32_t flags, uint32_t top_k,
                    uint8_t *buf, int32_t *err_bits)
{
    int64_t p, j, n = (int64_t)seq_len * hidden;
    if (orc_wire_bytes(fmt, seq_len, hidden) < 0) return -1;
    orc_store_u32le(buf + 0, layer);
    orc_store_u32le(buf + 4, (uint32_t)seq_len);
    orc_store_u32le(buf + 8, flags);
    orc_store_u32le(buf + 12, top_k);
    if (fmt == ORC_WIRE_F32) {
        for (j = 0; j < n; ++j) orc_store_u32le(buf + 16 + 4 * j, orc_bits_from_f32(x[j]));
    } else if (fmt == ORC_WIRE_F16) {
        for (j = 0; j < n; ++j) {
            uint16_t h = orc_f16_from_f32_sat(x[j]);
            buf[16 + 2 * j] = (uint8_t)(h & 0xff);
            buf[16 + 2 * j + 1] = (uint8_t)(h >> 8);
        }
    } else {
        for (p = 0; p < seq_len; ++p)
            orc_i8_encode_position(x + p * hidden, hidden,
                                   buf + 16 + p * (8 + (int64_t)hidden), err_bits);
    }
    return 0;
}

/* Decode.  Readings: the header's seq_len must equal the caller's seq_len,
 * otherwise MALFORMED is set and x is left untouched; for i8, a position
 * whose zero_point is not 0 is not the symmetric format, so it sets
 * MALFORMED and that position is left untouched (the others decode). */
int orc_wire_decode(int fmt, const uint8_t *buf, int64_t buf_bytes, int32_t seq_len,
                    int32_t hidden, float *x, int32_t *err_bits)
{
    int64_t need = orc_wire_bytes(fmt, seq_len, hidden);
    int64_t p, j, n = (int64_t)seq_len * hidden;
    if (need < 0) return -1;
    if (buf_bytes < need) return -2;
    if (orc_load_u32le(buf + 4) != (uint32_t)seq_len) {
        *err_bits |= ORC_ERR_MALFORMED;
        return 0;
    }
    if (fmt == ORC_WIRE_F32) {
        for (j = 0; j < n; ++j) x[j] = orc_f32_from_bits(orc_load_u32le(buf + 16 + 4 * j));
    } else if (fmt == ORC_WIRE_F16) {
        for (j = 0; j < n; ++j) x[j] = (float)orc_f16_value(orc_load_u16le(buf + 16 + 2 * j));
    } else {
        for (p = 0; p < seq_len; ++p) {
            const uint8_t *pos = buf + 16 + p * (8 + (int64_t)hidden);
            float scale = orc_f32_from_bits(orc_load_u32le(pos));
            float zp = orc_f32_from_bits(orc_load_u32le(pos + 4));
            if (zp != 0.0f) {
                *err_bits |= ORC_ERR_MALFORMED;
                continue;
            }
            for (j = 0; j < hidden; ++j) {
                float q = (float)(int8_t)pos[8 + j];
                x[p * hidden + j] = q * scale;    /* binary32 multiply */
            }
        }
    }
    return 0;
}

/* Single-layer response ([ADR-0009] Wire Layout, "Single-layer response"):
 * [layer u32 LE][seq_len u32 LE][latency_ms f32 LE], then the payload the
 * request carries (the same f32 / f16 arrays, the same i8 positions).
 * Reading: the three formats share this 12-byte header, since the page
 * keeps every header field unchanged across the formats and calls the i8
 * response "the same structure" as the request's positions.  The payload
 * is produced and read by the request codecs above, so the two layouts
 * cannot drift apart. */
#define ORC_WIRE_RESPONSE_HEADER 12

int64_t orc_wire_response_bytes(int fmt, int32_t seq_len, int32_t hidden)
{
    int64_t req = orc_wire_bytes(fmt, seq_len, hidden);
    return req < 0 ? -1 : req - ORC_WIRE_HEADER + ORC_WIRE_RESPONSE_HEADER;
}

int orc_wire_encode_response(int fmt, const float *x, int32_t seq_len, int32_t hidden,
                             uint32_t layer, float latency_ms, uint8_t *buf, int32_t *err_bits)
{
    int64_t req = orc_wire_bytes(fmt, seq_len, hidden);
    uint8_t *tmp;
    int rc;
    if (req < 0) return -1;
    tmp = (uint8_t *)malloc((size_t)req);
    if (!tmp) return -3;
    rc = orc_wire_encode(fmt, x, seq_len, hidden, layer, 0u, 0u, tmp, err_bits);
    if (rc == 0) {
        orc_store_u32le(buf + 0, layer);
        orc_store_u32le(buf + 4, (uint32_t)seq_len);
        orc_store_u32le(buf + 8, orc_bits_from_f32(latency_ms));
        memcpy(buf + ORC_WIRE_RESPONSE_HEADER, tmp + ORC_WIRE_HEADER, (size_t)(req - ORC_WIRE_HEADER));
    }
    free(tmp);
    return rc;
}

/* Decode a response: the same readings as orc_wire_decode (seq_len checked,
 * i8 zero_point 0). */
int orc_wire_decode_response(int fmt, const uint8_t *buf, int64_t buf_bytes, int32_t seq_len,
                             int32_t hidden, float *x, int32_t *err_bits)
{
    int64_t need = orc_wire_response_bytes(fmt, seq_len, hidden);
    uint8_t *tmp;
    int rc;
    if (need < 0) return -1;
    if (buf_bytes < need) return -2;
    tmp = (uint8_t *)calloc((size_t)(need - ORC_WIRE_RESPONSE_HEADER + ORC_WIRE_HEADER), 1);
    if (!tmp) return -3;
    memcpy(tmp, buf, 8);                          /* layer, seq_len */
    memcpy(tmp + ORC_WIRE_HEADER, buf + ORC_WIRE_RESPONSE_HEADER,
           (size_t)(need - ORC_WIRE_RESPONSE_HEADER));
    rc = orc_wire_decode(fmt, tmp, need - ORC_WIRE_RESPONSE_HEADER + ORC_WIRE_HEADER, seq_len, hidden,
                         x, err_bits);
    free(tmp);
    return rc;
}

/* Array forms of the binary16 helpers (test convenience). */
void orc_f16_value_array(const uint16_t *src, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_f16_value(src[i]);
}

void orc_f16_from_f32_sat_array(const float *src, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_f16_from_f32_sat(src[i]);
}
