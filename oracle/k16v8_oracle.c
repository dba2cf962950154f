/*
 * k16v8 oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU restatement of what the K16/V8 paged attention
 * path computes.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library; the product path never does.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Subject page: "Phi-4: quality transfer and interrupted throughput studies"
 * (knlp.io).  The intro section fixes the storage format (FP16 keys, E4M3 FP8
 * values, per-model value scales) and the geometry (40 layers, 40 query
 * heads, 10 KV heads, head dimension 128); the same section gives the
 * per-layer token-slot pool of the 32 GiB budget; section "Matched
 * diagnostic profiles" names the attention kernels, the merge kernels and the
 * value-gather / compressed-cache write.  Where the page is silent (layout,
 * rounding, scale granularity, split size) the readings used here are the
 * plainest ones:
 *   - E4M3 is OCP E4M3FN: bias 7, subnormals m*2^-9, codes 0x7F/0xFF are NaN,
 *     no infinities, largest finite 448.
 *   - A value is quantised as fl32(v / scale) (IEEE fp32 division, round to
 *     nearest) followed by ONE round-to-nearest-even to E4M3, saturating
 *     finite overflow and +-inf to +-448.
 *   - Cache layout is page-major then KV head: element (page, head, offset, d)
 *     sits at ((page*Hkv + head)*page_size + offset)*D + d.
 *   - slot = page*page_size + offset; a negative slot means "skip".
 *   - q head h reads KV head h / (Hq/Hkv).
 *   - lse is the natural log of sum_j exp(sm_scale * q.k_j).
 *   - A split-KV chunk c covers positions [c*chunk, min((c+1)*chunk, L)); an
 *     empty chunk has o = 0, lse = -inf; L == 0 gives out = 0, lse = -inf.
 *   - Causal prefill query i of a sequence with qlen new tokens and L cached
 *     tokens (the new ones included) sits at position L - qlen + i and sees
 *     positions 0..L - qlen + i.
 *
 * Parity pins (tests/): the E4M3 decode table against torch.float8_e4m3fn,
 * the encoder by brute-force nearest-even search and against the library
 * cast, the pool sizes against the figures printed on the page, attention
 * against torch's scaled_dot_product_attention on unpaged float64 tensors,
 * closed forms (uniform keys, one-hot scores) and split/merge invariances.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OK 0
#define ERR_ARG 1
#define ERR_BOUNDS 5

/* ---- number formats ---------------------------------------------------- */

/* IEEE binary16 -> double, from the format definition (1 sign, 5 exponent
 * bits with bias 15, 10 fraction bits). */
double k16v8o_half_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)m, e - 25);
    return s ? -v : v;
}

/* E4M3FN code -> double: sign, 4 exponent bits (bias 7), 3 fraction bits.
 * Exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN. */
double k16v8o_e4m3_to_double(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* fp32 -> E4M3FN, round to nearest even, saturating to +-448.  Integer
 * operations on the fp32 bit pattern only. */
uint8_t k16v8o_e4m3_from_float(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    uint8_t sign = (uint8_t)((b >> 24) & 0x80u);
    uint32_t a = b & 0x7FFFFFFFu;
    if (a > 0x7F800000u)
        return sign | 0x7Fu; /* NaN stays NaN */
    if (a == 0x7F800000u)
        return sign | 0x7Eu; /* +-inf saturates */
    if ((a >> 23) == 0)
        return sign; /* fp32 zero/subnormal: below 2^-126, rounds to 0 */
    int E = (int)(a >> 23) - 127;
    if (E >= -6) {
        /* E4M3 normal binade: keep 3 fraction bits, ties to even.  The
         * increment may carry into the exponent, which is what we want. */
        uint32_t lsb = (a >> 20) & 1u;
        uint32_t r = (a + 0x7FFFFu + lsb) >> 20;
        int E2 = (int)(r >> 3) - 127;
        uint32_t m2 = r & 7u;
        if (E2 > 8 || (E2 == 8 && m2 == 7u))
            return sign | 0x7Eu; /* beyond 448 after rounding: saturate */
        return (uint8_t)(sign | (uint32_t)(((E2 + 7) << 3) | (int)m2));
    }
    /* Below the least normal 2^-6 the grid is k * 2^-9, k = 0..8.
     * x * 2^9 = sig * 2^(E - 14) with sig the 24-bit significand. */
    uint32_t sig = (a & 0x7FFFFFu) | 0x800000u;
    int s = 14 - E; /* >= 21 here */
    if (s >= 32)
        return sign;
    uint32_t q = sig >> s;
    uint32_t rem = sig & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q++;
    return (uint8_t)(sign | q); /* q == 8 is code 0x08, the least normal */
}

/* The value quantiser: one fp32 IEEE division by the per-head scale, then
 * one rounding to E4M3. */
uint8_t k16v8o_quantize_value(float v, float scale)
{
    volatile float x = v / scale;
    return k16v8o_e4m3_from_float(x);
}

/* Element-wise fp32 -> E4M3 over an array (for exhaustive checks). */
void k16v8o_e4m3_encode_n(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = k16v8o_e4m3_from_float(x[i]);
}

/* Element-wise quantiser over an array: out[i] = E4M3(fl32(v[i] / scale)). */
void k16v8o_quantize_n(const float *v, float scale, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = k16v8o_quantize_value(v[i], scale);
}

/* ---- pool sizing ------------------------------------------------------- */

/* Token slots per layer of a KV budget, rounded down to whole pages. */
int64_t k16v8o_pool_slots(double budget_bytes, int32_t layers,
                          int64_t bytes_per_token, int32_t page_size)
{
    double per_layer = budget_bytes / (double)layers;
    double pages = floor(per_layer / ((double)bytes_per_token * page_size));
    return (int64_t)pages * page_size;
}

/* ---- kv_append (value gather + compressed cache write) ----------------- */

/* k: fp16 bits [T][Hkv][D] with token stride k_ts (elements);
 * v: fp16 bits or fp32 [T][Hkv][D] with token stride v_ts.
 * Writes k_cache (fp16 bits) and v_cache (E4M3 codes) in place. */
int k16v8o_kv_append(const uint16_t *k, int64_t k_ts, const void *v,
                     int32_t v_is_f32, int64_t v_ts,
                     const int64_t *slot_mapping, int32_t T,
                     const float *v_scale, uint16_t *k_cache, uint8_t *v_cache,
                     int32_t num_pages, int32_t Hkv, int32_t D,
                     int32_t page_size)
{
    if (T < 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0)
        return ERR_ARG;
    int64_t nslots = (int64_t)num_pages * page_size;
    for (int32_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= nslots)
            return ERR_BOUNDS;
        int64_t page = slot / page_size, off = slot % page_size;
        for (int32_t h = 0; h < Hkv; ++h) {
            for (int32_t d = 0; d < D; ++d) {
                int64_t dst = ((page * Hkv + h) * page_size + off) * D + d;
                int64_t ks = (int64_t)t * k_ts + (int64_t)h * D + d;
                int64_t vs = (int64_t)t * v_ts + (int64_t)h * D + d;
                k_cache[dst] = k[ks];
                float vf = v_is_f32 ? ((const float *)v)[vs]
                                    : (float)k16v8o_half_to_double(
                                          ((const uint16_t *)v)[vs]);
                v_cache[dst] = k16v8o_quantize_value(vf, v_scale[h]);
            }
        }
    }
    return OK;
}

/* ---- exact softmax attention over the dequantised paged cache ---------- */

/* Attention of one query row (fp16 bits, D) against cache positions
 * [lo, hi) of one sequence for one KV head.  Returns lse (natural log of
 * the sum of exp(score)); writes the normalised output into out[D].
 * Returns ERR_BOUNDS through *err for page ids outside [0, num_pages). */
static double attend_range(const uint16_t *qrow, const uint16_t *k_cache,
                           const void *v_cache, int v_f16, double vscale,
                           const int32_t *btab, int32_t g, int32_t Hkv,
                           int32_t D, int32_t page_size, int32_t num_pages,
                           double sm_scale, int64_t lo, int64_t hi,
                           double *out, double *s_buf, int *err)
{
    for (int32_t d = 0; d < D; ++d)
        out[d] = 0.0;
    if (hi <= lo)
        return -INFINITY;
    double qd[512];
    for (int32_t d = 0; d < D; ++d)
        qd[d] = k16v8o_half_to_double(qrow[d]);
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
        int32_t page = btab[j / page_size];
        if (page < 0 || page >= num_pages) {
            *err = ERR_BOUNDS;
            return NAN;
        }
        int64_t base = (((int64_t)page * Hkv + g) * page_size + j % page_size) * D;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += qd[d] * k16v8o_half_to_double(k_cache[base + d]);
        double s = sm_scale * dot;
        s_buf[j - lo] = s;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        int32_t page = btab[j / page_size];
        int64_t base = (((int64_t)page * Hkv + g) * page_size + j % page_size) * D;
        double p = exp(s_buf[j - lo] - m);
        l += p;
        for (int32_t d = 0; d < D; ++d)
            out[d] += p * (v_f16 ? k16v8o_half_to_double(((const uint16_t *)v_cache)[base + d])
                                 : vscale * k16v8o_e4m3_to_double(((const uint8_t *)v_cache)[base + d]));
    }
    for (int32_t d = 0; d < D; ++d)
        out[d] /= l;
    return m + log(l);
}

/* Work distribution: a plain static split of item indices over threads. */
typedef struct {
    int (*fn)(void *ctx, int64_t item, double *scratch);
    void *ctx;
    int64_t n_items;
    int64_t scratch_len;
    int32_t tid, nthreads;
    int err;
} job_t;

static void *job_run(void *arg)
{
    job_t *j = (job_t *)arg;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(j->scratch_len + 1));
    if (!scratch) {
        j->err = ERR_ARG;
        return NULL;
    }
    for (int64_t it = j->tid; it < j->n_items; it += j->nthreads) {
        int e = j->fn(j->ctx, it, scratch);
        if (e) {
            j->err = e;
            break;
        }
    }
    free(scratch);
    return NULL;
}

static int run_parallel(int (*fn)(void *, int64_t, double *), void *ctx,
                        int64_t n_items, int64_t scratch_len, int32_t nthreads)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int32_t)n : 1;
    }
    if (nthreads > 256)
        nthreads = 256;
    if (n_items < nthreads)
        nthreads = n_items > 0 ? (int32_t)n_items : 1;
    job_t jobs[256];
    pthread_t th[256];
    for (int32_t i = 0; i < nthreads; ++i) {
        jobs[i] = (job_t){fn, ctx, n_items, scratch_len, i, nthreads, 0};
        if (i > 0)
            pthread_create(&th[i], NULL, job_run, &jobs[i]);
    }
    job_run(&jobs[0]);
    int err = jobs[0].err;
    for (int32_t i = 1; i < nthreads; ++i) {
        pthread_join(th[i], NULL);
        if (jobs[i].err)
            err = jobs[i].err;
    }
    return err;
}

/* ---- decode (split-KV partials and the full result) -------------------- */

typedef struct {
    const uint16_t *q, *k_cache;
    const void *v_cache;
    int v_f16;
    const float *v_scale;
    const int32_t *block_table, *seq_lens;
    int32_t max_pages, Hq, Hkv, D, page_size, num_pages;
    double sm_scale;
    int32_t split_chunk, max_chunks;
    double *out, *lse, *partial_o, *partial_lse;
} decode_ctx;

static int decode_item(void *vctx, int64_t item, double *scratch)
{
    decode_ctx *c = (decode_ctx *)vctx;
    int64_t b = item / c->Hq;
    int32_t h = (int32_t)(item % c->Hq);
    int32_t g = h / (c->Hq / c->Hkv);
    int64_t L = c->seq_lens[b];
    const uint16_t *qrow = c->q + (b * c->Hq + h) * c->D;
    const int32_t *btab = c->block_table + b * c->max_pages;
    int err = OK;
    if (L < 0 || (L + c->page_size - 1) / c->page_size > c->max_pages)
        return ERR_ARG;
    double vs = c->v_f16 ? 1.0 : (double)c->v_scale[g];
    if (c->out) {
        double l = attend_range(qrow, c->k_cache, c->v_cache, c->v_f16, vs, btab, g,
                                c->Hkv, c->D, c->page_size, c->num_pages,
                                c->sm_scale, 0, L, c->out + (b * c->Hq + h) * c->D,
                                scratch, &err);
        if (err)
            return err;
        c->lse[b * c->Hq + h] = l;
    }
    if (c->partial_o && c->split_chunk > 0) {
        for (int32_t ch = 0; ch < c->max_chunks; ++ch) {
            int64_t lo = (int64_t)ch * c->split_chunk;
            int64_t hi = lo + c->split_chunk < L ? lo + c->split_chunk : L;
            int64_t idx = (b * c->Hq + h) * c->max_chunks + ch;
            double l = attend_range(qrow, c->k_cache, c->v_cache, c->v_f16, vs, btab, g,
                                    c->Hkv, c->D, c->page_size, c->num_pages,
                                    c->sm_scale, lo, hi, c->partial_o + idx * c->D,
                                    scratch, &err);
            if (err)
                return err;
            c->partial_lse[idx] = l;
        }
    }
    return OK;
}

static int paged_decode_impl(const uint16_t *q, const uint16_t *k_cache, const void *v_cache,
                             int v_f16, const float *v_scale, const int32_t *block_table,
                             int32_t max_pages, const int32_t *seq_lens, int32_t B, int32_t Hq,
                             int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
                             double sm_scale, int32_t split_chunk, int32_t max_chunks,
                             double *out, double *lse, double *partial_o, double *partial_lse,
                             int32_t nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || D > 512 ||
        page_size <= 0)
        return ERR_ARG;
    int64_t maxL = 0;
    for (int32_t b = 0; b < B; ++b)
        if (seq_lens[b] > maxL)
            maxL = seq_lens[b];
    decode_ctx c = {q, k_cache, v_cache, v_f16, v_scale, block_table, seq_lens,
                    max_pages, Hq, Hkv, D, page_size, num_pages, sm_scale,
                    split_chunk, max_chunks, out, lse, partial_o, partial_lse};
    return run_parallel(decode_item, &c, (int64_t)B * Hq, maxL, nthreads);
}

/* q: fp16 bits [B][Hq][D]; caches as in kv_append; block_table int32
 * [B][max_pages]; seq_lens int32 [B].  out [B][Hq][D] and lse [B][Hq] (may be
 * NULL to skip); partial_o [B][Hq][max_chunks][D], partial_lse
 * [B][Hq][max_chunks] (may be NULL) for split chunks of split_chunk tokens. */
int k16v8o_paged_decode(const uint16_t *q, const uint16_t *k_cache,
                        const uint8_t *v_cache, const float *v_scale,
                        const int32_t *block_table, int32_t max_pages,
                        const int32_t *seq_lens, int32_t B, int32_t Hq,
                        int32_t Hkv, int32_t D, int32_t page_size,
                        int32_t num_pages, double sm_scale, int32_t split_chunk,
                        int32_t max_chunks, double *out, double *lse,
                        double *partial_o, double *partial_lse, int32_t nthreads)
{
    return paged_decode_impl(q, k_cache, v_cache, 0, v_scale, block_table, max_pages, seq_lens,
                             B, Hq, Hkv, D, page_size, num_pages, sm_scale, split_chunk,
                             max_chunks, out, lse, partial_o, partial_lse, nthreads);
}

/* The FP16-KV control: the same attention over a cache whose values are
 * stored as fp16 (no quantisation, no scale). */
int k16v8o_paged_decode_v16(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache16, const int32_t *block_table,
                            int32_t max_pages, const int32_t *seq_lens, int32_t B,
                            int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                            int32_t num_pages, double sm_scale, double *out, double *lse,
                            int32_t nthreads)
{
    return paged_decode_impl(q, k_cache, v_cache16, 1, NULL, block_table, max_pages, seq_lens,
                             B, Hq, Hkv, D, page_size, num_pages, sm_scale, 0, 0, out, lse,
                             NULL, NULL, nthreads);
}

/* FP16-KV control cache write: K and V copied as fp16. */
int k16v8o_kv_append_v16(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                         int32_t T, uint16_t *k_cache, uint16_t *v_cache16, int32_t num_pages,
                         int32_t Hkv, int32_t D, int32_t page_size)
{
    if (T < 0 || Hkv <= 0 || D <= 0 || page_size <= 0 || num_pages < 0)
        return ERR_ARG;
    int64_t nslots = (int64_t)num_pages * page_size;
    for (int32_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= nslots)
            return ERR_BOUNDS;
        int64_t page = slot / page_size, off = slot % page_size;
        for (int32_t h = 0; h < Hkv; ++h)
            for (int32_t d = 0; d < D; ++d) {
                int64_t dst = ((page * Hkv + h) * page_size + off) * D + d;
                int64_t src = ((int64_t)t * Hkv + h) * D + d;
                k_cache[dst] = k[src];
                v_cache16[dst] = v[src];
            }
    }
    return OK;
}

/* ---- log-sum-exp merge of split partials ------------------------------- */

/* partial_o [B][Hq][max_chunks][D], partial_lse [B][Hq][max_chunks]; the
 * first n_chunks[b] chunks of sequence b are merged:
 *   lse = M + ln sum_c exp(lse_c - M),  out = sum_c exp(lse_c - lse) o_c. */
int k16v8o_merge(const double *partial_o, const double *partial_lse,
                 const int32_t *n_chunks, int32_t B, int32_t Hq,
                 int32_t max_chunks, int32_t D, double *out, double *lse)
{
    for (int32_t b = 0; b < B; ++b) {
        int32_t nc = n_chunks[b];
        if (nc < 0 || nc > max_chunks)
            return ERR_ARG;
        for (int32_t h = 0; h < Hq; ++h) {
            const double *pl = partial_lse + ((int64_t)b * Hq + h) * max_chunks;
            const double *po = partial_o + ((int64_t)b * Hq + h) * max_chunks * D;
            double *o = out + ((int64_t)b * Hq + h) * D;
            double M = -INFINITY;
            for (int32_t c = 0; c < nc; ++c)
                if (pl[c] > M)
                    M = pl[c];
            for (int32_t d = 0; d < D; ++d)
                o[d] = 0.0;
            if (M == -INFINITY) {
                lse[(int64_t)b * Hq + h] = -INFINITY;
                continue;
            }
            double S = 0.0;
            for (int32_t c = 0; c < nc; ++c)
                S += exp(pl[c] - M);
            double total = M + log(S);
            for (int32_t c = 0; c < nc; ++c) {
                double w = exp(pl[c] - total);
                for (int32_t d = 0; d < D; ++d)
                    o[d] += w * po[(int64_t)c * D + d];
            }
            lse[(int64_t)b * Hq + h] = total;
        }
    }
    return OK;
}

/* ---- causal prefill over the paged cache ------------------------------- */

typedef struct {
    const uint16_t *q, *k_cache;
    const uint8_t *v_cache;
    const float *v_scale;
    const int32_t *qo_indptr, *block_table, *seq_lens;
    int32_t B, max_pages, Hq, Hkv, D, page_size, num_pages;
    double sm_scale;
    const int64_t *rows; /* optional subset of query-token rows */
    double *out, *lse;
} prefill_ctx;

static int prefill_item(void *vctx, int64_t item, double *scratch)
{
    prefill_ctx *c = (prefill_ctx *)vctx;
    int64_t ri = item / c->Hq;
    int32_t h = (int32_t)(item % c->Hq);
    int64_t row = c->rows ? c->rows[ri] : ri;
    /* find the sequence that owns this query row */
    int32_t b = 0;
    while (b < c->B && c->qo_indptr[b + 1] <= row)
        ++b;
    if (b >= c->B || row < c->qo_indptr[b])
        return ERR_ARG;
    int64_t qlen = c->qo_indptr[b + 1] - c->qo_indptr[b];
    int64_t L = c->seq_lens[b];
    if (qlen > L || (L + c->page_size - 1) / c->page_size > c->max_pages)
        return ERR_ARG;
    int64_t pos = L - qlen + (row - c->qo_indptr[b]);
    int32_t g = h / (c->Hq / c->Hkv);
    int err = OK;
    double l = attend_range(c->q + (row * c->Hq + h) * c->D, c->k_cache,
                            c->v_cache, 0, (double)c->v_scale[g],
                            c->block_table + (int64_t)b * c->max_pages, g,
                            c->Hkv, c->D, c->page_size, c->num_pages,
                            c->sm_scale, 0, pos + 1,
                            c->out + (ri * c->Hq + h) * c->D, scratch, &err);
    if (err)
        return err;
    c->lse[ri * c->Hq + h] = l;
    return OK;
}

/* q: fp16 bits [total_q][Hq][D] ragged by qo_indptr [B+1]; seq_lens[b] counts
 * the cached tokens including this call's qlen_b new ones.  rows: NULL for
 * every query row, else n_rows row indices to evaluate; out [n_rows][Hq][D],
 * lse [n_rows][Hq] in that order. */
int k16v8o_paged_prefill(const uint16_t *q, const int32_t *qo_indptr,
                         int32_t B, const uint16_t *k_cache,
                         const uint8_t *v_cache, const float *v_scale,
                         const int32_t *block_table, int32_t max_pages,
                         const int32_t *seq_lens, int32_t Hq, int32_t Hkv,
                         int32_t D, int32_t page_size, int32_t num_pages,
                         double sm_scale, const int64_t *rows, int64_t n_rows,
                         double *out, double *lse, int32_t nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || D > 512 ||
        page_size <= 0)
        return ERR_ARG;
    int64_t maxL = 0;
    for (int32_t b = 0; b < B; ++b)
        if (seq_lens[b] > maxL)
            maxL = seq_lens[b];
    if (!rows)
        n_rows = qo_indptr[B];
    prefill_ctx c = {q, k_cache, v_cache, v_scale, qo_indptr, block_table,
                     seq_lens, B, max_pages, Hq, Hkv, D, page_size,
                     num_pages, sm_scale, rows, out, lse};
    return run_parallel(prefill_item, &c, n_rows * Hq, maxL, nthreads);
}
