/*
 * k16v8.h -- C ABI of libk16v8.so: paged grouped-query attention over an
 * asymmetric KV cache that keeps keys in FP16 and values in E4M3 FP8 with one
 * FP32 scale per (layer, KV head) -- the "K16/V8" route of
 * "Phi-4: quality transfer and interrupted throughput studies" (knlp.io).
 *
 * What the page fixes (intro section): the candidate stores FP16 keys and
 * E4M3 FP8 values with the model's own scales, in a per-layer token-slot pool
 * of a 32 GiB budget; the geometry is 40 layers, 40 query heads, 10 KV heads,
 * head dimension 128.  Section "Matched diagnostic profiles" names the work
 * this library implements: the attention kernels, the merge kernels, and the
 * value gather that writes the compressed cache.
 *
 * Conventions shared by every call
 *  - Pointers named as device pointers must point to device memory of the
 *    current device; the caller owns all memory.  The library allocates
 *    nothing and keeps no state between calls, apart from the built-in
 *    scratch array of k16v8_paged_decode_attention_static.
 *  - Every launching call is asynchronous on `stream` (a cudaStream_t passed
 *    as void*; NULL is the legacy default stream).  Only
 *    k16v8_read_device_error synchronises.
 *  - Arguments are validated on the host before anything is launched; a
 *    non-OK status means nothing was launched.
 *  - Cache layout (pages of K16V8_PAGE_SIZE tokens), element (page, kv head,
 *    offset, d) at ((page*num_kv_heads + head)*16 + offset)*head_dim + d:
 *      k_cache  fp16  [num_pages][num_kv_heads][16][head_dim]
 *      v_cache  E4M3  [num_pages][num_kv_heads][16][head_dim]  (one byte)
 *      v_scale  fp32  [num_kv_heads]   value = v_scale[h] * e4m3(code)
 *  - A slot is page*16 + offset.  block_table[b][i] holds the page of
 *    positions 16i..16i+15 of sequence b.
 *  - Supported shapes: head_dim == 128; attention calls need
 *    num_qo_heads == 4*num_kv_heads (query head h reads KV head h/4).  Other
 *    shapes return K16V8_ERR_UNSUPPORTED_SHAPE.
 *  - Out-of-range slots, page ids or sequence lengths met on the device are
 *    never dereferenced: the kernel skips or masks them and ORs a
 *    K16V8_DEVERR_* bit into the caller's int32 error word (if non-NULL),
 *    which k16v8_read_device_error returns.
 */
#ifndef K16V8_H
#define K16V8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K16V8_PAGE_SIZE 16
#define K16V8_HEAD_DIM 128
#define K16V8_GQA_GROUP 4
#define K16V8_MAX_SPLIT_CHUNK 8192

typedef enum {
    K16V8_OK = 0,
    K16V8_ERR_INVALID_ARG = 1,        /* null pointer, negative size, misalignment */
    K16V8_ERR_UNSUPPORTED_SHAPE = 2,  /* head_dim / GQA group not supported */
    K16V8_ERR_WORKSPACE_TOO_SMALL = 3,
    K16V8_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
    K16V8_ERR_DEVICE_BOUNDS = 5,      /* returned by k16v8_read_device_error */
    K16V8_ERR_STATIC_SCRATCH_LIMIT = 6 /* problem too large for the built-in scratch */
} k16v8_status;

typedef enum { K16V8_F16 = 0, K16V8_F32 = 1 } k16v8_dtype;

/* Bits of the device error word. */
#define K16V8_DEVERR_SLOT 0x1    /* kv_append: slot >= num_pages*16 */
#define K16V8_DEVERR_PAGE 0x2    /* block_table entry outside [0, num_pages) */
#define K16V8_DEVERR_SEQLEN 0x4  /* seq_len < 0, > max_seq_len, or > 16*max_pages_per_seq */
#define K16V8_DEVERR_TIMEOUT 0x8 /* a bounded wait on an async copy gave up */
#define K16V8_DEVERR_INTERNAL 0x10 /* a kernel's own layout check failed; nothing was written */

/*
 * kv_append -- "the candidate also gathers values and writes the compressed
 * cache" ("Matched diagnostic profiles"); storage format from the intro.
 *
 * For every token t with slot s = slot_mapping[t] >= 0 and every KV head h:
 *   k_cache[s/16][h][s%16][:] = k[t][h][:]                      (fp16 copy)
 *   v_cache[s/16][h][s%16][:] = E4M3_rn_satfinite(fl32(v[t][h][:]) / v_scale[h])
 * The division is IEEE fp32 round-to-nearest; the E4M3 rounding is
 * round-to-nearest-even with finite overflow and +-inf saturating to +-448
 * (NaN stays NaN).  Negative slots are skipped (padding).  Slots at or above
 * num_pages*16 are skipped and flag K16V8_DEVERR_SLOT.  Duplicate slots in
 * one call leave an unspecified one of the writers.
 *
 *   k              device, fp16 [num_tokens][num_kv_heads][head_dim], token
 *                  stride k_token_stride elements (0 = num_kv_heads*head_dim)
 *   v              device, fp16 or fp32 (v_dtype) likewise, v_token_stride
 *   slot_mapping   device, int64 [num_tokens]
 *   v_scale        device, fp32 [num_kv_heads]
 *   k_cache/v_cache device, the layer's pool (written in place)
 *   dev_error      device int32 word or NULL
 * k, v, caches: 16-byte aligned; token strides multiples of 8 elements.
 */
int32_t k16v8_kv_append(const void *k, int64_t k_token_stride, const void *v,
                        int32_t v_dtype, int64_t v_token_stride,
                        const int64_t *slot_mapping, int32_t num_tokens,
                        const float *v_scale, void *k_cache, uint8_t *v_cache,
                        int32_t num_pages, int32_t num_kv_heads, int32_t head_dim,
                        int32_t *dev_error, void *stream);

/*
 * Workspace for split-KV decode: partial outputs fp32
 * [batch][num_qo_heads][max_chunks][head_dim] followed by partial LSEs fp32
 * [batch][num_qo_heads][max_chunks], max_chunks = ceil(max_seq_len /
 * split_chunk) (at least 1), each region 256-byte aligned.  Returns 0 for
 * invalid arguments.
 */
size_t k16v8_decode_workspace_size(int32_t batch, int32_t num_qo_heads,
                                   int32_t head_dim, int32_t max_seq_len,
                                   int32_t split_chunk);

/* Byte offsets of the two workspace regions and max_chunks (host only). */
int32_t k16v8_decode_workspace_layout(int32_t batch, int32_t num_qo_heads,
                                      int32_t head_dim, int32_t max_seq_len,
                                      int32_t split_chunk,
                                      size_t *partial_o_offset,
                                      size_t *partial_lse_offset,
                                      int32_t *max_chunks);

/*
 * paged_decode_split -- the attention kernels of "Matched diagnostic
 * profiles", split over the KV sequence.
 *
 * One decode query per sequence.  For sequence b, query head h (KV head
 * g = h/4) and chunk c covering positions [c*split_chunk,
 * min((c+1)*split_chunk, L_b)), with s_j = sm_scale * q[b][h].k_j and
 * v_j = v_scale[g] * e4m3(v8_j):
 *   m_c = max_j s_j,  l_c = sum_j exp(s_j - m_c),
 *   partial_o[b][h][c][:] = sum_j exp(s_j - m_c) v_j / l_c
 *   partial_lse[b][h][c]  = m_c + ln l_c           (natural log)
 * Chunks at or beyond ceil(L_b / split_chunk) are not written.
 *
 *   q            device, fp16 [batch][num_qo_heads][head_dim], 16-B aligned
 *   block_table  device, int32 [batch][max_pages_per_seq]
 *   seq_lens     device, int32 [batch]; each <= max_seq_len (host hint that
 *                sizes the grid without a device->host copy)
 *   split_chunk  tokens per chunk: a multiple of 16 in [16, 8192]
 *   workspace    device, >= k16v8_decode_workspace_size(...) bytes, 256-B
 *                aligned; receives the partials
 *   sm_scale     softmax scale (1/sqrt(head_dim) for plain attention)
 */
int32_t k16v8_paged_decode_split(const void *q, const void *k_cache,
                                 const uint8_t *v_cache, const float *v_scale,
                                 const int32_t *block_table,
                                 int32_t max_pages_per_seq,
                                 const int32_t *seq_lens, int32_t max_seq_len,
                                 int32_t batch, int32_t num_qo_heads,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 int32_t num_pages, float sm_scale,
                                 int32_t split_chunk, void *workspace,
                                 size_t workspace_bytes, int32_t *dev_error,
                                 void *stream);

/*
 * merge_states -- the merge kernels of "Matched diagnostic profiles": the
 * log-sum-exp combination of split-KV partials.  For each (b, h), over the
 * n_b = ceil(min(L_b, max_chunks*split_chunk) / split_chunk) live chunks:
 *   lse = M + ln sum_c exp(lse_c - M)   (M = max_c lse_c)
 *   out = sum_c exp(lse_c - lse) * o_c       -> fp16, lse -> fp32
 * n_b == 0 (an empty sequence) gives out = 0, lse = -inf.
 *
 *   partial_o    device, fp32 [batch][num_qo_heads][max_chunks][head_dim]
 *   partial_lse  device, fp32 [batch][num_qo_heads][max_chunks]
 *   seq_lens     device, int32 [batch]
 *   out          device, fp16 [batch][num_qo_heads][head_dim], 8-B aligned
 *   lse          device, fp32 [batch][num_qo_heads] or NULL
 */
int32_t k16v8_merge_states(const float *partial_o, const float *partial_lse,
                           int32_t batch, int32_t num_qo_heads,
                           int32_t max_chunks, int32_t head_dim,
                           const int32_t *seq_lens, int32_t split_chunk,
                           void *out, float *lse, void *stream);

/*
 * paged_decode_attention -- k16v8_paged_decode_split followed by
 * k16v8_merge_states on the same stream, writing fp16 out
 * [batch][num_qo_heads][head_dim] and fp32 lse [batch][num_qo_heads] (lse may
 * be NULL).  Arguments as for the two calls.  When max_seq_len <= split_chunk
 * (one chunk per sequence) only the split kernel is launched: each CTA
 * writes its rows of out / lse directly (zero rows and -inf for an empty
 * sequence), bit-equal to the merge of the single partial, and the
 * workspace is not written (it must still be given and large enough).
 * out must be 8-byte aligned.
 */
int32_t k16v8_paged_decode_attention(const void *q, const void *k_cache,
                                     const uint8_t *v_cache, const float *v_scale,
                                     const int32_t *block_table,
                                     int32_t max_pages_per_seq,
                                     const int32_t *seq_lens, int32_t max_seq_len,
                                     int32_t batch, int32_t num_qo_heads,
                                     int32_t num_kv_heads, int32_t head_dim,
                                     int32_t num_pages, float sm_scale,
                                     int32_t split_chunk, void *workspace,
                                     size_t workspace_bytes, void *out, float *lse,
                                     int32_t *dev_error, void *stream);

/*
 * paged_decode_attention_balanced -- the same result as
 * k16v8_paged_decode_attention (split-KV attention, then the log-sum-exp
 * merge, "Matched diagnostic profiles"), with the split chosen by the device
 * instead of a fixed split_chunk: all (sequence, KV head, page) tiles are
 * cut into one full wave of equal CTA ranges (SMs x 4 CTAs), so ragged
 * batches leave no tail wave.  Two launches (attention, merge) on `stream`.
 *
 *   batch        0 .. 8192 (0: nothing is launched)
 *   workspace    device, 256-B aligned, at least
 *                k16v8_decode_balanced_workspace_size(batch, num_qo_heads,
 *                head_dim) bytes, sized for the CURRENT device's SM count;
 *                contents need no initialisation and are overwritten
 *   seq_lens     device int32 [batch]; no max_seq_len is needed
 *   flags        0, or K16V8_DECODE_METADATA_READY: the caller guarantees
 *                that block_table and seq_lens are not written by the kernel
 *                launched immediately before this call on `stream` (host
 *                copies and earlier kernels are fine).  The attention kernel
 *                then reads them, plans its work and asks L2 to prefetch
 *                each warp's first cache pages before it waits for that
 *                kernel to finish (programmatic dependent launch); nothing
 *                of the cache reaches the SMs, and q, the workspace and the
 *                outputs are not touched, until after the wait.  Without
 *                the flag nothing is read before the wait.
 * Other arguments, outputs and device errors as for
 * k16v8_paged_decode_attention.  batch * max_pages_per_seq * num_kv_heads
 * and num_pages * num_kv_heads must stay below 2^31 - 1
 * (K16V8_ERR_INVALID_ARG otherwise).
 */
#define K16V8_DECODE_METADATA_READY 0x1

size_t k16v8_decode_balanced_workspace_size(int32_t batch, int32_t num_qo_heads,
                                            int32_t head_dim);

/*
 * The two launches of paged_decode_attention_balanced, for callers that
 * schedule them separately (same arguments; the workspace carries the work
 * plan and the partials from the first to the second).
 * paged_decode_balanced_split already writes the rows of every (sequence,
 * KV head) segment that one CTA held whole; merge_balanced writes the rest
 * (cut segments, and empty sequences: zeros and LSE -inf).
 */
int32_t k16v8_paged_decode_balanced_split(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
    float *lse, int32_t flags, int32_t *dev_error, void *stream);

int32_t k16v8_merge_balanced(const void *workspace, size_t workspace_bytes, int32_t batch,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                             void *out, float *lse, void *stream);

int32_t k16v8_paged_decode_attention_balanced(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
    float *lse, int32_t flags, int32_t *dev_error, void *stream);

/*
 * paged_decode_append_balanced_split / paged_decode_append_attention_balanced
 * -- the load-balanced decode with the step's cache write folded in:
 * equivalent to k16v8_kv_append of each sequence's new token at position
 * seq_lens[b] - 1 (slot block_table[b][(L-1)/16]*16 + (L-1)%16) followed by
 * k16v8_paged_decode_balanced_split (and, for _attention_balanced,
 * k16v8_merge_balanced), one kernel fewer per step ("Matched diagnostic
 * profiles": the candidate writes the compressed cache during decode).
 *   k_new, v_new  device fp16 [batch][num_kv_heads][head_dim], contiguous,
 *                 16-B aligned: the K and V of each sequence's new token
 *                 (read after the dependency wait)
 *   seq_lens      lengths INCLUDING the new token (L = 0: nothing appended)
 * Other arguments, flags, outputs and errors as for
 * k16v8_paged_decode_balanced_split / _attention_balanced; the cache row is
 * written with the rounding of k16v8_kv_append.  A row whose page id is
 * rejected is neither written nor attended (K16V8_DEVERR_PAGE).
 */
int32_t k16v8_paged_decode_append_balanced_split(
    const void *q, const void *k_new, const void *v_new, void *k_cache, uint8_t *v_cache,
    const float *v_scale, const int32_t *block_table, int32_t max_pages_per_seq,
    const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes,
    void *out, float *lse, int32_t flags, int32_t *dev_error, void *stream);

int32_t k16v8_paged_decode_append_attention_balanced(
    const void *q, const void *k_new, const void *v_new, void *k_cache, uint8_t *v_cache,
    const float *v_scale, const int32_t *block_table, int32_t max_pages_per_seq,
    const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, void *workspace, size_t workspace_bytes,
    void *out, float *lse, int32_t flags, int32_t *dev_error, void *stream);

/*
 * paged_decode_append_split / paged_decode_append_attention -- one decode
 * step's cache write fused into the attention kernel: equivalent to
 * k16v8_kv_append of each sequence's new token at position seq_lens[b] - 1
 * (slot block_table[b][(L-1)/16]*16 + (L-1)%16) followed by
 * k16v8_paged_decode_split (and, for _attention, k16v8_merge_states), in one
 * kernel instead of two.  "The candidate also gathers values and writes the
 * compressed cache" ("Matched diagnostic profiles") is the step folded in.
 *
 *   k_new, v_new  device fp16 [batch][num_kv_heads][head_dim], contiguous,
 *                 16-B aligned: the K and V of each sequence's new token
 *   seq_lens      lengths INCLUDING the new token (a sequence with L = 0 has
 *                 no new token and is skipped)
 * Other arguments as for k16v8_paged_decode_split / _attention (including
 * the one-chunk case of _attention: a single launch that writes out / lse).
 * The cache row is written with the same rounding as k16v8_kv_append.
 */
int32_t k16v8_paged_decode_append_split(const void *q, const void *k_new, const void *v_new,
                                        void *k_cache, uint8_t *v_cache, const float *v_scale,
                                        const int32_t *block_table, int32_t max_pages_per_seq,
                                        const int32_t *seq_lens, int32_t max_seq_len,
                                        int32_t batch, int32_t num_qo_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t num_pages, float sm_scale, int32_t split_chunk,
                                        void *workspace, size_t workspace_bytes,
                                        int32_t *dev_error, void *stream);

int32_t k16v8_paged_decode_append_attention(
    const void *q, const void *k_new, const void *v_new, void *k_cache, uint8_t *v_cache,
    const float *v_scale, const int32_t *block_table, int32_t max_pages_per_seq,
    const int32_t *seq_lens, int32_t max_seq_len, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale,
    int32_t split_chunk, void *workspace, size_t workspace_bytes, void *out, float *lse,
    int32_t *dev_error, void *stream);

/*
 * FP16-KV control: the same cache write and split-KV decode for a pool that
 * stores values as fp16 ([num_pages][num_kv_heads][16][head_dim], 2 bytes,
 * no scale) -- the native controls of the subject page store FP16 keys and
 * values (intro), 5,120 B per token per layer instead of 3,840.  Kept to
 * measure the asymmetric format against it on the same kernels.
 *   k16v8_kv_append_v16: k, v fp16 [num_tokens][num_kv_heads][head_dim]
 *     (token strides as for k16v8_kv_append) copied to the caches.
 *   k16v8_paged_decode_split_v16 / _attention_v16: as the K16/V8 calls,
 *     with v_cache16 in place of (v_cache, v_scale).  Within a 16-token page
 *     the P.V products are summed in fp16, so |v| must stay below 4,094.
 */
int32_t k16v8_kv_append_v16(const void *k, int64_t k_token_stride, const void *v,
                            int64_t v_token_stride, const int64_t *slot_mapping,
                            int32_t num_tokens, void *k_cache, void *v_cache16,
                            int32_t num_pages, int32_t num_kv_heads, int32_t head_dim,
                            int32_t *dev_error, void *stream);

int32_t k16v8_paged_decode_split_v16(const void *q, const void *k_cache, const void *v_cache16,
                                     const int32_t *block_table, int32_t max_pages_per_seq,
                                     const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
                                     int32_t num_qo_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t num_pages, float sm_scale,
                                     int32_t split_chunk, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_error, void *stream);

int32_t k16v8_paged_decode_attention_v16(const void *q, const void *k_cache,
                                         const void *v_cache16, const int32_t *block_table,
                                         int32_t max_pages_per_seq, const int32_t *seq_lens,
                                         int32_t max_seq_len, int32_t batch,
                                         int32_t num_qo_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t num_pages, float sm_scale,
                                         int32_t split_chunk, void *workspace,
                                         size_t workspace_bytes, void *out, float *lse,
                                         int32_t *dev_error, void *stream);

/*
 * paged_prefill_attention -- causal attention of a chunk of new prompt tokens
 * against the paged cache, on tensor cores.  The page's throughput metric
 * includes prefill ("Fixed throughput studies"); its 8K profile admits fresh
 * prompts before batch-16 decode ("Matched diagnostic profiles").  The
 * cache must already hold the chunk (call k16v8_kv_append first).
 *
 * Sequence b has qlen_b = qo_indptr[b+1] - qo_indptr[b] new tokens: the last
 * qlen_b of its seq_lens[b] cached positions.  Query row i of that sequence
 * sits at position p = seq_lens[b] - qlen_b + (i - qo_indptr[b]) and attends
 * to positions 0..p (causal).  With s_j = sm_scale * q[i][h].k_j and
 * v_j = v_scale[h/4] * e4m3(v8_j):
 *   out[i][h][:] = sum_{j<=p} exp(s_j - lse) v_j,   lse[i][h] = ln sum_{j<=p} exp(s_j)
 *
 *   q           device fp16 [total_q][num_qo_heads][head_dim], 16-B aligned
 *   qo_indptr   device int32 [batch+1], non-decreasing, qo_indptr[0] = 0,
 *               qo_indptr[batch] = total_q
 *   max_qlen    host hint: the largest qlen_b (sizes the grid)
 *   block_table, seq_lens, caches, v_scale: as for decode
 *   out         device fp16 [total_q][num_qo_heads][head_dim], 16-B aligned
 *   lse         device fp32 [total_q][num_qo_heads] or NULL
 * A sequence with qlen_b > seq_lens[b], seq_lens[b] > 16*max_pages_per_seq
 * or rows outside [0, total_q) flags K16V8_DEVERR_SEQLEN and is skipped; page ids outside [0, num_pages)
 * flag K16V8_DEVERR_PAGE and are not read.  No workspace is needed.
 */
int32_t k16v8_paged_prefill_attention(const void *q, const int32_t *qo_indptr,
                                      int32_t total_q, int32_t max_qlen,
                                      const void *k_cache, const uint8_t *v_cache,
                                      const float *v_scale, const int32_t *block_table,
                                      int32_t max_pages_per_seq, const int32_t *seq_lens,
                                      int32_t batch, int32_t num_qo_heads,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      int32_t num_pages, float sm_scale, void *out,
                                      float *lse, int32_t *dev_error, void *stream);

/*
 * paged_prefill_attention_split -- the same causal prefill with the KV range
 * of each work item (a pair of 32-token query tiles of one sequence and KV
 * head) cut into up to 4 parts that run as separate CTAs, for calls whose
 * items would not fill the GPU in whole waves (e.g. one 1,024-token chunk of
 * one prompt: 16 pairs x 10 KV heads = 160 items on 152 SMs leaves a
 * near-empty second wave).  Every part writes its rows normalised by its own
 * softmax sum (fp16) and their LSE to the workspace; the part that finishes
 * last (an atomic counter per item, no waiting) combines them,
 * o = sum_p e^(lse_p - lse) o_p with lse = log sum_p e^lse_p, and writes out
 * and lse.  The fp16 rounding of the parts adds at most one fp16 ulp of each
 * part's share to the fp16 output.
 *   kv_splits   0: chosen from max_qlen, batch, num_kv_heads and the SM
 *               count (1 unless the items make less than two waves, then
 *               the count of 1..4 that best fills whole waves); 1..4 forced.
 *               A part holds at least 8 KV tiles (1,024 positions), so items
 *               with fewer than 16 tiles are not split whatever the count.
 *   max_seq_len an upper bound on this call's seq_lens, or 0 if unknown: with
 *               kv_splits = 0 it caps the parts at what the longest pair can
 *               use (one per 8 KV tiles), so calls over short prefixes
 *               launch no CTAs that would find nothing to do.  Only a hint:
 *               longer sequences are still computed correctly.
 *   workspace   device, k16v8_prefill_workspace_size(max_qlen, batch,
 *               num_qo_heads, num_kv_heads, head_dim, kv_splits,
 *               max_seq_len) bytes
 *               (0: no split, NULL allowed), 256-B aligned, zero-filled
 *               before its first use; a call that raises no device error
 *               leaves it ready for the next call (its counters back at 0).
 *               Calls that overlap on the GPU must not share one.
 * Other arguments, outputs and errors as for k16v8_paged_prefill_attention;
 * K16V8_ERR_WORKSPACE_TOO_SMALL if workspace_bytes is short,
 * K16V8_ERR_INVALID_ARG for kv_splits < 0, max_seq_len < 0 or a NULL /
 * unaligned workspace that is needed.
 */
size_t k16v8_prefill_workspace_size(int32_t max_qlen, int32_t batch, int32_t num_qo_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t kv_splits,
                                    int32_t max_seq_len);

int32_t k16v8_paged_prefill_attention_split(
    const void *q, const int32_t *qo_indptr, int32_t total_q, int32_t max_qlen,
    const void *k_cache, const uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale, int32_t kv_splits,
    int32_t max_seq_len, void *workspace, size_t workspace_bytes, void *out, float *lse,
    int32_t *dev_error, void *stream);

/*
 * paged_decode_attention_static -- the same computation as
 * k16v8_paged_decode_attention, for callers that cannot allocate device
 * memory: a host that runs inside an engine whose memory manager owns every
 * byte of the device, or code that must not call the CUDA allocator at all
 * (hard real-time paths, plug-ins loaded into a process that forbids it).
 * There is no counterpart in the paper; this is a packaging variant only.
 *
 * The split-KV partials go to a scratch array built into the library
 * (K16V8_STATIC_SCRATCH_BYTES bytes of device memory that every GPU which
 * loads the library keeps until the process exits) instead of a caller
 * workspace.  The call allocates nothing.
 *  - Needs k16v8_decode_workspace_size(batch, num_qo_heads, head_dim,
 *    max_seq_len, split_chunk) <= K16V8_STATIC_SCRATCH_BYTES, else returns
 *    K16V8_ERR_STATIC_SCRATCH_LIMIT and launches nothing.
 *  - The first call on a device looks up that device's address of the
 *    array (with the device current); make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array, and nothing in it needs to
 *    start at zero (each call writes every partial it reads).  Calls whose
 *    kernels overlap on the GPU (different streams, or concurrent host
 *    threads) race on it: serialise them.
 * Other arguments, layouts and errors as for k16v8_paged_decode_attention.
 */
#define K16V8_STATIC_SCRATCH_BYTES (32u << 20)
int32_t k16v8_paged_decode_attention_static(
    const void *q, const void *k_cache, const uint8_t *v_cache, const float *v_scale,
    const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
    int32_t max_seq_len, int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_pages, float sm_scale, int32_t split_chunk, void *out,
    float *lse, int32_t *dev_error, void *stream);

/*
 * Test hooks of the bounded waits.  Every wait of a k16v8 kernel on an
 * asynchronous copy or a hand-off between warp roles gives up after a
 * bounded number of polls, sets K16V8_DEVERR_TIMEOUT in the error word,
 * lets the copies and tensor-core operations it did issue complete, and
 * returns, so a lost hand-off never hangs the GPU and the stream stays
 * usable.  The page records failures rather than hiding them ("Fixed
 * throughput studies"); these two calls let a test reach that path without
 * any fault: each runs the named call with the same arguments, except that
 * the first CTA of the grid withholds one copy (issues nothing and arrives
 * nowhere for it) and waits for it with a short limit.
 *   k16v8_paged_decode_split_wait_test: as k16v8_paged_decode_split; warp
 *     0 of CTA (chunk 0, KV head 0, sequence 0) withholds its first page.
 *   k16v8_paged_prefill_attention_wait_test: as
 *     k16v8_paged_prefill_attention; CTA (0, 0, 0) (the last query-tile
 *     pair of sequence 0, KV head 0) withholds its first KV tile.
 * The withholding CTA's results are incomplete (its partial, or its output
 * rows, are not valid); every other CTA computes normally.  After the call
 * the error word holds K16V8_DEVERR_TIMEOUT (if that CTA had work) and
 * later calls on the stream run normally.  Not for production use.
 */
int32_t k16v8_paged_decode_split_wait_test(const void *q, const void *k_cache,
                                           const uint8_t *v_cache, const float *v_scale,
                                           const int32_t *block_table,
                                           int32_t max_pages_per_seq,
                                           const int32_t *seq_lens, int32_t max_seq_len,
                                           int32_t batch, int32_t num_qo_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t num_pages, float sm_scale,
                                           int32_t split_chunk, void *workspace,
                                           size_t workspace_bytes, int32_t *dev_error,
                                           void *stream);

int32_t k16v8_paged_prefill_attention_wait_test(
    const void *q, const int32_t *qo_indptr, int32_t total_q, int32_t max_qlen,
    const void *k_cache, const uint8_t *v_cache, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch, int32_t num_qo_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t num_pages, float sm_scale, void *out,
    float *lse, int32_t *dev_error, void *stream);

/*
 * Wait for `stream`, then copy the device error word to *host_value and
 * return K16V8_OK when it is zero, K16V8_ERR_DEVICE_BOUNDS otherwise
 * (K16V8_ERR_CUDA if the synchronisation or copy fails).
 */
int32_t k16v8_read_device_error(const int32_t *dev_error, void *stream,
                                int32_t *host_value);

/* Static, human-readable name of a status code. */
const char *k16v8_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* K16V8_H */
