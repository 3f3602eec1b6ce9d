/*
 * attn_varlen.h -- C ABI of the GB300 (sm_103a) attention library.
 *
 * Exact scaled-dot-product attention O = softmax(scale * Q K^T) V computed in
 * one pass per query tile with the online-softmax recurrence (running max m,
 * proxy denominator d', proxy output o' rescaled by e^(m_old - m_new)), so the
 * logits X and probabilities A never reach device memory.  Source of the
 * method and of the call shapes: "从零实现 vLLM (1.3)：如何加速 Attention 计算"
 * (blog.xiaohansong.com), sections "减少遍历次数的“在线 Softmax”",
 * "FlashAttention 的最终实现", "计算流程（1-Pass 算法与分块）",
 * "Attention 源码分析", "Prefill" and "Decode".
 *
 * Conventions shared by every entry point
 *  - Tensors are bf16 (IEEE bfloat16 bit patterns), row-major, the head_dim
 *    axis contiguous and the head axis packed right above it.  Only the token
 *    ("row") stride may be chosen; it is given in ELEMENTS and must keep every
 *    row 16-byte aligned (stride * 2 % 16 == 0).  A row stride of 0 means the
 *    packed default (num_heads * head_dim).
 *  - Every pointer is a DEVICE pointer unless stated otherwise.  The caller
 *    owns all memory (inputs, outputs, lse, workspace); the library allocates
 *    nothing and keeps no state besides cached device attributes and one
 *    device-side error word.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    = the legacy default stream).  A returned ATTN_OK means the arguments were
 *    accepted and the kernels were launched.
 *  - Index data that lives on the device (cu_seqlens, block_table,
 *    cache_seqlens, slot_mapping) is not read on the host.  Kernels never
 *    access memory outside the sizes given here: a bad index is skipped and
 *    recorded in the device error word (attn_get_last_device_error).
 *  - head_dim must be 64 or 128; num_heads_q must be a multiple of
 *    num_heads_kv (GQA: query head h reads KV head h / (num_heads_q /
 *    num_heads_kv)).  The prefill kernels (attn_varlen_fwd, attn_padded_fwd,
 *    the prefill route of attn_kvcache_fwd) take a group size
 *    G = num_heads_q / num_heads_kv up to 128: a 128-row query slot packs
 *    floor(128 / G) tokens x G heads (for G = 3, 5, 6, 7, ... the last
 *    128 - floor(128 / G) G rows of a slot stay idle, and the slot's output
 *    rows are written row by row instead of by TMA boxes).  Larger groups
 *    return ATTN_ERR_UNSUPPORTED there; the decode kernels take any G up to 64.
 *  - No function aborts, throws or prints.
 */
#ifndef ATTN_VARLEN_H
#define ATTN_VARLEN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 2

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,        /* null pointer, negative size, Hq % Hkv != 0, misaligned stride */
    ATTN_ERR_UNSUPPORTED = 2,        /* head_dim, GQA group or block_size outside what is built;
                                        device older than sm_103 */
    ATTN_ERR_WORKSPACE_TOO_SMALL = 3,
    ATTN_ERR_LAUNCH_FAILED = 4,      /* a CUDA runtime or driver call failed */
    ATTN_ERR_DEVICE_TIMEOUT = 5,     /* a kernel's bounded wait ran out (reported by the error word) */
    ATTN_ERR_DEVICE_INDEX = 6,       /* a device-side index was out of range (reported by the error word) */
    ATTN_ERR_NO_DEVICE = 7,          /* no CUDA device, or the device query failed */
    ATTN_ERR_DEVICE_RANGE = 8        /* an input value outside the range a kernel handles (reported by the
                                        error word; see attn_varlen_fwd) */
} attn_status;

/* ------------------------------------------------------------------------
 * attn_varlen_fwd -- varlen prefill ("flash_attn_varlen_func" in the article's
 * Prefill section), causal or not, with contiguous or paged K/V.
 *
 *   q            [total_q, num_heads_q, head_dim]; sequence b owns query rows
 *                [cu_seqlens_q[b], cu_seqlens_q[b+1])
 *   k, v         contiguous (block_table == NULL): [total_k, num_heads_kv,
 *                head_dim], sequence b owns key rows [cu_seqlens_k[b],
 *                cu_seqlens_k[b+1]);
 *                paged (block_table != NULL, the article's prefix cache): the
 *                caches [num_blocks, block_size, num_heads_kv, head_dim];
 *                logical key j of sequence b is cache row
 *                block_table[b * block_table_stride + j / block_size] *
 *                block_size + j % block_size, and cu_seqlens_k counts each
 *                sequence's whole context (cached + new)
 *   out          [total_q, num_heads_q, head_dim] bf16, written
 *   lse          nullable; [num_heads_q, total_q] float32, natural-log
 *                log-sum-exp of the scaled logits of each row (-inf for a row
 *                that sees no key, whose output is 0)
 *   cu_seqlens_q/_k  int32 [batch + 1], non-decreasing, starting at 0
 *   total_q      rows of q / out; kernels never touch rows beyond them
 *   total_k      contiguous: rows of k / v; paged: an upper bound of
 *                cu_seqlens_k[batch] (all sequences' context lengths), e.g.
 *                batch * max_seqlen_k.  It sizes the workspace.
 *   max_seqlen_q/_k  host-side upper bounds of the per-sequence lengths
 *   causal       nonzero: bottom-right aligned mask, query i of a sequence
 *                with Lq queries and Lk keys sees keys j <= Lk - Lq + i
 *   block_size   paged only: a power of two >= 16; num_blocks > 0
 *   v16_cache    nullable, paged only: an fp16 cache [num_blocks, block_size,
 *                num_heads_kv, head_dim] holding V / 16 for every cached key,
 *                kept by store_kvcache (its v16_cache argument).  The P V
 *                product then reads V / 16 from it through the block table and
 *                the call converts nothing; without it each call writes an fp16
 *                copy of the V rows it reads into the workspace, except when
 *                head_dim is 128 and every sequence fits one query slot
 *                (max_seqlen_q <= 128 / G): that kernel loads bf16 V tiles and
 *                converts each to V / 16 in shared memory.  (A paged V tile
 *                past a sequence's last key is zeroed in shared memory, so
 *                cache slots past the end may hold anything.)
 *   workspace    device scratch of at least attn_varlen_workspace_size(...)
 *                bytes, 256-byte aligned: without v16_cache (and outside the
 *                one-slot case above) it receives an fp16 copy of V (V / 16)
 *                laid out by logical key, which the P V product reads; with
 *                v16_cache size it with total_k = 0 (the size function itself
 *                leaves the copy out for one-slot sizes at head_dim 128)
 * Value range: the P V product runs in fp16 on 16 P and V / 16, so V entries
 * must satisfy |v| < 2^20; larger (or non-finite) entries are clamped and
 * reported as ATTN_ERR_DEVICE_RANGE by attn_get_last_device_error.
 * Limits: head_dim 64 or 128, and G = num_heads_q / num_heads_kv at most 128
 * (any G, dividing 128 or not); anything else returns ATTN_ERR_UNSUPPORTED.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 * ATTN_ERR_WORKSPACE_TOO_SMALL, ATTN_ERR_LAUNCH_FAILED or ATTN_ERR_NO_DEVICE.
 * ------------------------------------------------------------------------ */
ATTN_API attn_status attn_varlen_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            int batch, int64_t total_q, int64_t total_k,
                            int max_seqlen_q, int max_seqlen_k,
                            int num_heads_q, int num_heads_kv, int head_dim,
                            float softmax_scale, int causal,
                            const int32_t *block_table, int block_table_stride,
                            int block_size, int64_t num_blocks, const void *v16_cache,
                            int64_t q_row_stride, int64_t k_row_stride, int64_t v_row_stride,
                            int64_t out_row_stride,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace attn_varlen_fwd needs for these sizes (total_k as
 * passed to attn_varlen_fwd). */
ATTN_API size_t attn_varlen_workspace_size(int batch, int num_heads_q, int num_heads_kv, int head_dim,
                                           int max_seqlen_q, int64_t total_k);

/* ------------------------------------------------------------------------
 * attn_varlen_fwd_host -- attn_varlen_fwd (contiguous K/V) for a caller whose
 * q, k, v and output live in HOST memory: the article's Prefill call with the
 * transfers to and from the device made part of it.
 *
 * The batch is cut into `num_groups` groups of whole sequences with about the
 * same number of query tokens (the last two groups 0.6 and 0.3 of the others,
 * so that less work trails the last copy in).  Group i's host -> device copies
 * (on copy_in_stream) overlap the attention of group i-1 (on `stream`) and the
 * device -> host copy of group i-2's output (on copy_out_stream): one
 * cudaMemcpyAsync per group, tensor and direction, ordered by the two events.
 * Each group is one attn_varlen_fwd call whose cu_seqlens point into the full
 * arrays, so rows are addressed in place and the output is bit-identical to
 * one attn_varlen_fwd call over the whole batch.
 *
 *   q_host, k_host, v_host  packed [total, heads, head_dim] bf16 in host
 *                memory; page-locked (pinned) for the copies to overlap
 *   out_host     packed [total_q, num_heads_q, head_dim] bf16 host buffer, written
 *   cu_seqlens_q_host, cu_seqlens_k_host  int32 [batch + 1] in HOST memory,
 *                starting at 0, non-decreasing, lengths <= max_seqlen_q / _k
 *                (checked here: ATTN_ERR_INVALID_ARG otherwise); total_q =
 *                cu_seqlens_q_host[batch], total_k = cu_seqlens_k_host[batch]
 *   q_dev, k_dev, v_dev, out_dev  device staging buffers of the same packed
 *                shapes (caller-owned); cu_dev int32 [2 * (batch + 1)] device
 *   workspace    attn_varlen_workspace_size(batch, num_heads_q, num_heads_kv,
 *                head_dim, max_seqlen_q, total_k) bytes, 256-byte aligned
 *   num_groups   1..64
 *   stream, copy_in_stream, copy_out_stream  three distinct cudaStream_t; the
 *                copies start after the work already queued on `stream`, and
 *                `stream` waits for the last copy out, so synchronising `stream`
 *                (or an event recorded on it after this call) means out_host is
 *                complete
 *   event_a, event_b  two caller-created cudaEvent_t the call records and waits
 *                on (reused for every group; timing may be disabled)
 * Everything is asynchronous: host buffers must stay valid, and unmodified,
 * until `stream` has passed this call.  The library allocates nothing.
 * Returns the statuses of attn_varlen_fwd (ATTN_ERR_LAUNCH_FAILED if a copy
 * or event call fails).
 * ------------------------------------------------------------------------ */
ATTN_API attn_status attn_varlen_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                                          void *out_host, const int32_t *cu_seqlens_q_host,
                                          const int32_t *cu_seqlens_k_host, int batch, int max_seqlen_q,
                                          int max_seqlen_k, int num_heads_q, int num_heads_kv, int head_dim,
                                          float softmax_scale, int causal, void *q_dev, void *k_dev, void *v_dev,
                                          void *out_dev, int32_t *cu_dev, void *workspace, size_t workspace_bytes,
                                          int num_groups, void *stream, void *copy_in_stream,
                                          void *copy_out_stream, void *event_a, void *event_b);

/* ------------------------------------------------------------------------
 * attn_decode_paged -- one new query token per sequence against its paged
 * cache ("flash_attn_with_kvcache(q.unsqueeze(1), k_cache, v_cache,
 * cache_seqlens, block_table, softmax_scale, causal=True)" in the article's
 * Decode section).  With one query the bottom-right causal mask lets it see
 * every cached key, so causality needs no argument.
 *
 *   q            [batch, num_heads_q, head_dim] (the article's [B, 1, H, D]
 *                with the unit axis dropped); row stride q_row_stride
 *   k_cache, v_cache  [num_blocks, block_size, num_heads_kv, head_dim]
 *   out          [batch, num_heads_q, head_dim] bf16; row stride out_row_stride
 *   lse          nullable; [batch, num_heads_q] float32
 *   num_heads_q  a multiple of num_heads_kv, at most 64 query heads per KV
 *                head (ATTN_ERR_UNSUPPORTED above); past 16 the heads of a
 *                KV head are spread over several CTAs in groups of 16
 *   cache_seqlens int32 [batch]: keys 0 .. cache_seqlens[b]-1 are attended
 *                (they include the current token, stored beforehand); values
 *                outside [0, max_cache_seqlen] are clamped and reported as
 *                ATTN_ERR_DEVICE_INDEX
 *   block_table  int32 [batch, block_table_stride]
 *   max_cache_seqlen host-side upper bound of cache_seqlens
 *   num_splits   0 = chosen by the library; otherwise the number of KV splits
 *                per sequence (1..64).  Split partials are merged exactly by a
 *                log-sum-exp combine.
 *   workspace    at least attn_decode_workspace_size(...) bytes
 * ------------------------------------------------------------------------ */
ATTN_API attn_status attn_decode_paged(const void *q, const void *k_cache, const void *v_cache, void *out,
                              float *lse, const int32_t *cache_seqlens, const int32_t *block_table,
                              int block_table_stride, int batch, int num_heads_q, int num_heads_kv,
                              int head_dim, int block_size, int64_t num_blocks, int max_cache_seqlen,
                              float softmax_scale, int num_splits,
                              int64_t q_row_stride, int64_t out_row_stride,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace attn_decode_paged needs for these sizes
 * (the same num_splits rule as attn_decode_paged, 0 = the library's choice). */
ATTN_API size_t attn_decode_workspace_size(int batch, int num_heads_q, int num_heads_kv, int head_dim,
                                  int max_cache_seqlen, int num_splits);

/* The split count attn_decode_paged uses for these sizes (num_splits as passed). */
ATTN_API int attn_decode_num_splits(int batch, int num_heads_kv, int max_cache_seqlen, int num_splits);

/* ------------------------------------------------------------------------
 * attn_decode_paged_noalloc -- attn_decode_paged for callers that cannot
 * allocate device memory when they decode.  The article has no counterpart:
 * this entry point exists for deployments such as a serving loop that gave
 * all free device memory to its paged KV-cache pool at start-up, or a hot
 * path that must not call cudaMalloc because it can synchronise the device.
 *
 * Arguments and results are those of attn_decode_paged without the
 * workspace: the split partials go to a scratch array reserved statically in
 * the library (ATTN_DECODE_NOALLOC_SCRATCH_BYTES, 32 MiB, held on every GPU
 * that loads the library until the process exits).  The call allocates
 * nothing.
 *  - The first call on a device looks up the scratch address on that device
 *    (with it current); make that first call before any stream capture.
 *  - Every call shares the one array: calls that overlap on the GPU (on
 *    streams with no ordering between them) race and give wrong results.
 *    Nothing in the array needs clearing between calls.
 *  - num_splits = 0 picks the library's split count, lowered until the
 *    partials fit the scratch (one split needs none).  An explicit num_splits
 *    whose partials (batch * num_heads_q * num_splits * (head_dim + 1) floats)
 *    do not fit is rejected with ATTN_ERR_WORKSPACE_TOO_SMALL.
 * ------------------------------------------------------------------------ */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)

ATTN_API attn_status attn_decode_paged_noalloc(const void *q, const void *k_cache, const void *v_cache, void *out,
                                               float *lse, const int32_t *cache_seqlens,
                                               const int32_t *block_table, int block_table_stride, int batch,
                                               int num_heads_q, int num_heads_kv, int head_dim, int block_size,
                                               int64_t num_blocks, int max_cache_seqlen, float softmax_scale,
                                               int num_splits, int64_t q_row_stride, int64_t out_row_stride,
                                               void *stream);

/* ------------------------------------------------------------------------
 * store_kvcache -- scatter this step's K/V rows into the paged caches before
 * attention (the article's Prefill section: store_kvcache(k, v, k_cache,
 * v_cache, slot_mapping)).
 *
 *   k, v          [num_tokens, num_heads_kv, head_dim], row strides
 *                 k_row_stride / v_row_stride (elements, 0 = packed)
 *   k_cache, v_cache  viewed as [num_slots, num_heads_kv, head_dim]
 *                 (num_slots = num_blocks * block_size)
 *   v16_cache     nullable: an fp16 cache shaped like v_cache that also
 *                 receives V / 16 (round to nearest) at the same slots, for
 *                 attn_varlen_fwd's and attn_kvcache_fwd's v16_cache argument;
 *                 values with |v| >= 2^20 (or non-finite) saturate and are
 *                 reported as ATTN_ERR_DEVICE_RANGE
 *   slot_mapping  int64 [num_tokens]: flat slot block_id * block_size +
 *                 offset; a negative slot skips the token; a slot >=
 *                 num_slots is skipped and flagged in the error word.
 *                 Duplicate slots are a caller error (last writer undefined).
 * head_dim may be any even value here (the copy is type-agnostic).
 * ------------------------------------------------------------------------ */
ATTN_API attn_status store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache,
                          void *v16_cache, const int64_t *slot_mapping, int64_t num_tokens,
                          int num_heads_kv, int head_dim, int64_t k_row_stride, int64_t v_row_stride,
                          int64_t num_slots, void *stream);

/* ------------------------------------------------------------------------
 * attn_padded_fwd -- prefill of a padded batch: every sequence occupies a
 * fixed number of rows and only its first seqlens[b] rows are real (the layout
 * the article contrasts with varlen packing, section "Prefill": padding plus a
 * mask instead of cu_seqlens).  Same attention as attn_varlen_fwd; the padding
 * rows are never read as keys or values that count, whatever they hold.
 *
 *   q, out       [batch, seqlen_q, num_heads_q, head_dim] bf16, packed
 *   k, v         [batch, seqlen_k, num_heads_kv, head_dim] bf16, packed
 *   lse          nullable; [num_heads_q, batch * seqlen_q] float32
 *   seqlens_q    nullable int32 [batch]: real query rows of sequence b
 *                (NULL: all seqlen_q); seqlens_k likewise for the keys.  Values
 *                outside [0, seqlen] are clamped and reported as
 *                ATTN_ERR_DEVICE_INDEX.
 *   causal       bottom-right on the real lengths (query i sees keys
 *                j <= seqlens_k[b] - seqlens_q[b] + i)
 *   workspace    at least attn_padded_workspace_size(...) bytes, 256-byte aligned
 * Output rows and lse entries of padding rows are left as they were.
 * Returns the statuses of attn_varlen_fwd.
 * ------------------------------------------------------------------------ */
ATTN_API attn_status attn_padded_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                                     const int32_t *seqlens_q, const int32_t *seqlens_k, int batch, int seqlen_q,
                                     int seqlen_k, int num_heads_q, int num_heads_kv, int head_dim,
                                     float softmax_scale, int causal, void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Workspace bytes attn_padded_fwd needs (0 for invalid sizes). */
ATTN_API size_t attn_padded_workspace_size(int batch, int seqlen_q, int seqlen_k, int num_heads_q,
                                           int num_heads_kv, int head_dim);

/* ------------------------------------------------------------------------
 * attn_kvcache_fwd -- several new query tokens per sequence against a paged
 * KV cache ([A] "Decode": flash_attn_with_kvcache(q, k_cache, v_cache,
 * cache_seqlens, block_table, softmax_scale, causal) with q of shape
 * [B, seqlen_q, H, D] and seqlen_q >= 1: chunked append, speculative
 * verification).  Two routes, chosen from the sizes and from whether
 * v16_cache is given:
 *  - seqlen_q * (num_heads_q / num_heads_kv) <= 64 at head_dim 64, <= 16 at
 *    head_dim 128 or with v16_cache: the split-KV decode kernel of attn_decode_paged with
 *    one query column per (new token, head), up to 16 columns per CTA; the
 *    cache is read from HBM once (CTAs holding other columns of the same KV
 *    head re-read it from L2).  With seqlen_q = 1 the result equals
 *    attn_decode_paged's bit for bit.
 *  - otherwise: cu_seqlens_q = b * seqlen_q and cu_seqlens_k = prefix sums of
 *    cache_seqlens are computed on the device, then the paged varlen prefill
 *    (attn_varlen_fwd) runs; up to 128 query rows per KV head at head_dim 128
 *    that is the one-slot kernel, which converts V tiles itself when no
 *    v16_cache is given.
 *
 *   q, out       [batch * seqlen_q, num_heads_q, head_dim] bf16, packed
 *                (the article's [B, seqlen_q, H, D])
 *   lse          nullable; [num_heads_q, batch * seqlen_q] float32
 *   cache_seqlens int32 [batch]: keys 0 .. cache_seqlens[b]-1 of sequence b,
 *                including its seqlen_q new tokens (stored beforehand); values
 *                outside [0, max_cache_seqlen] are clamped and reported as
 *                ATTN_ERR_DEVICE_INDEX
 *   causal       bottom-right: new token i sees keys j <= cache_seqlens[b] -
 *                seqlen_q + i; 0 = every cached key
 *   block_table, block_size, num_blocks: as for attn_varlen_fwd (paged mode)
 *   v16_cache    nullable: the fp16 V / 16 cache kept by store_kvcache.  Both
 *                routes then read V / 16 from it instead of V: the prefill route
 *                converts nothing, and the decode route multiplies it by one fp16
 *                term 16 P (11 significant bits) instead of P's two bf16 terms,
 *                half the P V work
 *   workspace    at least attn_kvcache_workspace_size(...) bytes (enough for
 *                either route, with or without v16_cache), 256-byte
 *                aligned.  On the decode route it holds the split partials
 *                (at most 64 splits of fp32 rows); on the prefill route without
 *                v16_cache and past one query slot (or at head_dim 64) the fp16
 *                copy of V for batch * max_cache_seqlen keys, so there it grows
 *                with the cache length.
 * Returns the statuses of attn_varlen_fwd.
 * ------------------------------------------------------------------------ */
ATTN_API attn_status attn_kvcache_fwd(const void *q, const void *k_cache, const void *v_cache, void *out,
                                      float *lse, const int32_t *cache_seqlens, const int32_t *block_table,
                                      int block_table_stride, int batch, int seqlen_q, int num_heads_q,
                                      int num_heads_kv, int head_dim, int block_size, int64_t num_blocks,
                                      int max_cache_seqlen, float softmax_scale, int causal,
                                      const void *v16_cache, void *workspace, size_t workspace_bytes,
                                      void *stream);

/* Workspace bytes attn_kvcache_fwd needs on either route, with or without
 * v16_cache (0 for invalid sizes). */
ATTN_API size_t attn_kvcache_workspace_size(int batch, int seqlen_q, int num_heads_q, int num_heads_kv,
                                            int head_dim, int max_cache_seqlen);

/* ------------------------------------------------------------------------
 * attn_softmax_rows -- y = softmax(x) along every row of a matrix, with the
 * online two-pass algorithm of the article's section 减少遍历次数的“在线
 * Softmax”: pass 1 runs the maximum m and the proxy denominator
 * d' = d' * e^(m_old - m_new) + e^(x - m_new) (partial (m, d') pairs of
 * threads, warps and CTAs merge by the same rule), pass 2 writes
 * e^(x - m) / d'.  Arithmetic in fp32; no overflow for any finite input.
 *
 *   x, y          [rows, cols], row strides x_row_stride / y_row_stride in
 *                 elements (0 = cols); y may be x (in place)
 *   dtype         ATTN_DTYPE_F32 (x and y float32) or ATTN_DTYPE_BF16 (x and
 *                 y bfloat16, y rounded to nearest even)
 * A row whose maximum is not finite (all -inf, or a +inf or NaN in it) gives
 * NaN, as the definition does.  HBM-bound: one read and one write of the
 * matrix for 16-byte-aligned rows of up to 512 KB (a warp, a CTA or a
 * thread-block cluster per row, the row held on chip between the passes);
 * longer or unaligned rows are read twice, the second time mostly from L2.
 * A bounded wait that gives up (rows up to 16 KB, streamed through shared
 * memory) is reported by attn_get_last_device_error as
 * ATTN_ERR_DEVICE_TIMEOUT.
 * ------------------------------------------------------------------------ */
enum { ATTN_DTYPE_F32 = 0, ATTN_DTYPE_BF16 = 1 };

ATTN_API attn_status attn_softmax_rows(const void *x, void *y, int64_t rows, int cols, int64_t x_row_stride,
                                       int64_t y_row_stride, int dtype, void *stream);

/* ------------------------------------------------------------------------
 * Diagnostics
 * ------------------------------------------------------------------------ */

/* Static text for a status code. */
ATTN_API const char *attn_status_string(attn_status status);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns ATTN_OK if no kernel recorded a problem since the
 * last call, else ATTN_ERR_DEVICE_INDEX, ATTN_ERR_DEVICE_TIMEOUT or
 * ATTN_ERR_DEVICE_RANGE (in that order of precedence), or
 * ATTN_ERR_LAUNCH_FAILED if the stream itself reports a CUDA error.  *detail (nullable) receives the raw error word. */
ATTN_API attn_status attn_get_last_device_error(void *stream, uint32_t *detail);

/* Failure-detection self-test: one small kernel in which a bounded mbarrier
 * wait runs out on purpose (nothing ever completes the barrier; no fault, no
 * trap).  The first waiter gives up after the library's wait limit (about one
 * second), records ATTN_ERR_DEVICE_TIMEOUT in the device error word and raises
 * the kernel's abort flag; a second waiter, which started half a limit later,
 * must give up on seeing that flag before its own limit runs out.  Synchronises
 * `stream`.  result (host, 4 entries): the first waiter's success flag (0 when
 * it gave up, as it must) and nanoseconds waited, then the same for the
 * second.  The context stays usable; attn_get_last_device_error then reports
 * ATTN_ERR_DEVICE_TIMEOUT and clears the word.  Returns ATTN_OK,
 * ATTN_ERR_INVALID_ARG (result NULL), ATTN_ERR_NO_DEVICE, ATTN_ERR_UNSUPPORTED
 * or ATTN_ERR_LAUNCH_FAILED. */
ATTN_API attn_status attn_selftest_bounded_wait(void *stream, unsigned long long *result);

/* ATTN_ABI_VERSION of the loaded library. */
ATTN_API int attn_abi_version(void);

/* Measurement hook (no counterpart in the article: it exists so that a
 * benchmark can time the dominant kernel of a call by itself).  `before` and
 * `after` are the caller's cudaEvent_t handles (cast to void *); the library
 * neither creates nor destroys them.  While both are non-NULL, every later
 * attn_varlen_fwd, attn_decode_paged, attn_decode_paged_noalloc and
 * store_kvcache call made from the same host thread records `before` on its
 * stream just before launching its main kernel (the attention kernel of the
 * prefill; the split-KV kernel of the decode; the scatter kernel of the store)
 * and `after` just after it, so
 * cudaEventElapsedTime(before, after) is that kernel's device time.  The
 * scheduling and V-conversion kernels of the prefill and the combine kernel
 * of the decode fall outside.  Pass NULL, NULL to switch it off (the
 * default).  Event-record errors are not reported. */
ATTN_API void attn_set_kernel_events(void *before, void *after);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_VARLEN_H */
