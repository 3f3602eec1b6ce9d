// kernels.h -- host-side declarations shared by the C-ABI layer (api.cu) and
// the kernel translation units.  Parameter blocks are plain structs passed by
// value to the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// devices the per-device lazy set-ups (function attributes, symbol addresses) cover
constexpr int kMaxDev = 64;

struct DecodeParams {
    const __nv_bfloat16 *q;      // [B * Sq, Hq, D], row stride q_row_stride
    __nv_bfloat16 *out;          // [B * Sq, Hq, D], row stride out_row_stride
    float *lse;                  // null, or element (row, h) at row * lse_row_stride + h * lse_head_stride
    float *o_part;               // [B * Sq, Hq, S, D]  split partial outputs (normalised)
    float *lse_part;             // [B * Sq, Hq, S]     split partial log2-sum-exp
    const int32_t *cache_seqlens;
    const int32_t *block_table;
    int64_t q_row_stride, out_row_stride;
    int64_t lse_row_stride, lse_head_stride;
    int bt_stride, block_size, rows_per_box, num_splits, split_tokens;
    int64_t num_blocks;
    int Hq, Hkv, G;
    int Sq;                      // query tokens per sequence; Sq * G <= 64
    int ncg;                     // column groups: CTAs per (split, KV head, sequence), 16 columns each
    int causal;                  // bottom-right: token t sees keys j <= L - Sq + t
    int max_seqlen;              // cache_seqlens outside [0, max_seqlen] are clamped and reported
    int v16;                     // 1: V tiles are the fp16 V / 16 cache (PV on one fp16 term P' = 16 P)
    float scale_log2;            // softmax_scale * log2(e)
    uint32_t *err;
};

struct PrefillParams {
    const __nv_bfloat16 *v;      // contiguous [total_k, Hkv, D] (row stride v_row_stride) or the V cache
    __half *v16;                 // workspace: V / 16 in fp16, [total_k, Hkv, D] by logical key
    __nv_bfloat16 *out;          // [total_q, Hq, D], row stride out_row_stride
    float *lse;                  // [Hq, total_q] or null
    const int32_t *cu_q, *cu_k;
    const int32_t *seqused_q;    // null, or [batch]: sequence b uses the first seqused_q[b] rows of its range
    const int32_t *seqused_k;    // null, or [batch]: the same for its keys
    const int32_t *block_table;  // null: contiguous K/V
    int64_t total_q, total_k, out_row_stride, v_row_stride;
    int64_t num_blocks;
    int bt_stride, block_size, rows_per_box;
    int batch, Hq, Hkv, G, causal, head_dim, max_seqlen_k;
    int max_pairs;               // slot pairs per sequence at max_seqlen_q
    int v16_paged;               // 1: V' tiles come from a paged fp16 V / 16 cache through the block
                                 //    table (written by store_kvcache); no conversion pass
    int num_ctas;                // grid size: persistent CTAs (one per SM, at most the possible units)
    int one_slot;                // 1: max_seqlen_q <= 128 / G, every sequence fits one query slot
    int v_cvt;                   // 1 (one-slot launches without a V' cache): V tiles are loaded as bf16
                                 //    from v and converted to V' in shared memory; no conversion pass
    int2 *units;                 // workspace: (sequence, pair | kv_head << 16), scheduled order
    int *unit_count;             // workspace: [0] number of units
    float scale_log2;            // softmax_scale * log2(e), > 0
    uint32_t *err;
};

cudaError_t launch_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache, void *v16_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens, int row_elems,
                                 int64_t k_stride, int64_t v_stride, int64_t num_slots, int num_sms,
                                 uint32_t *err, cudaStream_t stream);

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p, int batch,
                          int head_dim, cudaStream_t stream);

// static scratch of the allocation-free decode entry point (device address on
// the current device, looked up on first use)
cudaError_t decode_noalloc_scratch(float **ptr, size_t *bytes);

// rows per query slot of the prefill kernel (a slot packs 128 / G tokens x G heads)
constexpr int kPrefillSlotRows = 128;
constexpr int kPrefillKeyTile = 128;

// measurement hook: record the caller's events (if set on this thread) right
// before and right after the main kernel of a call
void main_kernel_event_before(cudaStream_t stream);
void main_kernel_event_after(cudaStream_t stream);

cudaError_t launch_softmax_rows(const void *x, void *y, int64_t rows, int cols, int64_t x_row_stride,
                                int64_t y_row_stride, int bf16, int sms, uint32_t *err, cudaStream_t stream);

cudaError_t launch_padded_cu(int batch, int seqlen_q, int seqlen_k, int32_t *cu_q, int32_t *cu_k,
                             cudaStream_t stream);

cudaError_t launch_kvcache_cu(const int32_t *cache_seqlens, int batch, int seqlen_q, int max_cache_seqlen,
                              int32_t *cu_q, int32_t *cu_k, uint32_t *err, cudaStream_t stream);

cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const CUtensorMap &omap, const PrefillParams &p, int head_dim, cudaStream_t stream);

}  // namespace attn
