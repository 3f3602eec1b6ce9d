// store_kvcache.cu -- scatter of this step's K/V rows into the paged caches
// by slot_mapping ("从零实现 vLLM (1.3)：如何加速 Attention 计算", section
// "Prefill": store_kvcache(k, v, k_cache, v_cache, slot_mapping) runs before
// the attention call).
//
// Pure data movement, HBM-bound: every token moves 2 * row_bytes in and out.
// One CTA handles kTokPerIter tokens per loop trip; each thread owns 16-byte
// chunks, issuing all its loads before its stores so several requests are
// in flight per thread.  The grid is a multiple of the SM count and strides
// over the tokens.
#include "common.cuh"
#include "kernels.h"

namespace attn {

constexpr int kStoreThreads = 256;
constexpr int kTokPerIter = 4;

// row_chunks = row bytes / 16 (K and V rows have the same size)
__global__ void __launch_bounds__(kStoreThreads) store_kvcache_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, const int64_t *__restrict__ slot_mapping, int64_t num_tokens, int row_chunks,
    int64_t k_stride_chunks, int64_t v_stride_chunks, int64_t num_slots, uint32_t *err) {
    const int per_tok = 2 * row_chunks;  // K chunks then V chunks
    for (int64_t t0 = (int64_t)blockIdx.x * kTokPerIter; t0 < num_tokens; t0 += (int64_t)gridDim.x * kTokPerIter) {
        int64_t slot[kTokPerIter];
#pragma unroll
        for (int u = 0; u < kTokPerIter; ++u) {
            int64_t t = t0 + u;
            int64_t s = t < num_tokens ? __ldg(slot_mapping + t) : -1;
            if (s >= num_slots) {
                if (threadIdx.x == 0) record_error(err, ERR_INDEX | SRC_STORE);
                s = -1;
            }
            slot[u] = s;
        }
        for (int c = threadIdx.x; c < per_tok; c += kStoreThreads) {
            const bool is_v = c >= row_chunks;
            const int e = is_v ? c - row_chunks : c;
            uint4 val[kTokPerIter];
#pragma unroll
            for (int u = 0; u < kTokPerIter; ++u) {
                if (slot[u] >= 0) {
                    const int64_t t = t0 + u;
                    val[u] = is_v ? __ldg(v + t * v_stride_chunks + e) : __ldg(k + t * k_stride_chunks + e);
                }
            }
#pragma unroll
            for (int u = 0; u < kTokPerIter; ++u) {
                if (slot[u] >= 0) {
                    uint4 *dst = (is_v ? v_cache : k_cache) + slot[u] * row_chunks + e;
                    *dst = val[u];
                }
            }
        }
    }
}

// Fallback for rows that are not a multiple of 16 bytes (2-byte elements).
__global__ void __launch_bounds__(kStoreThreads) store_kvcache_kernel_b16(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, uint16_t *__restrict__ k_cache,
    uint16_t *__restrict__ v_cache, const int64_t *__restrict__ slot_mapping, int64_t num_tokens, int row_elems,
    int64_t k_stride, int64_t v_stride, int64_t num_slots, uint32_t *err) {
    for (int64_t t = blockIdx.x; t < num_tokens; t += gridDim.x) {
        int64_t s = __ldg(slot_mapping + t);
        if (s < 0) continue;
        if (s >= num_slots) {
            if (threadIdx.x == 0) record_error(err, ERR_INDEX | SRC_STORE);
            continue;
        }
        for (int e = threadIdx.x; e < row_elems; e += kStoreThreads) {
            k_cache[s * row_elems + e] = k[t * k_stride + e];
            v_cache[s * row_elems + e] = v[t * v_stride + e];
        }
    }
}

cudaError_t launch_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens, int row_elems,
                                 int64_t k_stride, int64_t v_stride, int64_t num_slots, int num_sms,
                                 uint32_t *err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const bool vec = (row_elems % 8 == 0) && (k_stride % 8 == 0) && (v_stride % 8 == 0) &&
                     ((uintptr_t)k % 16 == 0) && ((uintptr_t)v % 16 == 0) && ((uintptr_t)k_cache % 16 == 0) &&
                     ((uintptr_t)v_cache % 16 == 0);
    if (vec) {
        int64_t iters = (num_tokens + kTokPerIter - 1) / kTokPerIter;
        int64_t grid = num_sms * 8;
        if (grid > iters) grid = iters;
        store_kvcache_kernel<<<(unsigned)grid, kStoreThreads, 0, stream>>>(
            (const uint4 *)k, (const uint4 *)v, (uint4 *)k_cache, (uint4 *)v_cache, slot_mapping, num_tokens,
            row_elems / 8, k_stride / 8, v_stride / 8, num_slots, err);
    } else {
        int64_t grid = num_sms * 8;
        if (grid > num_tokens) grid = num_tokens;
        store_kvcache_kernel_b16<<<(unsigned)grid, kStoreThreads, 0, stream>>>(
            (const uint16_t *)k, (const uint16_t *)v, (uint16_t *)k_cache, (uint16_t *)v_cache, slot_mapping,
            num_tokens, row_elems, k_stride, v_stride, num_slots, err);
    }
    return cudaGetLastError();
}

}  // namespace attn
