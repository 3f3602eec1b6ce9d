// store_kvcache.cu -- scatter of this step's K/V rows into the paged caches
// by slot_mapping ("从零实现 vLLM (1.3)：如何加速 Attention 计算", section
// "Prefill": store_kvcache(k, v, k_cache, v_cache, slot_mapping) runs before
// the attention call).
//
// Pure data movement, HBM-bound: every token moves 2 * row_bytes in and out.
// The work is a flat list of 16-byte chunks (token, K or V, chunk of the row).
// One wave of CTAs covers it (the grid is what fits on the SMs at once), each
// thread taking chunks idx, idx + T, idx + 2T, ... (T = threads in the grid) in
// batches of kStoreUnroll: all loads of a batch (data and slot) are issued
// before its stores, so a thread keeps 128 bytes in flight.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace attn {

constexpr int kStoreThreads = 256;
constexpr int kStoreUnroll = 8;
constexpr int kStoreMinBlocks = 3;   // CTAs per SM the register budget must allow

// row_chunks = row bytes / 16 (K and V rows have the same size).  v16_cache
// (nullable): also write V / 16 as fp16 at the same slot, the form the paged
// prefill's P V product reads; |v| >= 2^20 (or non-finite) does not fit and is
// clamped and reported.
__global__ void __launch_bounds__(kStoreThreads, kStoreMinBlocks) store_kvcache_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, uint4 *__restrict__ v16_cache, const int64_t *__restrict__ slot_mapping,
    int64_t num_tokens, int row_chunks, int64_t k_stride_chunks, int64_t v_stride_chunks, int64_t num_slots,
    uint32_t *err) {
    const int64_t per_tok = 2 * (int64_t)row_chunks;   // K chunks then V chunks
    const int64_t total = num_tokens * per_tok;
    const int64_t T = (int64_t)gridDim.x * kStoreThreads;
    uint32_t big = 0;
    bool bad = false;
    for (int64_t base = (int64_t)blockIdx.x * kStoreThreads + threadIdx.x; base < total; base += T * kStoreUnroll) {
        uint4 val[kStoreUnroll];
        int64_t slot[kStoreUnroll];
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const int64_t idx = base + u * T;
            slot[u] = -1;
            if (idx < total) {
                const int64_t tok = idx / per_tok;
                const int c = (int)(idx - tok * per_tok);
                slot[u] = __ldg(slot_mapping + tok);
                val[u] = c >= row_chunks ? ldg_stream16(v + tok * v_stride_chunks + (c - row_chunks))
                                         : ldg_stream16(k + tok * k_stride_chunks + c);
            }
        }
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            int64_t s = slot[u];
            if (s >= num_slots) {
                bad = true;
                s = -1;
            }
            if (s < 0) continue;
            const int c = (int)((base + u * T) % per_tok);   // recomputed: fewer live registers
            const bool is_v = c >= row_chunks;
            const int64_t d = s * row_chunks + (is_v ? c - row_chunks : c);
            (is_v ? v_cache : k_cache)[d] = val[u];
            if (is_v && v16_cache) {
                const uint4 w = val[u];
                big = __vmaxu2(big, __vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu));
                big = __vmaxu2(big, __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
                v16_cache[d] = make_uint4(bf16x2_to_f16x2_div16(w.x), bf16x2_to_f16x2_div16(w.y),
                                          bf16x2_to_f16x2_div16(w.z), bf16x2_to_f16x2_div16(w.w));
            }
        }
    }
    // 0x4980 is the bf16 bit pattern of 2^20
    const bool range = (big & 0xFFFFu) >= 0x4980u || (big >> 16) >= 0x4980u;
    const unsigned any_bad = __ballot_sync(0xffffffffu, bad), any_range = __ballot_sync(0xffffffffu, range);
    if ((threadIdx.x & 31) == 0) {
        if (any_bad) record_error(err, ERR_INDEX | SRC_STORE);
        if (any_range) record_error(err, ERR_RANGE | SRC_STORE);
    }
}

// Fallback for rows that are not a multiple of 16 bytes (2-byte elements).
__global__ void __launch_bounds__(kStoreThreads) store_kvcache_kernel_b16(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, uint16_t *__restrict__ k_cache,
    uint16_t *__restrict__ v_cache, __half *__restrict__ v16_cache, const int64_t *__restrict__ slot_mapping,
    int64_t num_tokens, int row_elems, int64_t k_stride, int64_t v_stride, int64_t num_slots, uint32_t *err) {
    bool big = false;
    for (int64_t t = blockIdx.x; t < num_tokens; t += gridDim.x) {
        int64_t s = __ldg(slot_mapping + t);
        if (s < 0) continue;
        if (s >= num_slots) {
            if (threadIdx.x == 0) record_error(err, ERR_INDEX | SRC_STORE);
            continue;
        }
        for (int e = threadIdx.x; e < row_elems; e += kStoreThreads) {
            k_cache[s * row_elems + e] = k[t * k_stride + e];
            const uint16_t w = v[t * v_stride + e];
            v_cache[s * row_elems + e] = w;
            if (v16_cache) {
                big = big || (w & 0x7FFFu) >= 0x4980u;
                const float x = __uint_as_float((uint32_t)w << 16) * 0.0625f;
                v16_cache[s * row_elems + e] = __float2half_rn(fminf(fmaxf(x, -65504.f), 65504.f));
            }
        }
    }
    if (big) record_error(err, ERR_RANGE | SRC_STORE);
}

cudaError_t launch_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache, void *v16_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens, int row_elems,
                                 int64_t k_stride, int64_t v_stride, int64_t num_slots, int num_sms,
                                 uint32_t *err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const bool vec = (row_elems % 8 == 0) && (k_stride % 8 == 0) && (v_stride % 8 == 0) &&
                     ((uintptr_t)k % 16 == 0) && ((uintptr_t)v % 16 == 0) && ((uintptr_t)k_cache % 16 == 0) &&
                     ((uintptr_t)v_cache % 16 == 0) && ((uintptr_t)v16_cache % 16 == 0);
    if (vec) {
        // one wave: the CTAs that fit on the SMs together (looked up once per device)
        static std::once_flag once[kMaxDev];
        static int per_sm[kMaxDev];
        int dev = 0;
        cudaError_t e0 = cudaGetDevice(&dev);
        if (e0 != cudaSuccess) return e0;
        if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
        std::call_once(once[dev], [&] {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, store_kvcache_kernel, kStoreThreads, 0) !=
                    cudaSuccess ||
                n < 1) {
                cudaGetLastError();
                n = kStoreMinBlocks;
            }
            per_sm[dev] = n;
        });
        const int64_t chunks = num_tokens * (row_elems / 4);   // 16-byte chunks of K and V
        const int64_t need = (chunks + (int64_t)kStoreThreads * kStoreUnroll - 1) / ((int64_t)kStoreThreads * kStoreUnroll);
        int64_t grid = (int64_t)num_sms * per_sm[dev];
        if (grid > need) grid = need;
        main_kernel_event_before(stream);
        store_kvcache_kernel<<<(unsigned)grid, kStoreThreads, 0, stream>>>(
            (const uint4 *)k, (const uint4 *)v, (uint4 *)k_cache, (uint4 *)v_cache, (uint4 *)v16_cache, slot_mapping,
            num_tokens, row_elems / 8, k_stride / 8, v_stride / 8, num_slots, err);
        main_kernel_event_after(stream);
    } else {
        int64_t grid = num_sms * 8;
        if (grid > num_tokens) grid = num_tokens;
        main_kernel_event_before(stream);
        store_kvcache_kernel_b16<<<(unsigned)grid, kStoreThreads, 0, stream>>>(
            (const uint16_t *)k, (const uint16_t *)v, (uint16_t *)k_cache, (uint16_t *)v_cache, (__half *)v16_cache,
            slot_mapping, num_tokens, row_elems, k_stride, v_stride, num_slots, err);
        main_kernel_event_after(stream);
    }
    return cudaGetLastError();
}

}  // namespace attn
