// api.cu -- the C ABI (include/attn_varlen.h): argument checks, TMA tensor-map
// encoding, launch sizing, and the device error word.
//
// Call shapes follow "从零实现 vLLM (1.3)：如何加速 Attention 计算", section
// "Attention 源码分析": store_kvcache(k, v, k_cache, v_cache, slot_mapping),
// flash_attn_varlen_func(q, k, v, max_seqlen_q, cu_seqlens_q, max_seqlen_k,
// cu_seqlens_k, softmax_scale, causal, block_table) and
// flash_attn_with_kvcache(q.unsqueeze(1), k_cache, v_cache, cache_seqlens,
// block_table, softmax_scale, causal).
#include <math.h>

#include <mutex>
#include <stdint.h>
#include <string.h>

#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "kernels.h"

using namespace attn;

namespace {

constexpr int kMaxDevices = 64;

// one error word per device; kernels get its address
__device__ uint32_t g_attn_error_word;

struct DevInfo {
    attn_status st = ATTN_ERR_NO_DEVICE;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *err = nullptr;
};
DevInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

// Attributes of the current device, queried once per device (also when several
// host threads make their first call together).
attn_status dev_info(DevInfo **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return ATTN_ERR_NO_DEVICE;
    }
    DevInfo &d = g_dev[dev];
    std::call_once(g_dev_once[dev], [&] {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_attn_error_word) != cudaSuccess) {
            cudaGetLastError();
            d.st = ATTN_ERR_NO_DEVICE;
        } else {
            d.st = ATTN_OK;
        }
    });
    if (d.st != ATTN_OK) return d.st;
    *out = &d;
    return ATTN_OK;
}

// the kernels are built for sm_103a only
attn_status check_arch(const DevInfo *d) {
    return (d->cc_major == 10 && d->cc_minor == 3) ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's cuTensorMapEncodeTiled, looked up once (a function-local static
// is initialised once even under concurrent first calls)
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
        return (EncodeTiledFn) nullptr;
    }();
    return fn;
}

// bf16 tensor [rows, heads, dim] with a row stride (elements) viewed as a 3-D
// TMA map (dim, heads, rows), 128-byte swizzle, box (64, box_heads, box_rows).
bool make_map(CUtensorMap *map, const void *base, int64_t rows, int heads, int dim, int64_t row_stride,
              int box_heads, int box_rows, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)row_stride * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, dtype, 3, const_cast<void *>(base), gdim, gstride, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Row stride in elements: 0 selects the packed default; otherwise it must
// cover a row and keep rows 16-byte aligned.
bool fix_stride(int64_t *stride, int64_t packed) {
    if (*stride == 0) *stride = packed;
    return *stride >= packed && (*stride % 8) == 0;
}

constexpr int kMaxSplits = 64;
constexpr int kDecodeMaxColumns = 64;   // Sq x G query columns per KV head on the decode kernel
// ... with the fp16 V / 16 cache: past one column group of 16 the paged prefill
// (tcgen05, no conversion pass with that cache) streams the cache faster
constexpr int kDecodeMaxColumnsV16 = 16;
// ... and without it at head_dim 128: past one column group the one-slot prefill,
// converting each V tile in shared memory, streams the cache faster
constexpr int kDecodeMaxColumnsCvt = 16;
constexpr int kDecodeTile = 64;

// Tokens a split streams at most when the library chooses the split count: long
// enough that a CTA's fixed costs (query columns, barriers, the merge of its warps,
// its partials and their combine) stay small, short enough to balance very
// different lengths.  When a KV head's query columns span several column-group
// CTAs those fixed costs are paid once per group: longer splits.
constexpr int kSplitTokens = 4096;
constexpr int kSplitTokensGroups = 8192;

int choose_splits(int num_sms, int batch, int num_heads_kv, int max_len, int requested,
                  int split_cap = kSplitTokens) {
    if (max_len <= 0) return 1;
    const int max_tiles = (max_len + kDecodeTile - 1) / kDecodeTile;
    int s;
    if (requested > 0) {
        s = requested;
    } else {
        // each split streams at most split_cap tokens, and there are at least ~2
        // CTAs per SM in total
        const int s_balance = (max_len + split_cap - 1) / split_cap;
        const int64_t units = (int64_t)batch * num_heads_kv;
        const int s_par = (int)((2LL * 2 * num_sms + units - 1) / units);
        s = s_balance > s_par ? s_balance : s_par;
    }
    if (s > kMaxSplits) s = kMaxSplits;
    if (s > max_tiles) s = max_tiles;
    if (s < 1) s = 1;
    return s;
}

int split_tokens_for(int max_len, int splits) {
    int per = (max_len + splits - 1) / splits;
    return ((per + kDecodeTile - 1) / kDecodeTile) * kDecodeTile;
}

// Split plan of the decode kernel: the split count for these sizes and the
// tokens per split (a multiple of the 64-token tile), with splits * tokens
// covering max_len.
void decode_plan(int num_sms, int batch, int num_heads_kv, int max_len, int requested, int *splits, int *split_tok,
                 int split_cap = kSplitTokens) {
    int s = choose_splits(num_sms, batch, num_heads_kv, max_len, requested, split_cap);
    const int tok = split_tokens_for(max_len > 0 ? max_len : 1, s);
    s = max_len > 0 ? (max_len + tok - 1) / tok : 1;
    *splits = s < 1 ? 1 : s;
    *split_tok = tok;
}

// Bytes of split partials: an fp32 output row and a log-sum-exp per query row,
// head and split.
size_t decode_partial_bytes(int batch, int seqlen_q, int num_heads_q, int head_dim, int splits) {
    return splits > 1 ? (size_t)batch * seqlen_q * num_heads_q * splits * (head_dim + 1) * sizeof(float) : 0;
}

// The kv-cache entry runs on the decode kernel when the Sq x G query rows of a
// KV head fit four column groups of 16 (one group at head_dim 128, with or without
// the fp16 V / 16 cache, and with that cache at head_dim 64, where the prefill can
// take the group size); otherwise on the paged varlen prefill.
bool kvcache_on_decode(int batch, int seqlen_q, int num_heads_q, int num_heads_kv, int head_dim, bool v16) {
    if (num_heads_q <= 0 || num_heads_kv <= 0 || num_heads_q % num_heads_kv) return false;
    if (head_dim != 64 && head_dim != 128) return false;
    if (batch > 65535 || num_heads_kv > 65535) return false;
    const int G = num_heads_q / num_heads_kv;
    // the prefill packs 128 / G tokens x G heads per query slot: larger groups stay here
    const bool prefill_ok = G <= kPrefillSlotRows;
    int cap = kDecodeMaxColumns;
    if (prefill_ok && v16) cap = kDecodeMaxColumnsV16;
    else if (prefill_ok && head_dim == 128) cap = kDecodeMaxColumnsCvt;
    return (int64_t)seqlen_q * G <= cap;
}

struct DecodeCall {
    const void *q, *k_cache, *v_cache;
    void *out;
    float *lse;
    const int32_t *cache_seqlens, *block_table;
    int bt_stride, batch, seqlen_q, Hq, Hkv, head_dim, block_size;
    int64_t num_blocks;
    int max_len, causal, num_splits;
    float scale;
    int64_t q_row_stride, out_row_stride, lse_row_stride, lse_head_stride;
    const void *v16_cache;   // null, or the fp16 V / 16 cache read instead of v_cache
};

// Host checks shared by the decode-kernel entries (strides already resolved).
attn_status decode_check(const DecodeCall &c) {
    if (!c.q || !c.k_cache || !c.v_cache || !c.out || !c.cache_seqlens || !c.block_table) return ATTN_ERR_INVALID_ARG;
    if (c.batch <= 0 || c.seqlen_q <= 0 || c.Hq <= 0 || c.Hkv <= 0 || c.Hq % c.Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (c.max_len < 0 || c.num_splits < 0 || c.bt_stride <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(c.scale > 0.f) || !isfinite(c.scale)) return ATTN_ERR_INVALID_ARG;
    if (!pow2(c.block_size) || c.block_size < 16 || c.num_blocks <= 0) return ATTN_ERR_INVALID_ARG;
    if (c.head_dim != 64 && c.head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if ((int64_t)c.seqlen_q * (c.Hq / c.Hkv) > kDecodeMaxColumns) return ATTN_ERR_UNSUPPORTED;
    if (c.batch > 65535 || c.Hkv > 65535) return ATTN_ERR_UNSUPPORTED;
    if (c.num_blocks * (int64_t)c.block_size >= (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    if ((int64_t)c.batch * c.seqlen_q * c.Hq >= (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(c.q) || !aligned16(c.k_cache) || !aligned16(c.v_cache) || !aligned16(c.out))
        return ATTN_ERR_INVALID_ARG;
    if (c.v16_cache && !aligned16(c.v16_cache)) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// Launch the split and combine kernels.  partials: at least
// decode_partial_bytes(...) bytes for the given plan, 16-byte aligned (unused
// with one split).
attn_status decode_launch(const DecodeCall &c, const DevInfo *d, int splits, int split_tok, float *partials,
                          void *stream) {
    DecodeParams p;
    memset(&p, 0, sizeof p);
    if (splits > 1) {
        p.o_part = partials;
        p.lse_part = partials + (size_t)c.batch * c.seqlen_q * c.Hq * splits * c.head_dim;
    }
    const int rpb = c.block_size < kDecodeTile ? c.block_size : kDecodeTile;
    const int64_t rows = c.num_blocks * (int64_t)c.block_size;
    const int64_t row_stride = (int64_t)c.Hkv * c.head_dim;
    CUtensorMap kmap, vmap;
    if (!make_map(&kmap, c.k_cache, rows, c.Hkv, c.head_dim, row_stride, 1, rpb) ||
        !make_map(&vmap, c.v16_cache ? c.v16_cache : c.v_cache, rows, c.Hkv, c.head_dim, row_stride, 1, rpb,
                  c.v16_cache ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return ATTN_ERR_LAUNCH_FAILED;
    p.v16 = c.v16_cache ? 1 : 0;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(c.q);
    p.out = reinterpret_cast<__nv_bfloat16 *>(c.out);
    p.lse = c.lse;
    p.cache_seqlens = c.cache_seqlens;
    p.block_table = c.block_table;
    p.q_row_stride = c.q_row_stride;
    p.out_row_stride = c.out_row_stride;
    p.lse_row_stride = c.lse_row_stride;
    p.lse_head_stride = c.lse_head_stride;
    p.bt_stride = c.bt_stride;
    p.block_size = c.block_size;
    p.rows_per_box = rpb;
    p.num_splits = splits;
    p.split_tokens = split_tok;
    p.num_blocks = c.num_blocks;
    p.Hq = c.Hq;
    p.Hkv = c.Hkv;
    p.G = c.Hq / c.Hkv;
    p.Sq = c.seqlen_q;
    {
        const int cols = c.seqlen_q * p.G;   // 16 columns per CTA (8 when one n8 tile covers them)
        p.ncg = cols <= 8 ? 1 : (cols + 15) / 16;
    }
    p.causal = c.causal ? 1 : 0;
    p.max_seqlen = c.max_len;
    p.scale_log2 = c.scale * 1.4426950408889634f;
    p.err = d->err;
    cudaError_t e = launch_decode(kmap, vmap, p, c.batch, c.head_dim, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return ATTN_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Failure-detection self-test (attn_selftest_bounded_wait).  One CTA, two
// warps.  Lane 0 of warp 0 waits on an mbarrier that nothing completes: its
// bounded wait gives up after the wait limit, records a timeout in the error
// word and raises the CTA's abort flag.  Lane 0 of warp 1 first idles for
// half that limit, then waits on another such mbarrier with the same abort
// flag: it must give up as soon as it sees the flag, before its own limit.
// Each records whether its wait succeeded and how long it waited.
// ---------------------------------------------------------------------------
namespace attn {
namespace {
constexpr uint32_t SRC_SELFTEST = 1u << 13;
static __device__ unsigned long long g_selftest_out[4];

__global__ void __launch_bounds__(64) attn_selftest_wait_kernel(uint32_t *err) {
    __shared__ uint64_t bars[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        if (w == 1) {   // idle for half the limit (bounded by the clock)
            const uint64_t t = globaltimer_ns();
            while (globaltimer_ns() - t < kWaitLimitNs / 2) {
            }
        }
        const uint64_t t0 = globaltimer_ns();
        // phase 0 of a fresh barrier never completes: nothing arrives on it
        const bool ok = mbar_wait(&bars[w], 0u, &abort_flag, err, SRC_SELFTEST);
        g_selftest_out[2 * w] = ok ? 1ull : 0ull;
        g_selftest_out[2 * w + 1] = globaltimer_ns() - t0;
    }
}
}  // namespace
}  // namespace attn

// measurement hook (see attn_set_kernel_events)
static thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;

namespace attn {
void main_kernel_event_before(cudaStream_t stream) {
    if (g_ev_before && g_ev_after) cudaEventRecord(g_ev_before, stream);
}

void main_kernel_event_after(cudaStream_t stream) {
    if (g_ev_before && g_ev_after) cudaEventRecord(g_ev_after, stream);
}
}  // namespace attn

extern "C" {

void attn_set_kernel_events(void *before, void *after) {
    g_ev_before = reinterpret_cast<cudaEvent_t>(before);
    g_ev_after = reinterpret_cast<cudaEvent_t>(after);
}

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

attn_status attn_selftest_bounded_wait(void *stream, unsigned long long *result) {
    if (!result) return ATTN_ERR_INVALID_ARG;
    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    attn_selftest_wait_kernel<<<1, 64, 0, s>>>(d->err);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyFromSymbol(result, g_selftest_out, sizeof(g_selftest_out)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return ATTN_OK;
}

const char *attn_status_string(attn_status s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case ATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case ATTN_ERR_LAUNCH_FAILED: return "CUDA launch or runtime call failed";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
        case ATTN_ERR_DEVICE_INDEX: return "a device-side index was out of range";
        case ATTN_ERR_NO_DEVICE: return "no usable CUDA device";
        case ATTN_ERR_DEVICE_RANGE: return "an input value was outside the range a kernel handles";
    }
    return "unknown status";
}

attn_status attn_get_last_device_error(void *stream, uint32_t *detail) {
    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, d->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    if (word) {
        const uint32_t zero = 0;
        if (cudaMemcpy(d->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_LAUNCH_FAILED;
        }
    }
    if (detail) *detail = word;
    if (word & ERR_INDEX) return ATTN_ERR_DEVICE_INDEX;
    if (word & ERR_TIMEOUT) return ATTN_ERR_DEVICE_TIMEOUT;
    if (word & ERR_RANGE) return ATTN_ERR_DEVICE_RANGE;
    return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Workspace: a 256-byte header (unit count), the fp16 copy of V (V / 16,
// [total_k, Hkv, D] by logical key), then the unit list (one int2 per
// (sequence, query pair, KV head)).
static const size_t kWsHeader = 256;

// derived cu_seqlens arrays at the head of a workspace (kv-cache and padded entries)
static size_t kvcache_cu_bytes(int batch) { return ((size_t)2 * (batch + 1) * sizeof(int32_t) + 255) & ~(size_t)255; }

static int64_t varlen_max_pairs(int num_heads_q, int num_heads_kv, int max_seqlen_q) {
    if (num_heads_kv <= 0 || num_heads_q <= 0 || num_heads_q % num_heads_kv || max_seqlen_q < 0) return -1;
    const int G = num_heads_q / num_heads_kv;
    if (G > kPrefillSlotRows) return -1;   // a slot holds at least one token's G heads
    const int64_t tps = kPrefillSlotRows / G;
    return ((int64_t)max_seqlen_q + 2 * tps - 1) / (2 * tps);
}

// Launches whose sequences all fit one query slot (max_seqlen_q <= 128 / G) at
// head_dim 128 run the one-slot instance, which converts bf16 V tiles to V' in
// shared memory when no V' cache is given.
static bool one_slot_cvt(int num_heads_q, int num_heads_kv, int head_dim, int max_seqlen_q) {
    const int G = num_heads_q / num_heads_kv;
    return head_dim == 128 && G >= 1 && G <= kPrefillSlotRows && max_seqlen_q <= kPrefillSlotRows / G;
}

static size_t v16_bytes(int num_heads_kv, int head_dim, int64_t total_k) {
    const size_t b = (size_t)total_k * (size_t)num_heads_kv * (size_t)head_dim * 2;
    return (b + 255) & ~(size_t)255;
}

size_t attn_varlen_workspace_size(int batch, int num_heads_q, int num_heads_kv, int head_dim, int max_seqlen_q,
                                  int64_t total_k) {
    const int64_t mp = varlen_max_pairs(num_heads_q, num_heads_kv, max_seqlen_q);
    if (batch <= 0 || mp < 0 || head_dim <= 0 || total_k < 0) return 0;
    // a one-slot launch at head_dim 128 converts V in the kernel: no V' copy
    if (one_slot_cvt(num_heads_q, num_heads_kv, head_dim, max_seqlen_q)) total_k = 0;
    return kWsHeader + v16_bytes(num_heads_kv, head_dim, total_k) +
           (size_t)batch * (size_t)mp * (size_t)num_heads_kv * sizeof(int2);
}

}  // extern "C"

// attn_varlen_fwd with optional per-sequence used lengths (a padded batch)
static attn_status varlen_impl(const void *q, const void *k, const void *v, void *out, float *lse,
                               const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, const int32_t *seqused_q,
                               const int32_t *seqused_k, int batch, int64_t total_q, int64_t total_k,
                               int max_seqlen_q, int max_seqlen_k, int num_heads_q, int num_heads_kv, int head_dim,
                               float softmax_scale, int causal, const int32_t *block_table, int block_table_stride,
                               int block_size, int64_t num_blocks, const void *v16_cache, int64_t q_row_stride,
                               int64_t k_row_stride, int64_t v_row_stride, int64_t out_row_stride, void *workspace,
                               size_t workspace_bytes, void *stream) {

    if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    if (batch <= 0 || num_heads_q <= 0 || num_heads_kv <= 0 || num_heads_q % num_heads_kv != 0)
        return ATTN_ERR_INVALID_ARG;
    if (total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    const int G = num_heads_q / num_heads_kv;
    if (G > kPrefillSlotRows) return ATTN_ERR_UNSUPPORTED;
    if (batch > 65535 || num_heads_kv > 65535) return ATTN_ERR_UNSUPPORTED;
    const bool paged = block_table != nullptr;
    if (paged) {
        if (!pow2(block_size) || block_size < 16 || num_blocks <= 0 || block_table_stride <= 0)
            return ATTN_ERR_INVALID_ARG;
        if (num_blocks * (int64_t)block_size >= (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    }
    if (total_k >= (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    if (total_q >= (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_INVALID_ARG;
    if (v16_cache && (!paged || !aligned16(v16_cache))) return ATTN_ERR_INVALID_ARG;   // a cache goes with a block table
    if (!fix_stride(&q_row_stride, (int64_t)num_heads_q * head_dim) ||
        !fix_stride(&out_row_stride, (int64_t)num_heads_q * head_dim) ||
        !fix_stride(&k_row_stride, (int64_t)num_heads_kv * head_dim) ||
        !fix_stride(&v_row_stride, (int64_t)num_heads_kv * head_dim))
        return ATTN_ERR_INVALID_ARG;
    if (paged && (k_row_stride != (int64_t)num_heads_kv * head_dim || v_row_stride != k_row_stride))
        return ATTN_ERR_INVALID_ARG;   // caches are packed [num_blocks, block_size, Hkv, D]

    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    if (total_q == 0 || max_seqlen_q == 0) return ATTN_OK;

    const int tps = kPrefillSlotRows / G;
    const int64_t max_pairs = varlen_max_pairs(num_heads_q, num_heads_kv, max_seqlen_q);
    if (max_pairs <= 0 || max_pairs > 0xFFFF || num_heads_kv > 0x7FFF ||
        (int64_t)batch * max_pairs * num_heads_kv > (int64_t)INT32_MAX / 4)
        return ATTN_ERR_UNSUPPORTED;
    // the one-slot instance (head_dim 128, every sequence within one slot) converts
    // bf16 V tiles to V' in shared memory itself: no conversion pass, no V' copy
    const bool v_cvt = !v16_cache && one_slot_cvt(num_heads_q, num_heads_kv, head_dim, max_seqlen_q);
    // with a paged V' cache, or converting in the kernel, the workspace holds no V'
    // copy (sized for total_k = 0)
    const int64_t ws_keys = (v16_cache || v_cvt) ? 0 : total_k;
    const size_t ws_need = attn_varlen_workspace_size(batch, num_heads_q, num_heads_kv, head_dim, max_seqlen_q, ws_keys);
    if (!workspace || workspace_bytes < ws_need) return ATTN_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    void *v16 = ws + kWsHeader;
    const int64_t kv_rows = paged ? num_blocks * (int64_t)block_size : total_k;
    const int kv_box = paged ? (block_size < kPrefillKeyTile ? block_size : kPrefillKeyTile) : kPrefillKeyTile;
    CUtensorMap qmap, kmap, vmap, omap;
    // output boxes: one warp's 32 rows of a slot (min(G, 32) heads x 32 / min(G, 32) tokens)
    const int obh = G < 32 ? G : 32;
    if (!make_map(&qmap, q, total_q, num_heads_q, head_dim, q_row_stride, G, tps) ||
        !make_map(&kmap, k, kv_rows, num_heads_kv, head_dim, k_row_stride, 1, kv_box) ||
        !make_map(&omap, out, total_q, num_heads_q, head_dim, out_row_stride, obh, 32 / obh))
        return ATTN_ERR_LAUNCH_FAILED;
    bool vmap_ok;
    if (v16_cache)
        vmap_ok = make_map(&vmap, v16_cache, kv_rows, num_heads_kv, head_dim, (int64_t)num_heads_kv * head_dim, 1,
                           kv_box, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    else if (v_cvt)
        vmap_ok = make_map(&vmap, v, kv_rows, num_heads_kv, head_dim, v_row_stride, 1, kv_box);
    else
        vmap_ok = make_map(&vmap, v16, total_k, num_heads_kv, head_dim, (int64_t)num_heads_kv * head_dim, 1,
                           kPrefillKeyTile, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    if (!vmap_ok) return ATTN_ERR_LAUNCH_FAILED;

    PrefillParams p;
    memset(&p, 0, sizeof p);
    p.v = reinterpret_cast<const __nv_bfloat16 *>(v);
    p.v16 = v16_cache ? nullptr : reinterpret_cast<__half *>(v16);
    p.v16_paged = v16_cache ? 1 : 0;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.seqused_q = seqused_q;
    p.seqused_k = seqused_k;
    p.block_table = block_table;
    p.total_q = total_q;
    p.total_k = total_k;
    p.out_row_stride = out_row_stride;
    p.v_row_stride = v_row_stride;
    p.head_dim = head_dim;
    p.max_seqlen_k = max_seqlen_k;
    p.v_row_stride = v_row_stride;
    p.num_blocks = num_blocks;
    p.bt_stride = block_table_stride;
    p.block_size = block_size;
    p.rows_per_box = kv_box;
    p.batch = batch;
    p.Hq = num_heads_q;
    p.Hkv = num_heads_kv;
    p.G = G;
    p.causal = causal ? 1 : 0;
    p.max_pairs = (int)max_pairs;
    p.one_slot = max_seqlen_q <= tps ? 1 : 0;
    p.v_cvt = v_cvt ? 1 : 0;
    // persistent CTAs: one per SM (fewer when there are fewer possible units)
    const int64_t max_units = (int64_t)batch * max_pairs * num_heads_kv;
    p.num_ctas = (int)(max_units < d->num_sms ? max_units : d->num_sms);
    p.unit_count = reinterpret_cast<int *>(ws);
    p.units = reinterpret_cast<int2 *>(ws + kWsHeader + v16_bytes(num_heads_kv, head_dim, ws_keys));
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.err = d->err;
    cudaError_t e = launch_prefill(qmap, kmap, vmap, omap, p, head_dim, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return ATTN_OK;
}

extern "C" {

attn_status attn_varlen_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int batch, int64_t total_q,
                            int64_t total_k, int max_seqlen_q, int max_seqlen_k, int num_heads_q, int num_heads_kv,
                            int head_dim, float softmax_scale, int causal, const int32_t *block_table,
                            int block_table_stride, int block_size, int64_t num_blocks, const void *v16_cache,
                            int64_t q_row_stride, int64_t k_row_stride, int64_t v_row_stride, int64_t out_row_stride,
                            void *workspace, size_t workspace_bytes, void *stream) {
    return varlen_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, nullptr, nullptr, batch, total_q, total_k,
                       max_seqlen_q, max_seqlen_k, num_heads_q, num_heads_kv, head_dim, softmax_scale, causal,
                       block_table, block_table_stride, block_size, num_blocks, v16_cache, q_row_stride, k_row_stride,
                       v_row_stride, out_row_stride, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Host-resident inputs: whole sequences in groups of about equal query-token
// counts (the last two groups 0.6 and 0.3 of the others, so that less work
// trails the last copy in); group i's copy in (copy_in_stream) overlaps the
// attention of group i-1 (stream) and the copy out of group i-2
// (copy_out_stream).  Each group is one attn_varlen_fwd call on the device
// buffers with cu_seqlens pointing into the full arrays, so rows are addressed
// in place and the result equals one call over the whole batch.
static int host_groups(const int32_t *cu_q, int batch, int num_groups, int *bounds) {
    const int64_t total = cu_q[batch];
    double w_all = 0.0;
    for (int g = 0; g < num_groups; ++g)
        w_all += (num_groups >= 3 && g == num_groups - 2) ? 0.6 : (num_groups >= 3 && g == num_groups - 1) ? 0.3 : 1.0;
    int n = 0, b0 = 0;
    double acc = 0.0;
    bounds[0] = 0;
    for (int g = 0; g < num_groups && b0 < batch; ++g) {
        acc += (num_groups >= 3 && g == num_groups - 2) ? 0.6 : (num_groups >= 3 && g == num_groups - 1) ? 0.3 : 1.0;
        const int64_t target = (int64_t)llround((double)total * acc / w_all);
        int b1 = b0;
        while (b1 < batch && (cu_q[b1 + 1] <= target || b1 == b0)) ++b1;
        if (b1 > b0) bounds[++n] = b1;
        b0 = b1;
    }
    if (b0 < batch) bounds[++n] = batch;
    return n;
}

extern "C" attn_status attn_varlen_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                                            void *out_host, const int32_t *cu_seqlens_q_host,
                                            const int32_t *cu_seqlens_k_host, int batch, int max_seqlen_q,
                                            int max_seqlen_k, int num_heads_q, int num_heads_kv, int head_dim,
                                            float softmax_scale, int causal, void *q_dev, void *k_dev, void *v_dev,
                                            void *out_dev, int32_t *cu_dev, void *workspace, size_t workspace_bytes,
                                            int num_groups, void *stream, void *copy_in_stream,
                                            void *copy_out_stream, void *event_a, void *event_b) {
    if (!q_host || !k_host || !v_host || !out_host || !cu_seqlens_q_host || !cu_seqlens_k_host) return ATTN_ERR_INVALID_ARG;
    if (!q_dev || !k_dev || !v_dev || !out_dev || !cu_dev || !event_a || !event_b) return ATTN_ERR_INVALID_ARG;
    if (batch <= 0 || num_groups <= 0 || num_groups > 64 || max_seqlen_q < 0 || max_seqlen_k < 0)
        return ATTN_ERR_INVALID_ARG;
    if (num_heads_q <= 0 || num_heads_kv <= 0 || head_dim <= 0) return ATTN_ERR_INVALID_ARG;
    // the host offsets are readable here: check them once
    if (cu_seqlens_q_host[0] != 0 || cu_seqlens_k_host[0] != 0) return ATTN_ERR_INVALID_ARG;
    for (int b = 0; b < batch; ++b) {
        const int64_t lq = (int64_t)cu_seqlens_q_host[b + 1] - cu_seqlens_q_host[b];
        const int64_t lk = (int64_t)cu_seqlens_k_host[b + 1] - cu_seqlens_k_host[b];
        if (lq < 0 || lk < 0 || lq > max_seqlen_q || lk > max_seqlen_k) return ATTN_ERR_INVALID_ARG;
    }
    const int64_t total_q = cu_seqlens_q_host[batch], total_k = cu_seqlens_k_host[batch];
    const size_t need = attn_varlen_workspace_size(batch, num_heads_q, num_heads_kv, head_dim, max_seqlen_q, total_k);
    if (need == 0) return head_dim != 64 && head_dim != 128 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE_TOO_SMALL;
    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;

    cudaStream_t s_main = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t s_in = reinterpret_cast<cudaStream_t>(copy_in_stream);
    cudaStream_t s_out = reinterpret_cast<cudaStream_t>(copy_out_stream);
    cudaEvent_t ev_a = reinterpret_cast<cudaEvent_t>(event_a), ev_b = reinterpret_cast<cudaEvent_t>(event_b);
    const size_t qrow = (size_t)num_heads_q * head_dim * 2, kvrow = (size_t)num_heads_kv * head_dim * 2;
    int bounds[65];
    const int ng = host_groups(cu_seqlens_q_host, batch, num_groups, bounds);
    bool fail = false;
    auto ck = [&](cudaError_t e) {
        if (e != cudaSuccess) fail = true;
    };
    // the copy streams start after the work already queued on `stream`
    ck(cudaEventRecord(ev_b, s_main));
    ck(cudaStreamWaitEvent(s_in, ev_b, 0));
    ck(cudaStreamWaitEvent(s_out, ev_b, 0));
    ck(cudaMemcpyAsync(cu_dev, cu_seqlens_q_host, (size_t)(batch + 1) * 4, cudaMemcpyHostToDevice, s_in));
    ck(cudaMemcpyAsync(cu_dev + batch + 1, cu_seqlens_k_host, (size_t)(batch + 1) * 4, cudaMemcpyHostToDevice, s_in));
    uint8_t *qd = reinterpret_cast<uint8_t *>(q_dev), *kd = reinterpret_cast<uint8_t *>(k_dev);
    uint8_t *vd = reinterpret_cast<uint8_t *>(v_dev), *od = reinterpret_cast<uint8_t *>(out_dev);
    const uint8_t *qh = reinterpret_cast<const uint8_t *>(q_host), *kh = reinterpret_cast<const uint8_t *>(k_host);
    const uint8_t *vh = reinterpret_cast<const uint8_t *>(v_host);
    uint8_t *oh = reinterpret_cast<uint8_t *>(out_host);
    for (int g = 0; g < ng && !fail && st == ATTN_OK; ++g) {
        const int b0 = bounds[g], b1 = bounds[g + 1];
        const int64_t q0 = cu_seqlens_q_host[b0], q1 = cu_seqlens_q_host[b1];
        const int64_t k0 = cu_seqlens_k_host[b0], k1 = cu_seqlens_k_host[b1];
        int mq = 0, mk = 0;
        for (int b = b0; b < b1; ++b) {
            const int lq = cu_seqlens_q_host[b + 1] - cu_seqlens_q_host[b];
            const int lk = cu_seqlens_k_host[b + 1] - cu_seqlens_k_host[b];
            mq = lq > mq ? lq : mq;
            mk = lk > mk ? lk : mk;
        }
        if (q1 > q0) ck(cudaMemcpyAsync(qd + q0 * qrow, qh + q0 * qrow, (q1 - q0) * qrow, cudaMemcpyHostToDevice, s_in));
        if (k1 > k0) {
            ck(cudaMemcpyAsync(kd + k0 * kvrow, kh + k0 * kvrow, (k1 - k0) * kvrow, cudaMemcpyHostToDevice, s_in));
            ck(cudaMemcpyAsync(vd + k0 * kvrow, vh + k0 * kvrow, (k1 - k0) * kvrow, cudaMemcpyHostToDevice, s_in));
        }
        ck(cudaEventRecord(ev_a, s_in));
        ck(cudaStreamWaitEvent(s_main, ev_a, 0));
        if (fail) break;
        st = varlen_impl(q_dev, k_dev, v_dev, out_dev, nullptr, cu_dev + b0, cu_dev + batch + 1 + b0, nullptr, nullptr,
                         b1 - b0, total_q, total_k, mq, mk, num_heads_q, num_heads_kv, head_dim, softmax_scale,
                         causal, nullptr, 0, 0, 0, nullptr, 0, 0, 0, 0, workspace, workspace_bytes, stream);
        ck(cudaEventRecord(ev_b, s_main));
        ck(cudaStreamWaitEvent(s_out, ev_b, 0));
        if (q1 > q0) ck(cudaMemcpyAsync(oh + q0 * qrow, od + q0 * qrow, (q1 - q0) * qrow, cudaMemcpyDeviceToHost, s_out));
    }
    // `stream` ends after the last copy out
    ck(cudaEventRecord(ev_a, s_out));
    ck(cudaStreamWaitEvent(s_main, ev_a, 0));
    if (fail) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return st;
}

// ---------------------------------------------------------------------------
// padded batch: [cu_seqlens_q | cu_seqlens_k] (256-byte aligned), then the
// varlen workspace for total_k = batch * seqlen_k.
size_t attn_padded_workspace_size(int batch, int seqlen_q, int seqlen_k, int num_heads_q, int num_heads_kv,
                                  int head_dim) {
    if (batch <= 0 || seqlen_q <= 0 || seqlen_k < 0) return 0;
    const size_t v = attn_varlen_workspace_size(batch, num_heads_q, num_heads_kv, head_dim, seqlen_q,
                                                (int64_t)batch * seqlen_k);
    return v ? kvcache_cu_bytes(batch) + v : 0;
}

attn_status attn_padded_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                            const int32_t *seqlens_q, const int32_t *seqlens_k, int batch, int seqlen_q,
                            int seqlen_k, int num_heads_q, int num_heads_kv, int head_dim, float softmax_scale,
                            int causal, void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
    if (batch <= 0 || seqlen_q <= 0 || seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
    if ((int64_t)batch * seqlen_q >= (int64_t)INT32_MAX || (int64_t)batch * seqlen_k >= (int64_t)INT32_MAX)
        return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_padded_workspace_size(batch, seqlen_q, seqlen_k, num_heads_q, num_heads_kv, head_dim);
    if (need == 0) return ATTN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    int32_t *cu_q = reinterpret_cast<int32_t *>(workspace);
    int32_t *cu_k = cu_q + (batch + 1);
    const size_t cu_b = kvcache_cu_bytes(batch);
    if (launch_padded_cu(batch, seqlen_q, seqlen_k, cu_q, cu_k, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return varlen_impl(q, k, v, out, lse, cu_q, cu_k, seqlens_q, seqlens_k, batch, (int64_t)batch * seqlen_q,
                       (int64_t)batch * seqlen_k, seqlen_q, seqlen_k, num_heads_q, num_heads_kv, head_dim,
                       softmax_scale, causal, nullptr, 0, 0, 0, nullptr, 0, 0, 0, 0,
                       reinterpret_cast<uint8_t *>(workspace) + cu_b, workspace_bytes - cu_b, stream);
}

// ---------------------------------------------------------------------------
// kv-cache entry: [cu_seqlens_q | cu_seqlens_k] (256-byte aligned), then the
// varlen workspace for total_k = batch * max_cache_seqlen.

// split cap of the kv-cache entry's decode route: longer splits when the Sq x G
// query columns of a KV head need several column-group CTAs (more than 16)
static int kvcache_split_cap(int seqlen_q, int num_heads_q, int num_heads_kv) {
    return (int64_t)seqlen_q * (num_heads_q / num_heads_kv) > 16 ? kSplitTokensGroups : kSplitTokens;
}

static size_t kvcache_ws(int batch, int seqlen_q, int num_heads_q, int num_heads_kv, int head_dim,
                         int max_cache_seqlen, bool v16_cache) {
    if (batch <= 0 || seqlen_q <= 0 || max_cache_seqlen < 0) return 0;
    if (kvcache_on_decode(batch, seqlen_q, num_heads_q, num_heads_kv, head_dim, v16_cache)) {
        // split partials of the decode kernel (never 0: 0 means invalid sizes)
        DevInfo *d = nullptr;
        int sms = 148;
        if (dev_info(&d) == ATTN_OK) sms = d->num_sms;
        int splits = 1, tok = 0;
        decode_plan(sms, batch, num_heads_kv, max_cache_seqlen, 0, &splits, &tok,
                    kvcache_split_cap(seqlen_q, num_heads_q, num_heads_kv));
        return decode_partial_bytes(batch, seqlen_q, num_heads_q, head_dim, splits) + 256;
    }
    const size_t v = attn_varlen_workspace_size(batch, num_heads_q, num_heads_kv, head_dim, seqlen_q,
                                                v16_cache ? 0 : (int64_t)batch * max_cache_seqlen);
    return v ? kvcache_cu_bytes(batch) + v : 0;
}

size_t attn_kvcache_workspace_size(int batch, int seqlen_q, int num_heads_q, int num_heads_kv, int head_dim,
                                   int max_cache_seqlen) {
    // enough for either route: with or without the fp16 V / 16 cache
    const size_t a = kvcache_ws(batch, seqlen_q, num_heads_q, num_heads_kv, head_dim, max_cache_seqlen, false);
    const size_t b = kvcache_ws(batch, seqlen_q, num_heads_q, num_heads_kv, head_dim, max_cache_seqlen, true);
    return a == 0 || b == 0 ? 0 : (a > b ? a : b);
}

attn_status attn_kvcache_fwd(const void *q, const void *k_cache, const void *v_cache, void *out, float *lse,
                             const int32_t *cache_seqlens, const int32_t *block_table, int block_table_stride,
                             int batch, int seqlen_q, int num_heads_q, int num_heads_kv, int head_dim,
                             int block_size, int64_t num_blocks, int max_cache_seqlen, float softmax_scale,
                             int causal, const void *v16_cache, void *workspace, size_t workspace_bytes,
                             void *stream) {
    if (!q || !k_cache || !v_cache || !out || !cache_seqlens || !block_table) return ATTN_ERR_INVALID_ARG;
    if (batch <= 0 || seqlen_q <= 0 || max_cache_seqlen < 0) return ATTN_ERR_INVALID_ARG;
    if ((int64_t)batch * max_cache_seqlen >= (int64_t)INT32_MAX || (int64_t)batch * seqlen_q >= (int64_t)INT32_MAX)
        return ATTN_ERR_UNSUPPORTED;
    // the decode route reads the bf16 V cache; the prefill route reads v16_cache when given
    const size_t need = kvcache_ws(batch, seqlen_q, num_heads_q, num_heads_kv, head_dim, max_cache_seqlen,
                                   v16_cache != nullptr);
    if (need == 0) return ATTN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    if (kvcache_on_decode(batch, seqlen_q, num_heads_q, num_heads_kv, head_dim, v16_cache != nullptr)) {
        // Sq x G query rows per KV head fit the decode kernel: stream the cache
        // once, no fp16 copy of V.  lse is [Hq, batch * seqlen_q].
        DecodeCall c = {q, k_cache, v_cache, out, lse, cache_seqlens, block_table, block_table_stride, batch,
                        seqlen_q, num_heads_q, num_heads_kv, head_dim, block_size, num_blocks, max_cache_seqlen,
                        causal, 0, softmax_scale, (int64_t)num_heads_q * head_dim, (int64_t)num_heads_q * head_dim,
                        1, (int64_t)batch * seqlen_q, v16_cache};
        if ((st = decode_check(c)) != ATTN_OK) return st;
        int splits = 1, split_tok = 0;
        decode_plan(d->num_sms, batch, num_heads_kv, max_cache_seqlen, 0, &splits, &split_tok,
                    kvcache_split_cap(seqlen_q, num_heads_q, num_heads_kv));
        return decode_launch(c, d, splits, split_tok, reinterpret_cast<float *>(workspace), stream);
    }
    int32_t *cu_q = reinterpret_cast<int32_t *>(workspace);
    int32_t *cu_k = cu_q + (batch + 1);
    const size_t cu_b = kvcache_cu_bytes(batch);
    if (launch_kvcache_cu(cache_seqlens, batch, seqlen_q, max_cache_seqlen, cu_q, cu_k, d->err,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return attn_varlen_fwd(q, k_cache, v_cache, out, lse, cu_q, cu_k, batch, (int64_t)batch * seqlen_q,
                           (int64_t)batch * max_cache_seqlen, seqlen_q, max_cache_seqlen, num_heads_q, num_heads_kv,
                           head_dim, softmax_scale, causal, block_table, block_table_stride, block_size, num_blocks,
                           v16_cache, 0, 0, 0, 0, reinterpret_cast<uint8_t *>(workspace) + cu_b,
                           workspace_bytes - cu_b, stream);
}

// ---------------------------------------------------------------------------
attn_status attn_softmax_rows(const void *x, void *y, int64_t rows, int cols, int64_t x_row_stride,
                              int64_t y_row_stride, int dtype, void *stream) {
    if (!x || !y || rows < 0 || cols < 0 || (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_BF16))
        return ATTN_ERR_INVALID_ARG;
    // any stride that covers a row (the kernels use 16-byte accesses only where rows allow it)
    if (x_row_stride == 0) x_row_stride = cols;
    if (y_row_stride == 0) y_row_stride = cols;
    if (x_row_stride < cols || y_row_stride < cols) return ATTN_ERR_INVALID_ARG;
    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    if (rows == 0 || cols == 0) return ATTN_OK;
    if (launch_softmax_rows(x, y, rows, cols, x_row_stride, y_row_stride, dtype == ATTN_DTYPE_BF16 ? 1 : 0,
                            d->num_sms, d->err, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return ATTN_OK;
}

// ---------------------------------------------------------------------------
int attn_decode_num_splits(int batch, int num_heads_kv, int max_cache_seqlen, int num_splits) {
    DevInfo *d = nullptr;
    int sms = 148;
    if (dev_info(&d) == ATTN_OK) sms = d->num_sms;
    return choose_splits(sms, batch, num_heads_kv, max_cache_seqlen, num_splits);
}

size_t attn_decode_workspace_size(int batch, int num_heads_q, int num_heads_kv, int head_dim, int max_cache_seqlen,
                                  int num_splits) {
    if (batch <= 0 || num_heads_q <= 0 || num_heads_kv <= 0 || head_dim <= 0) return 0;
    DevInfo *d = nullptr;
    int sms = 148;
    if (dev_info(&d) == ATTN_OK) sms = d->num_sms;
    int splits = 1, tok = 0;
    decode_plan(sms, batch, num_heads_kv, max_cache_seqlen, num_splits, &splits, &tok);
    if (splits <= 1) return 0;
    return decode_partial_bytes(batch, 1, num_heads_q, head_dim, splits) + 256;
}

attn_status attn_decode_paged(const void *q, const void *k_cache, const void *v_cache, void *out, float *lse,
                              const int32_t *cache_seqlens, const int32_t *block_table, int block_table_stride,
                              int batch, int num_heads_q, int num_heads_kv, int head_dim, int block_size,
                              int64_t num_blocks, int max_cache_seqlen, float softmax_scale, int num_splits,
                              int64_t q_row_stride, int64_t out_row_stride, void *workspace, size_t workspace_bytes,
                              void *stream) {
    DecodeCall c = {q, k_cache, v_cache, out, lse, cache_seqlens, block_table, block_table_stride, batch, 1,
                    num_heads_q, num_heads_kv, head_dim, block_size, num_blocks, max_cache_seqlen, 1, num_splits,
                    softmax_scale, q_row_stride, out_row_stride, num_heads_q, 1};
    attn_status st = decode_check(c);
    if (st != ATTN_OK) return st;
    if (!fix_stride(&c.q_row_stride, (int64_t)num_heads_q * head_dim) ||
        !fix_stride(&c.out_row_stride, (int64_t)num_heads_q * head_dim))
        return ATTN_ERR_INVALID_ARG;
    DevInfo *d = nullptr;
    if ((st = dev_info(&d)) != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    int splits = 1, split_tok = 0;
    decode_plan(d->num_sms, batch, num_heads_kv, max_cache_seqlen, num_splits, &splits, &split_tok);
    if (splits > 1) {
        if (!workspace || workspace_bytes < decode_partial_bytes(batch, 1, num_heads_q, head_dim, splits))
            return ATTN_ERR_WORKSPACE_TOO_SMALL;
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return ATTN_ERR_INVALID_ARG;
    }
    return decode_launch(c, d, splits, split_tok, reinterpret_cast<float *>(workspace), stream);
}

// ---------------------------------------------------------------------------
attn_status attn_decode_paged_noalloc(const void *q, const void *k_cache, const void *v_cache, void *out,
                                      float *lse, const int32_t *cache_seqlens, const int32_t *block_table,
                                      int block_table_stride, int batch, int num_heads_q, int num_heads_kv,
                                      int head_dim, int block_size, int64_t num_blocks, int max_cache_seqlen,
                                      float softmax_scale, int num_splits, int64_t q_row_stride,
                                      int64_t out_row_stride, void *stream) {
    DecodeCall c = {q, k_cache, v_cache, out, lse, cache_seqlens, block_table, block_table_stride, batch, 1,
                    num_heads_q, num_heads_kv, head_dim, block_size, num_blocks, max_cache_seqlen, 1, num_splits,
                    softmax_scale, q_row_stride, out_row_stride, num_heads_q, 1};
    attn_status st = decode_check(c);
    if (st != ATTN_OK) return st;
    if (!fix_stride(&c.q_row_stride, (int64_t)num_heads_q * head_dim) ||
        !fix_stride(&c.out_row_stride, (int64_t)num_heads_q * head_dim))
        return ATTN_ERR_INVALID_ARG;
    DevInfo *d = nullptr;
    if ((st = dev_info(&d)) != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    float *scratch = nullptr;
    size_t scratch_bytes = 0;
    if (decode_noalloc_scratch(&scratch, &scratch_bytes) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    int splits = 1, split_tok = 0;
    decode_plan(d->num_sms, batch, num_heads_kv, max_cache_seqlen, num_splits, &splits, &split_tok);
    if (decode_partial_bytes(batch, 1, num_heads_q, head_dim, splits) > scratch_bytes) {
        if (num_splits > 0) return ATTN_ERR_WORKSPACE_TOO_SMALL;   // the asked split count does not fit
        // library's choice: the largest split count whose partials fit (1 needs none)
        const size_t per_split = (size_t)batch * num_heads_q * (head_dim + 1) * sizeof(float);
        int fit = (int)(scratch_bytes / per_split);
        if (fit < 2) fit = 1;
        split_tok = split_tokens_for(max_cache_seqlen, fit);
        splits = (max_cache_seqlen + split_tok - 1) / split_tok;
    }
    return decode_launch(c, d, splits, split_tok, scratch, stream);
}

// ---------------------------------------------------------------------------
attn_status store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache, void *v16_cache,
                          const int64_t *slot_mapping, int64_t num_tokens, int num_heads_kv, int head_dim,
                          int64_t k_row_stride, int64_t v_row_stride, int64_t num_slots, void *stream) {
    if (num_tokens < 0 || num_heads_kv <= 0 || head_dim <= 0 || num_slots < 0) return ATTN_ERR_INVALID_ARG;
    if (num_tokens == 0) return ATTN_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return ATTN_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_heads_kv * head_dim;
    if (k_row_stride == 0) k_row_stride = row;
    if (v_row_stride == 0) v_row_stride = row;
    if (k_row_stride < row || v_row_stride < row) return ATTN_ERR_INVALID_ARG;
    if (row > (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    DevInfo *d = nullptr;
    attn_status st = dev_info(&d);
    if (st != ATTN_OK) return st;
    if ((st = check_arch(d)) != ATTN_OK) return st;
    cudaError_t e = launch_store_kvcache(k, v, k_cache, v_cache, v16_cache, slot_mapping, num_tokens, (int)row,
                                         k_row_stride,
                                         v_row_stride, num_slots, d->num_sms, d->err,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH_FAILED;
    }
    return ATTN_OK;
}

}  // extern "C"
