// prefill.cu -- varlen (optionally paged) causal prefill on the sm_103a tensor
// cores: tcgen05.mma with TMEM accumulators fed by TMA, warp-specialised.
//
// Method ("从零实现 vLLM (1.3)：如何加速 Attention 计算"):
//   * "FlashAttention 的最终实现" / "计算流程（1-Pass 算法与分块）": one pass
//     over the key tiles keeping per query row the running max m, the proxy
//     denominator d' and the proxy output o'; when m grows, o' and d' are
//     rescaled by e^(m_old - m_new).  Logits and probabilities never leave the
//     chip.  Normalisation by d' is deferred to the epilogue (equal in exact
//     arithmetic to normalising at every step).
//   * "Prefill": varlen packing by cu_seqlens_q / cu_seqlens_k; with a block
//     table, K/V are read from the paged cache (prefix cache).
//   * causal masking is bottom-right aligned: query i of a sequence with Lq
//     queries and Lk keys sees keys j <= Lk - Lq + i.
//
// Work unit (taken from the scheduler's list; persistent CTAs, one per SM,
// take the next entry from a global counter when they start a unit): a
// sequence b, a KV head, and two query "slots" A and B
// of 128 rows each.  A slot packs floor(128 / G) consecutive tokens x the G query
// heads that share the KV head (row r = token_offset * G + g), so one K/V stream
// feeds 256 query rows (for a G that does not divide 128 a slot's last
// 128 - floor(128 / G) G rows are idle).  Slot B holds the tokens after slot A's.
//
// Roles (352 threads):
//   warps 0-3  softmax for slot A, one thread per row (TMEM lanes 0-127)
//   warps 4-7  softmax for slot B
//   warp 8     TMA producer: Q_A, Q_B once, then K_j, V_j tiles through a
//              3-stage ring (4 for head_dim 64) of 128 keys x head_dim,
//              128-byte swizzle, in the order K_0, K_1, V_0, K_2, V_1, ...
//   warp 9     TMEM allocator and the thread that issues every QK^T
//   warp 10    the thread that issues every PV
// TMEM (512 columns): S_A [0,128), S_B [128,256) fp32; O_A, O_B after them.
// When every sequence fits one slot (at most 128 / G tokens: a few new tokens
// per sequence against a cached context) slot B never has rows; the HALF
// instance then gives warps 4-7 the keys [64, 128) of slot A's tiles, so each
// softmax thread works on half a tile, and uses the freed Q_B / P'_B memory for
// a fourth and a fifth ring stage.
//
// PV runs in fp16: the softmax threads write P' = 16 P as fp16 into shared
// memory (one 128 x 128 tile per slot, K-major, 128-byte swizzle), and V comes
// as V' = fp16(V / 16): from a copy made by attn_prefill_prep_kernel before the
// attention kernel (laid out contiguously by sequence, also for a paged cache),
// from the paged fp16 V / 16 cache that store_kvcache keeps, or, in the one-slot
// instance without that cache, from bf16 V tiles that its softmax threads
// convert in shared memory.  The product P' V' equals P V, and the weights keep 11 significant
// bits: with bf16 weights (8 bits) the weight rounding adds about as much error
// as the bf16 output rounding and the result exceeds a 2e-3 relative RMS error.
// One MMA takes A and B of the same type, hence the fp16 copy of V.
//
// Because P' does not live in S's columns, S_X(t+1) can be computed as soon as
// the softmax threads of slot X have read S_X(t) into registers (s_free), while
// they still work on it: the QK^T of the next key tile overlaps the softmax of
// the current one, and the two slots need no fixed phase.  PV_X(t) starts when
// P'_X(t) is in shared memory (p_ready); the softmax of tile t+1 computes its
// exponentials first and waits for PV_X(t) to finish (pv_done) only before it
// overwrites P'_X or rescales O_X.  The two issuing threads feed the tensor
// core independently; each orders its own work (tcgen05 operations of one
// thread complete in order) and reports through tcgen05.commit.
//
// Persistence: barriers and TMEM are set up once per CTA and the barrier
// phases run on across units.  The producer warp takes unit indices
// (atomicAdd) and hands them to the other roles through a two-entry ring in
// shared memory.  The producer loads the next unit's Q as soon as the current
// unit's last QK^T has read Q (q_empty), and K/V tiles of the next unit as ring
// slots free up, so the tensor core starts the next unit while the softmax
// warps finish the current one.  A unit's output rows are written by the
// softmax threads during the first tile of their next unit, once the last PV
// of the unit is done and before P'_X(0) of the next one is published, so the
// wait for that PV overlaps the next tile's exponentials.
//
// The rescale is lazy: the reference max of a row moves only when the tile
// max exceeds it by more than 8 (log2 units), so P stays <= 256 and O is
// rarely touched; the final O / d' uses the same reference, so the result is
// unchanged.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace attn {

constexpr int kPfThreads = 352;
constexpr int BM = kPrefillSlotRows;   // 128 rows per slot
constexpr int BN = kPrefillKeyTile;    // 128 keys per tile
constexpr int kPBytes = BM * BN * 2;   // one slot's P' tile (fp16)
constexpr int kPPanelBytes = BM * 128; // 64 keys of P' per 128-byte-swizzled panel

// HALF (one query slot per unit): no Q_B and no P'_B; a fourth and a fifth ring
// stage and the two softmax halves' exchange area instead (the fifth fits because
// the dynamic shared memory is declared 1024-byte aligned, so no slack is kept)
template <int D, bool HALF = false>
struct PfSmem {
    static constexpr int kStages = HALF ? 5 : (D == 128 ? 3 : 4);   // K / V' ring stages
    static constexpr int kPanels = D / 64;
    static constexpr int kPanelBytes = 128 * 128;            // 128 rows x 128 B
    static constexpr int kTileBytes = kPanels * kPanelBytes; // one Q slot, K tile or V tile
    static constexpr int kRingOff = (HALF ? 1 : 2) * kTileBytes;
    static constexpr int kPOff = kRingOff + kStages * kTileBytes;
    static constexpr int kXchOff = kPOff + (HALF ? 1 : 2) * kPBytes;   // [parity][half][row] floats
    static constexpr int kBarOff = kXchOff + (HALF ? 2 * 2 * BM * 4 : 0);
    static constexpr int kNumBars = 3 * kStages + 24;
    static constexpr int kBytes = kBarOff + kNumBars * 8 + 16 + (HALF ? 0 : 1024) /*align slack*/;
    static_assert(kBytes <= 227 * 1024, "shared memory");
};

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_base, uint32_t k_base) {
    using S = PfSmem<D>;
    constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks / 4) * S::kPanelBytes + (ks % 4) * 32;
        tc_mma_ss(d_tmem, sw128_desc(q_base + off, 16, 1024), sw128_desc(k_base + off, 16, 1024), idesc, ks > 0);
    }
}

// O (+)= P' V': fp16 operands from shared memory, P' K-major (keys along the
// 128-byte rows), V' MN-major
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_base, uint32_t v_base, bool accumulate) {
    using S = PfSmem<D>;
    constexpr uint32_t idesc = idesc_f16_f32(BM, D, 1);
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t pd = sw128_desc(p_base + (kk / 4) * kPPanelBytes + (kk % 4) * 32, 16, 1024);
        const uint64_t vd = sw128_desc(v_base + kk * 16 * 128, S::kPanelBytes, 1024);
        tc_mma_ss(d_tmem, pd, vd, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// ---------------------------------------------------------------------------
// Rows of sequence b: queries [qs, qs + Lq), keys [ks, ks + Lk) of the packed
// tensors.  The range is cu_seqlens[b] .. cu_seqlens[b+1]; with seqused_q/k only
// its first seqused[b] rows are the sequence (a padded batch).  False, and the
// error word set when `report`, if the offsets are invalid; a used length
// outside [0, range] is clamped (and reported).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool seq_rows(const PrefillParams &p, int b, bool report, int &qs, int &Lq, int &ks,
                                         int &Lk) {
    qs = __ldg(p.cu_q + b);
    ks = __ldg(p.cu_k + b);
    const int qe = __ldg(p.cu_q + b + 1), ke = __ldg(p.cu_k + b + 1);
    if (qs < 0 || qe < qs || ks < 0 || ke < ks || (int64_t)qe > p.total_q || (int64_t)ke > p.total_k) {
        if (report) record_error(p.err, ERR_INDEX | SRC_PREFILL);
        return false;
    }
    Lq = qe - qs;
    Lk = ke - ks;
    if (p.seqused_q) {
        const int u = __ldg(p.seqused_q + b);
        if ((u < 0 || u > Lq) && report) record_error(p.err, ERR_INDEX | SRC_PREFILL);
        Lq = min(max(u, 0), Lq);
    }
    if (p.seqused_k) {
        const int u = __ldg(p.seqused_k + b);
        if ((u < 0 || u > Lk) && report) record_error(p.err, ERR_INDEX | SRC_PREFILL);
        Lk = min(max(u, 0), Lk);
    }
    return true;
}

// ---------------------------------------------------------------------------
// V -> V' = fp16(V / 16), laid out [total_k, Hkv, D] by logical key
// (cu_seqlens_k[b] + j), read contiguously or through the block table.
// One CTA per (32 keys, sequence).  |v| >= 2^20 (or non-finite) does not fit
// and is clamped and reported.  Up to 128 rows after each sequence's keys are
// zeroed (within its range; the last range runs to total_k): its last key tile
// reads them with zero weights, and they may hold padding or, with a paged
// cache (total_k an upper bound), stale workspace contents that could be NaN.
// Rows of a key whose block id is out of range are zeroed too.
// ---------------------------------------------------------------------------
constexpr int kCvtThreads = 256;
constexpr int kCvtKeys = 32;
constexpr int kEarlyMaxKeys = 4096;   // longest key range for which the next unit is taken a unit ahead
constexpr int kCvtUnroll = 8;   // 16-byte chunks each thread keeps in flight

__device__ __forceinline__ void v_to_f16_keys(const PrefillParams &p) {
    const int b = blockIdx.y - 1;   // row 0 of the grid is the scheduler's
    int qs, Lq, k0, Lk;
    if (!seq_rows(p, b, false, qs, Lq, k0, Lk)) return;   // reported by the scheduler
    const int key0 = blockIdx.x * kCvtKeys;
    const int row_chunks = p.Hkv * p.head_dim / 8;   // 16-byte chunks per key row
    if (blockIdx.x == 0) {
        // rows after the sequence's keys up to one key tile, inside its range
        // (the last sequence's range runs to total_k)
        const int64_t t0 = (int64_t)k0 + Lk;
        const int64_t lim = b == p.batch - 1 ? p.total_k : (int64_t)__ldg(p.cu_k + b + 1);
        const int64_t t1 = min(t0 + (int64_t)kPrefillKeyTile, lim);
        for (int64_t i = t0 * row_chunks + threadIdx.x; i < t1 * row_chunks; i += kCvtThreads)
            reinterpret_cast<uint4 *>(p.v16)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0 && key0 + kCvtKeys < Lk)
        record_error(p.err, ERR_INDEX | SRC_PREFILL);   // longer than the stated max_seqlen_k
    if (Lk <= 0 || key0 >= Lk) return;
    const int nkeys = min(kCvtKeys, Lk - key0);
    const int32_t *bt = p.block_table ? p.block_table + (int64_t)b * p.bt_stride : nullptr;
    uint32_t big = 0;
    // kCvtUnroll chunks per thread in flight: all loads of a batch before its stores
    const int total = nkeys * row_chunks;
    for (int base = threadIdx.x; base < total; base += kCvtThreads * kCvtUnroll) {
        uint4 v[kCvtUnroll];
        int64_t dst[kCvtUnroll];   // chunk of V' (-1: none)
#pragma unroll
        for (int u = 0; u < kCvtUnroll; ++u) {
            const int idx = base + u * kCvtThreads;
            dst[u] = -1;
            if (idx >= total) continue;
            const int kk = idx / row_chunks, ch = idx % row_chunks;
            const int key = key0 + kk;
            dst[u] = ((int64_t)k0 + key) * row_chunks + ch;
            int64_t src_row;
            if (bt) {
                const int blk = __ldg(bt + key / p.block_size);
                if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                    record_error(p.err, ERR_INDEX | SRC_PREFILL);
                    v[u] = make_uint4(0u, 0u, 0u, 0u);   // zeroed row
                    continue;
                }
                src_row = (int64_t)blk * p.block_size + key % p.block_size;
            } else {
                src_row = (int64_t)k0 + key;
            }
            v[u] = ldg_stream16(p.v + src_row * p.v_row_stride + ch * 8);
        }
#pragma unroll
        for (int u = 0; u < kCvtUnroll; ++u) {
            if (dst[u] < 0) continue;
            uint4 w = v[u];
            big = __vmaxu2(big, __vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu));
            big = __vmaxu2(big, __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
            w.x = bf16x2_to_f16x2_div16(w.x);
            w.y = bf16x2_to_f16x2_div16(w.y);
            w.z = bf16x2_to_f16x2_div16(w.z);
            w.w = bf16x2_to_f16x2_div16(w.w);
            reinterpret_cast<uint4 *>(p.v16)[dst[u]] = w;
        }
    }
    if (__any_sync(0xffffffffu, (big & 0xFFFFu) >= 0x4980u || (big >> 16) >= 0x4980u) && (threadIdx.x & 31) == 0)
        record_error(p.err, ERR_RANGE | SRC_PREFILL);
}

// ---------------------------------------------------------------------------
// Scheduler (one CTA of the pre-pass launch): writes the unit list that the
// persistent attention CTAs take entries from, in order, through a global
// counter.  Sequences come longest first (counting sort on the key tiles of
// their longest unit, the one of the last query pair: with a cached context
// that is not proportional to the number of query pairs), so the last units
// taken are short; inside a sequence units are grouped by KV head and run from
// the last query pair (most key tiles) to the first, so units running together
// share one K/V stream in L2.
// Entry = (sequence, pair | kv_head << 16).  Also flags invalid offsets and
// sequences longer than max_seqlen_q.
// ---------------------------------------------------------------------------
constexpr int kSchedThreads = kCvtThreads;   // the scheduler is one CTA of the pre-pass kernel
constexpr int kSchedBuckets = 4096;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kSchedWarpBatch = 1024;   // up to this many sequences, a warp writes each one's units

__device__ __forceinline__ int pf_pairs(const PrefillParams &p, int b, bool report, int &bucket) {
    const int tps = BM / p.G;
    int qs, Lq, ks, Lk;
    bucket = 0;
    if (!seq_rows(p, b, report, qs, Lq, ks, Lk)) return 0;
    // sort key: the key tiles of the sequence's longest unit (its last query pair)
    bucket = min((Lk + BN - 1) / BN, kSchedBuckets - 1);
    int pairs = (Lq + 2 * tps - 1) / (2 * tps);
    if (pairs > p.max_pairs) {   // longer than the stated max_seqlen_q
        if (report) record_error(p.err, ERR_INDEX | SRC_PREFILL);
        pairs = p.max_pairs;
    }
    return pairs;
}

__device__ __forceinline__ void schedule_units(const PrefillParams &p) {
    __shared__ int units_in[kSchedBuckets];   // units per pair-count bucket, then running offsets
    __shared__ int wsum[kSchedWarps];
    for (int i = threadIdx.x; i < kSchedBuckets; i += kSchedThreads) units_in[i] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < p.batch; b += kSchedThreads) {
        int bucket;
        const int pairs = pf_pairs(p, b, true, bucket);
        if (pairs) atomicAdd(&units_in[bucket], pairs * p.Hkv);
    }
    __syncthreads();
    // descending exclusive scan: offset of a bucket = units of all larger buckets
    constexpr int PER = kSchedBuckets / kSchedThreads;
    int local[PER], sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        local[i] = units_in[kSchedBuckets - 1 - (threadIdx.x * PER + i)];
        sum += local[i];
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int w = lane < kSchedWarps ? wsum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < kSchedWarps) wsum[lane] = wi - w;   // exclusive
    }
    __syncthreads();
    int run = wsum[wid] + incl - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        units_in[kSchedBuckets - 1 - (threadIdx.x * PER + i)] = run;
        run += local[i];
    }
    if (threadIdx.x == kSchedThreads - 1) {
        p.unit_count[0] = run;
        p.unit_count[1] = 0;   // the attention kernel's next-unit counter
    }
    __syncthreads();
    if (p.batch <= kSchedWarpBatch) {
        // few sequences (each with many units): a warp writes each sequence's entries
        for (int b = wid; b < p.batch; b += kSchedWarps) {
            int bucket;
            const int pairs = pf_pairs(p, b, false, bucket);
            if (!pairs) continue;
            int off = 0;
            if (lane == 0) off = atomicAdd(&units_in[bucket], pairs * p.Hkv);
            off = __shfl_sync(0xffffffffu, off, 0);
            for (int e = lane; e < pairs * p.Hkv; e += 32) {
                const int h = e / pairs, i = e % pairs;
                p.units[off + e] = make_int2(b, (pairs - 1 - i) | (h << 16));
            }
        }
    } else {
        for (int b = threadIdx.x; b < p.batch; b += kSchedThreads) {
            int bucket;
            const int pairs = pf_pairs(p, b, false, bucket);
            if (!pairs) continue;
            int off = atomicAdd(&units_in[bucket], pairs * p.Hkv);
            for (int h = 0; h < p.Hkv; ++h)
                for (int i = 0; i < pairs; ++i) p.units[off++] = make_int2(b, (pairs - 1 - i) | (h << 16));
        }
    }
}

// ---------------------------------------------------------------------------
// Pre-pass before the attention kernel, one launch: CTA (0, 0) writes the unit
// list (schedule_units); CTAs (x, b + 1) convert V of sequence b to V'
// (v_to_f16_keys).  With a paged V' cache (v16_paged), or when the one-slot
// instance converts V tiles itself (v_cvt), the launch is the scheduler's CTA alone.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kCvtThreads) attn_prefill_prep_kernel(const PrefillParams p) {
    // the attention kernel may be scheduled now (it waits for this grid before
    // reading anything it writes)
    asm volatile("griddepcontrol.launch_dependents;");
    if (p.v16_paged || p.v_cvt || blockIdx.y == 0) {
        // the scheduler (grid row 0, dispatched first); with a paged V' cache, or when
        // the attention kernel converts V itself, the launch is this one CTA
        if (blockIdx.x == 0) schedule_units(p);
        return;
    }
    v_to_f16_keys(p);
}

// Work of one unit: rows [t0A, t0A + tps) and [t0B, t0B + tps) of sequence b
// (tps = 128 / G tokens), nA / nB key tiles.  An invalid unit (bad offsets,
// reported by the scheduler) has no rows and no tiles.
struct PfUnit {
    int b, hkv, qs, Lq, ks0, Lk, off, t0A, t0B, nA, nB, n;
};

__device__ __forceinline__ PfUnit pf_unit(const PrefillParams &p, int u) {
    PfUnit w;
    const int2 e = p.units[u];
    w.b = e.x;
    w.hkv = e.y >> 16;
    const int pair = e.y & 0xFFFF, tps = BM / p.G;
    if (!seq_rows(p, w.b, false, w.qs, w.Lq, w.ks0, w.Lk) || pair * 2 * tps >= w.Lq) {
        w.qs = w.ks0 = w.Lk = w.off = w.nA = w.nB = w.n = 0;
        w.Lq = 0;
        w.t0A = w.t0B = 0;
        return w;
    }
    w.off = w.Lk - w.Lq;
    w.t0A = pair * 2 * tps;
    w.t0B = w.t0A + tps;
    auto tiles_for = [&](int t0) -> int {
        if (t0 >= w.Lq) return 0;
        const int t1 = min(t0 + tps, w.Lq);
        const int kend = p.causal ? min(max(t1 + w.off, 0), w.Lk) : w.Lk;
        return (kend + BN - 1) / BN;
    };
    w.nA = tiles_for(w.t0A);
    w.nB = tiles_for(w.t0B);
    w.n = max(w.nA, w.nB);
    return w;
}

// HALF: slot B is never used (a sequence longer than one slot, already reported
// against max_seqlen_q, keeps only slot A's rows)
template <bool HALF>
__device__ __forceinline__ PfUnit pf_unit_k(const PrefillParams &p, int u) {
    PfUnit w = pf_unit(p, u);
    if (HALF) {
        w.nB = 0;
        w.n = w.nA;
    }
    return w;
}

// Output rows of one slot, 32 rows per warp (warp-collective; every argument
// but l and m_ref is warp-uniform): O_X / d' -> bf16, read from TMEM when the
// slot had key tiles (zeros otherwise), and the lse.  The rows are staged in
// this warp's own rows of the slot's P' tile (free: the slot's last PV has
// completed) in the 128-byte-swizzled layout of an output box (64 dims x
// min(G, 32) heads x 32 / min(G, 32) tokens per panel), and one thread writes
// them with a TMA store per panel.  Panel by panel: a panel's two TMEM loads
// before one wait, its conversion, its staging and its store, so the first
// panel's store reads shared memory while the second is converted (all four
// loads at once need 128 registers here and spill).  A warp holding rows past the sequence's
// end (its last slot) writes its valid rows itself instead: a box would
// overwrite the next sequence's rows.  Out of line: it runs once per unit, and
// its registers then do not constrain the softmax's per-tile code.
template <int D, bool OBOX>
__device__ __noinline__ void pf_store_rows(const PrefillParams &p, const CUtensorMap *omap, uint32_t tO,
                                              uint8_t *pslot, bool has_tiles, int64_t qbase, int ntok, int hkv,
                                              float l, float m_ref) {
    const int G = p.G, lane = threadIdx.x & 31, wrow0 = ((threadIdx.x >> 5) & 3) * 32;
    if (wrow0 / G >= ntok) return;   // no valid row in this warp
    const int r = wrow0 + lane;
    const bool row_valid = r / G < ntok, whole = OBOX && (wrow0 + 31) / G < ntok;
    const float inv = l > 0.f ? 16.f / l : 0.f;   // l accumulated P' = 16 P
    uint8_t *srow = pslot + r * 128;
    __nv_bfloat16 *orow = p.out + (qbase + r / G) * p.out_row_stride + (int64_t)(hkv * G + r % G) * D;
    if (row_valid && p.lse)
        p.lse[(int64_t)(hkv * G + r % G) * p.total_q + qbase + r / G] =
            l > 0.f ? (m_ref + __log2f(l) - 4.0f) * 0.69314718055994531f : -INFINITY;
#pragma unroll 1
    for (int pn = 0; pn < D / 64; ++pn) {
        uint32_t o[2][32];
        if (has_tiles) {
            tmem_ld32(tO + (uint32_t)(pn * 64), o[0]);
            tmem_ld32(tO + (uint32_t)(pn * 64 + 32), o[1]);
            tc_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[0][i] = o[1][i] = 0u;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2(__uint_as_float(o[cc][2 * i]) * inv, __uint_as_float(o[cc][2 * i + 1]) * inv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v4 = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                const int ch = (2 * pn + cc) * 4 + i;   // 16-byte chunk of the row
                if (whole)
                    *reinterpret_cast<uint4 *>(srow + (ch >> 3) * kPPanelBytes + (((ch & 7) ^ (r & 7)) << 4)) = v4;
                else if (row_valid)
                    reinterpret_cast<uint4 *>(orow)[ch] = v4;
            }
        }
        if (whole) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                tma_store_3d(omap, pslot + pn * kPPanelBytes + wrow0 * 128, pn * 64, hkv * G + wrow0 % G,
                             (int)(qbase + wrow0 / G));
        }
    }
    if (whole) {
        if (lane == 0) {
            bulk_commit();
            bulk_wait_read();   // the staging rows are P' rows again right after
        }
        __syncwarp();
    }
}

// pf_store_rows for one half of the head dimension (HALF kernel): the warp's 32
// rows, dims [64 h, 64 h + 64) from O's columns of that half, staged in panel h
// of the slot's P' rows and written by one TMA store; half 0 writes the lse.
template <int D, bool OBOX>
__device__ __noinline__ void pf_store_rows_half(const PrefillParams &p, const CUtensorMap *omap, uint32_t tO,
                                                uint8_t *pslot, bool has_tiles, int64_t qbase, int ntok, int hkv,
                                                float l, float m_ref, int h) {
    const int G = p.G, lane = threadIdx.x & 31, wrow0 = ((threadIdx.x >> 5) & 3) * 32;
    if (wrow0 / G >= ntok) return;   // no valid row in this warp
    const int r = wrow0 + lane;
    const bool row_valid = r / G < ntok, whole = OBOX && (wrow0 + 31) / G < ntok;
    const float inv = l > 0.f ? 16.f / l : 0.f;   // l accumulated P' = 16 P
    uint8_t *srow = pslot + r * 128;
    __nv_bfloat16 *orow = p.out + (qbase + r / G) * p.out_row_stride + (int64_t)(hkv * G + r % G) * D;
#pragma unroll
    for (int c = 2 * h; c < 2 * h + 2; ++c) {
        uint32_t o[32];
        if (has_tiles) {
            tmem_ld32(tO + (uint32_t)(c * 32), o);
            tc_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v4 = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            const int ch = c * 4 + i;   // 16-byte chunk of the row
            if (whole)
                *reinterpret_cast<uint4 *>(srow + (ch >> 3) * kPPanelBytes + (((ch & 7) ^ (r & 7)) << 4)) = v4;
            else if (row_valid)
                reinterpret_cast<uint4 *>(orow)[ch] = v4;
        }
    }
    if (h == 0 && row_valid && p.lse)
        p.lse[(int64_t)(hkv * G + r % G) * p.total_q + qbase + r / G] =
            l > 0.f ? (m_ref + __log2f(l) - 4.0f) * 0.69314718055994531f : -INFINITY;
    if (whole) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(omap, pslot + h * kPPanelBytes + wrow0 * 128, h * 64, hkv * G + wrow0 % G,
                         (int)(qbase + wrow0 / G));
            bulk_commit();
            bulk_wait_read();   // the staging rows are P' rows again right after
        }
        __syncwarp();
    }
}

// One bf16 pair -> fp16(v / 16) pair: the scaling is exact in bf16 (a power of
// two), then each half widens to fp32 exactly and the pair rounds to fp16 (RNE,
// values past the fp16 range clamped).  The same values as scaling in fp32.
__device__ __forceinline__ uint32_t bf16x2_div16_to_f16x2(uint32_t w) {
    uint32_t q, r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(w), "r"(0x3D803D80u));   // x 0.0625
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r)
        : "f"(__uint_as_float(q & 0xFFFF0000u)), "f"(__uint_as_float(q << 16)));
    return r;
}

// Bit 15 / 31 set where that bf16 half has |v| >= 2^20 or is not finite: its
// magnitude bits plus 0x8000 - 0x4980 reach bit 15 (no carry crosses halves).
__device__ __forceinline__ uint32_t bf16x2_past_2p20(uint32_t w) {
    return ((w & 0x7FFF7FFFu) + 0x36803680u) & 0x80008000u;
}

// One-slot instance without a V' cache: the 256 softmax threads convert a bf16 V
// tile in its ring stage to V' = fp16(V / 16) in place (the 128-byte swizzle only
// permutes 16-byte chunks within a key row, so every chunk keeps its row and
// its element order).  Rows at or past `valid` (keys past the sequence's end)
// are zeroed; |v| >= 2^20 or non-finite is clamped and reported, as in the
// conversion pass.  The caller's proxy fence and p_ready arrival publish it.
template <int D>
__device__ __forceinline__ void v_tile_to_f16(uint8_t *tile, int valid, uint32_t *err, int ci, int cs) {
    constexpr int kChunks = (D / 64) * BN * 8;   // 16-byte chunks in the tile
    const bool whole = valid >= BN;
    uint32_t bad = 0;
    for (int c0 = ci; c0 < kChunks; c0 += 4 * cs) {
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (c0 + i * cs < kChunks) v[i] = *reinterpret_cast<const uint4 *>(tile + (c0 + i * cs) * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = c0 + i * cs;
            if (c >= kChunks) break;
            uint4 w = v[i];
            if (!whole && ((c >> 3) & (BN - 1)) >= valid) {
                w = make_uint4(0u, 0u, 0u, 0u);
            } else {
                bad |= bf16x2_past_2p20(w.x) | bf16x2_past_2p20(w.y) | bf16x2_past_2p20(w.z) |
                       bf16x2_past_2p20(w.w);
                w.x = bf16x2_div16_to_f16x2(w.x);
                w.y = bf16x2_div16_to_f16x2(w.y);
                w.z = bf16x2_div16_to_f16x2(w.z);
                w.w = bf16x2_div16_to_f16x2(w.w);
            }
            *reinterpret_cast<uint4 *>(tile + c * 16) = w;
        }
    }
    if (__any_sync(0xffffffffu, bad != 0u) && (threadIdx.x & 31) == 0) record_error(err, ERR_RANGE | SRC_PREFILL);
}

// CVT (HALF only, no V' cache): V tiles are loaded as bf16 from v and the softmax
// warps convert each to V' in its ring stage (no conversion pass).
template <int D, bool EARLY, bool HALF, bool OBOX, bool CVT>
__global__ void __launch_bounds__(kPfThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                        const PrefillParams p) {
    using S = PfSmem<D, HALF>;
    constexpr int ST = S::kStages;
    extern __shared__ __align__(1024) uint8_t psmem_raw[];
    if constexpr (HALF) {
        // no slack for aligning the base: a misaligned one is reported (no access made)
        if (smem_u32(psmem_raw) & 1023u) {
            if (threadIdx.x == 0) record_error(p.err, ERR_TIMEOUT | SRC_PREFILL);
            return;
        }
    }
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(psmem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = sm;
    uint8_t *sRing = sm + S::kRingOff;
    uint8_t *sP = sm + S::kPOff;                   // P'_A, P'_B
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *q_empty = bars + 1;                  // this unit's QK^T have read Q
    // A ring stage holds K and V' tiles in turn, and the two kinds have different
    // consumers (the QK^T and the PV thread).  Each kind completes its own
    // barrier of the stage, so a consumer only ever waits for the next phase
    // of a barrier whose previous phase it has itself observed.
    uint64_t *full_k = bars + 2;                   // [ST]: a K tile landed in the stage
    uint64_t *full_v = full_k + ST;                // [ST]: a V' tile landed in the stage
    uint64_t *empty = full_v + ST;                 // [ST]: the stage's tile has been read
    uint64_t *s_full = empty + ST;                 // [2]: S_X(t) in TMEM
    uint64_t *s_free = s_full + 2;                 // [2]: the softmax has read S_X(t)
    uint64_t *p_ready = s_free + 2;                // [2]: P'_X(t) in shared memory (and O_X rescaled)
    uint64_t *pv_done = p_ready + 2;               // [2]: PV_X(t) complete
    uint64_t *drain = pv_done + 2;                 // [2]: per issuing thread
    uint64_t *idx_full = drain + 2;                // [2]: unit_idx[s] written
    uint64_t *idx_empty = idx_full + 2;            // [2]: every role has read unit_idx[s]
    uint64_t *pair_bar = idx_empty + 2;            // [4] (HALF): the two warps of a lane group exchanged a value
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + S::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *unit_idx = reinterpret_cast<volatile int *>(tmem_slot + 2);   // [2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;
    int *next_unit = p.unit_count + 1;   // zeroed by the scheduler

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full_k[i], 1);
            mbar_init(&full_v[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&s_free[x], HALF && x == 0 ? 256 : 128);   // HALF: both halves read slot A's S
            mbar_init(&p_ready[x], HALF && x == 0 ? 256 : 128);
            mbar_init(&pv_done[x], 1);
            mbar_init(&drain[x], 1);
            mbar_init(&idx_full[x], 1);
            mbar_init(&idx_empty[x], 2 + 256);   // both MMA threads and every softmax thread
        }
        if (HALF)
            for (int g = 0; g < 4; ++g) mbar_init(&pair_bar[g], 64);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // When G does not divide 128 the Q loads fill rows [128 / G * G, 128) of a
    // slot with nothing: zero them once, so those rows' scores are 0 (their
    // outputs are never written)
    if constexpr (!OBOX) {
        const int pad = BM - (BM / G) * G;
        constexpr int kSlots = HALF ? 1 : 2;
        const int per_panel = pad * 8;   // 16-byte chunks
        for (int i = threadIdx.x; i < kSlots * S::kPanels * per_panel; i += kPfThreads) {
            const int panel = i / per_panel, c = i % per_panel;
            *reinterpret_cast<uint4 *>(sQ + panel * S::kPanelBytes + (BM - pad) * 128 + c * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();   // seen by the tensor core's reads
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched as a programmatic dependent of the pre-pass: everything above ran
    // while it finished; its unit list (and V') are read only after this
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int num_units = p.unit_count[0];

    if (warp == 8) {
        // ================================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
        const bool paged = p.block_table != nullptr;
        const int oob_row = paged ? (int)(p.num_blocks * p.block_size) : 0;
        int it = 0, k = 0;
        uint32_t kpar = 0, vpar = 0, kused = 0, vused = 0;   // per stage: parity of the loads of each kind, any load
        bool ok = true;
        // lane 0 (EARLY): publish the counter value v as unit kk's index (-1: none
        // left) in the ring entry kk & 1 once every role has read the entry's
        // previous index; -1 without publishing when that wait gives up
        auto publish = [&](int kk, int v) {
            const int q = kk >> 1;
            if (q > 0 && !mbar_wait(&idx_empty[kk & 1], (uint32_t)(q - 1) & 1u, abort_flag, p.err, SRC_PREFILL))
                return -1;
            if (v >= num_units) v = -1;
            unit_idx[kk & 1] = v;
            mbar_arrive(&idx_full[kk & 1]);
            return v;
        };
        int u_next = -1;   // EARLY: unit k's index, published during unit k - 1
        if constexpr (EARLY) {
            if (lane == 0) u_next = publish(0, atomicAdd(next_unit, 1));
        }
        for (;; ++k) {
            int u = -1;
            if constexpr (EARLY) {
                u = __shfl_sync(0xffffffffu, u_next, 0);
            } else {
                // next unit index (-1: none left) into the ring entry k & 1
                if (lane == 0) {
                    const int q = k >> 1;
                    if (q == 0 ||
                        mbar_wait(&idx_empty[k & 1], (uint32_t)(q - 1) & 1u, abort_flag, p.err, SRC_PREFILL)) {
                        u = atomicAdd(next_unit, 1);
                        if (u >= num_units) u = -1;
                        unit_idx[k & 1] = u;
                        mbar_arrive(&idx_full[k & 1]);
                    }
                }
                u = __shfl_sync(0xffffffffu, u, 0);
            }
            if (u < 0 || !ok) break;
            // EARLY: the next unit, taken now (its atomic lands while this unit's Q is set up)
            int taken = -1;
            if constexpr (EARLY) taken = lane == 0 ? atomicAdd(next_unit, 1) : -1;
            const PfUnit w = pf_unit_k<HALF>(p, u);
            const int32_t *bt = paged ? p.block_table + (int64_t)w.b * p.bt_stride : nullptr;
            // Q of this unit once the previous unit's QK^T are done with the Q buffers
            int got = 1;
            if (lane == 0 && k > 0)
                got = mbar_wait(q_empty, (uint32_t)(k - 1) & 1u, abort_flag, p.err, SRC_PREFILL);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) break;
            if (lane == 0) {
                if (w.n > 0) {
                    const bool activeB = !HALF && w.t0B < w.Lq;   // HALF: no Q_B buffer
                    // a Q box is 128 / G tokens x G heads: 128 rows unless G does not divide 128
                    const uint32_t q_bytes =
                        OBOX ? (uint32_t)S::kTileBytes : (uint32_t)((BM / G) * G) * 128u * S::kPanels;
                    mbar_arrive_expect_tx(q_full, q_bytes * (activeB ? 2u : 1u));
#pragma unroll
                    for (int pn = 0; pn < S::kPanels; ++pn)
                        tma_load_3d(sQ + pn * S::kPanelBytes, &qmap, q_full, pn * 64, w.hkv * G, w.qs + w.t0A);
                    if (activeB) {
#pragma unroll
                        for (int pn = 0; pn < S::kPanels; ++pn)
                            tma_load_3d(sQ + S::kTileBytes + pn * S::kPanelBytes, &qmap, q_full, pn * 64,
                                        w.hkv * G, w.qs + w.t0B);
                    }
                } else {
                    mbar_arrive(q_full);
                }
                if constexpr (EARLY) u_next = publish(k + 1, taken);
            }
            // ring order K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}: each K tile
            // one step ahead of the V' tile it pairs with, so the next QK^T's tile can land
            // while the PV of the current one still holds its stage.  CVT: K_0, V_0, K_1,
            // V_1, ...: a V tile lands before the softmax threads come to convert it
            for (int j = 0; j < w.n && ok; ++j) {
                for (int step = 0; step < 3; ++step) {
                    int wv, tj;   // 0: K tile, 1: V tile; key tile index
                    if constexpr (CVT) {   // K_j, V_j
                        if (step == 1) continue;
                        wv = step == 2 ? 1 : 0, tj = j;
                    } else if (step == 0) {
                        if (j > 0) continue;
                        wv = 0, tj = 0;
                    } else if (step == 1) {
                        if (j + 1 >= w.n) continue;
                        wv = 0, tj = j + 1;
                    } else {
                        wv = 1, tj = j;
                    }
                    const int st = it % ST;
                    const uint32_t ph = (uint32_t)(it / ST) & 1u;
                    got = 1;
                    if (lane == 0) got = mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.err, SRC_PREFILL);
                    got = __shfl_sync(0xffffffffu, got, 0);
                    if (!got) { ok = false; break; }
                    uint8_t *dst = sRing + st * S::kTileBytes;
                    const CUtensorMap *map = wv ? &vmap : &kmap;
                    const int key0 = tj * BN;
                    uint64_t *bar = wv ? &full_v[st] : &full_k[st];
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar, (uint32_t)S::kTileBytes);
                        // V' converted by the pre-pass is contiguous by logical key (rows past
                        // the sequence hold the next sequence's keys or zeroed rows); a paged
                        // V' cache, or bf16 V converted here, is read like K
                        if (!paged || (wv == 1 && !p.v16_paged && !CVT)) {
#pragma unroll
                            for (int pn = 0; pn < S::kPanels; ++pn)
                                tma_load_3d(dst + pn * S::kPanelBytes, map, bar, pn * 64, w.hkv, w.ks0 + key0);
                        } else {
                            const int rpb = p.rows_per_box;
                            for (int i = 0; i < BN / rpb; ++i) {
                                const int key = key0 + i * rpb;
                                int row = oob_row;   // past the end of the cache: zero-filled
                                if (key < w.Lk) {
                                    const int blk = __ldg(bt + key / p.block_size);
                                    if (blk < 0 || (int64_t)blk >= p.num_blocks)
                                        record_error(p.err, ERR_INDEX | SRC_PREFILL);
                                    else
                                        row = blk * p.block_size + key % p.block_size;
                                }
#pragma unroll
                                for (int pn = 0; pn < S::kPanels; ++pn)
                                    tma_load_3d(dst + pn * S::kPanelBytes + i * rpb * 128, map, bar, pn * 64,
                                                w.hkv, row);
                            }
                        }
                    }
                    if (wv) {
                        vpar ^= 1u << st;
                        vused |= 1u << st;
                    } else {
                        kpar ^= 1u << st;
                        kused |= 1u << st;
                    }
                    ++it;
                }
            }
        }
        if (lane == 0) {
            // every copy issued here lands before the CTA may exit (the last load of
            // each kind in each stage completes the phase of parity count - 1)
            for (int st = 0; st < ST; ++st) {
                if ((kused >> st) & 1u) mbar_wait(&full_k[st], ((kpar >> st) & 1u) ^ 1u, nullptr, p.err, SRC_PREFILL);
                if ((vused >> st) & 1u) mbar_wait(&full_v[st], ((vpar >> st) & 1u) ^ 1u, nullptr, p.err, SRC_PREFILL);
            }
            if (k > 0) mbar_wait(q_full, (uint32_t)(k - 1) & 1u, nullptr, p.err, SRC_PREFILL);
        }
    } else if (warp == 9) {
        // ================================================================ QK^T issuer
        // S_X(t) may be issued as soon as the softmax of slot X has read S_X(t-1)
        // into registers: P' lives in shared memory, so S_X does not wait for PV.
        if (lane == 0) {
            const uint32_t tS[2] = {tmem, tmem + 128};
            const uint32_t qX[2] = {smem_u32(sQ), smem_u32(sQ + S::kTileBytes)};
            const uint32_t ring = smem_u32(sRing);
            int itb = 0, tc[2] = {0, 0}, k = 0;   // ring items before this unit; S tiles issued per slot
            uint32_t kpar = 0;                    // per stage: parity of the K tiles read from it
            bool ok = true;
            for (;; ++k) {
                ok = mbar_wait(&idx_full[k & 1], (uint32_t)(k >> 1) & 1u, abort_flag, p.err, SRC_PREFILL);
                if (!ok) break;
                const int u = unit_idx[k & 1];
                mbar_arrive(&idx_empty[k & 1]);
                if (u < 0) break;
                const PfUnit w = pf_unit_k<HALF>(p, u);
                const int nX[2] = {w.nA, w.nB};
                ok = mbar_wait(q_full, (uint32_t)k & 1u, abort_flag, p.err, SRC_PREFILL);
                if (!ok) break;
                tc_fence_after();
                for (int j = 0; j < w.n && ok; ++j) {
                    const int itK = itb + (CVT ? 2 * j : (j == 0 ? 0 : 2 * j - 1)), stK = itK % ST;   // the producer's ring order
                    ok = mbar_wait(&full_k[stK], (kpar >> stK) & 1u, abort_flag, p.err, SRC_PREFILL);
                    kpar ^= 1u << stK;
                    if (!ok) break;
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (j >= nX[x]) continue;
                        if (tc[x] > 0)
                            ok = ok && mbar_wait(&s_free[x], (uint32_t)(tc[x] - 1) & 1u, abort_flag, p.err,
                                                 SRC_PREFILL);
                        if (!ok) break;
                        tc_fence_after();
                        issue_qk<D>(tS[x], qX[x], ring + stK * S::kTileBytes);
                        tc_commit(&s_full[x]);
                        ++tc[x];
                    }
                    if (!ok) break;
                    tc_commit(&empty[stK]);
                }
                if (!ok) break;
                tc_commit(q_empty);   // completes when every QK^T of the unit has read Q
                itb += 2 * w.n;
            }
            // no MMA may still run when TMEM is released
            tc_commit(&drain[0]);
            mbar_wait(&drain[0], 0, nullptr, p.err, SRC_PREFILL);
        }
        __syncwarp();
    } else if (warp == 10) {
        // ================================================================ PV issuer
        if (lane == 0) {
            const uint32_t tO[2] = {tmem + 256, tmem + 256 + D};
            const uint32_t pX[2] = {smem_u32(sP), smem_u32(sP + kPBytes)};
            const uint32_t ring = smem_u32(sRing);
            int itb = 0, tc[2] = {0, 0}, k = 0;   // ring items before this unit; PV tiles issued per slot
            uint32_t vpar = 0;                    // per stage: parity of the V' tiles read from it
            bool ok = true;
            for (;; ++k) {
                ok = mbar_wait(&idx_full[k & 1], (uint32_t)(k >> 1) & 1u, abort_flag, p.err, SRC_PREFILL);
                if (!ok) break;
                const int u = unit_idx[k & 1];
                mbar_arrive(&idx_empty[k & 1]);
                if (u < 0) break;
                const PfUnit w = pf_unit_k<HALF>(p, u);
                const int nX[2] = {w.nA, w.nB};
                // PV_X(0) of a unit writes O_X afresh: its p_ready comes after the
                // softmax threads have read O_X of the previous unit
                for (int j = 0; j < w.n && ok; ++j) {
                    const int itV = itb + (CVT ? 2 * j + 1 : (j < w.n - 1 ? 2 * j + 2 : 2 * w.n - 1)), stV = itV % ST;
                    ok = mbar_wait(&full_v[stV], (vpar >> stV) & 1u, abort_flag, p.err, SRC_PREFILL);
                    vpar ^= 1u << stV;
                    if (!ok) break;
                    if (p.v16_paged && (j + 1) * BN > w.Lk) {
                        // with a paged V' cache the tile's rows past the sequence's last key
                        // come from cache slots that may hold anything (NaN included, and
                        // 0 * NaN is NaN inside the MMA): zero them first
                        const int r0 = max(w.Lk - j * BN, 0);
                        uint8_t *tile = sRing + stV * S::kTileBytes;
                        for (int pn = 0; pn < S::kPanels; ++pn)
                            for (int rr = r0; rr < BN; ++rr) {
                                uint4 *row = reinterpret_cast<uint4 *>(tile + pn * S::kPanelBytes + rr * 128);
#pragma unroll
                                for (int c = 0; c < 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
                            }
                        fence_proxy_async_smem();
                    }
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (j >= nX[x]) continue;
                        ok = ok && mbar_wait(&p_ready[x], (uint32_t)tc[x] & 1u, abort_flag, p.err, SRC_PREFILL);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv<D>(tO[x], pX[x], ring + stV * S::kTileBytes, j > 0);
                        tc_commit(&pv_done[x]);
                        ++tc[x];
                    }
                    if (!ok) break;
                    tc_commit(&empty[stV]);
                }
                if (!ok) break;
                itb += 2 * w.n;
            }
            tc_commit(&drain[1]);
            mbar_wait(&drain[1], 0, nullptr, p.err, SRC_PREFILL);
        }
        __syncwarp();
    } else if constexpr (HALF) {
        // ================================================================ softmax, one slot per unit
        // Warps w and w + 4 share a TMEM lane group: both take the same 32 rows of
        // slot A, w keys [0, 64) and w + 4 keys [64, 128) of every tile, each its
        // half of O's columns and its 64-key panel of P'.  A tile's row max and a
        // unit's row sum are exchanged between the two through a shared-memory area
        // of their own, synchronised by a bounded mbarrier per lane group.
        const int h = warp >> 2, g4 = warp & 3;
        const int r = g4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(g4 * 32) << 16;
        const uint32_t tS = tmem + (uint32_t)(h * 64) + lane_off;
        const uint32_t tO = tmem + 256u + lane_off;   // the slot's O; this half's columns [64 h, 64 h + 64)
        uint8_t *prow = sP + r * 128 + h * kPPanelBytes;   // this row of P'_A, this half's panel
        float *xch = reinterpret_cast<float *>(sm + S::kXchOff);   // [parity][half][row]
        const float sl2 = p.scale_log2;
        int cX = 0, k = 0, xp = 0;   // S tiles of slot A before this unit; exchanges so far
        bool ok = true;
        // the partner warp's value for this row (every exchange is made by both
        // warps of the lane group, in the same order)
        auto exchange = [&](float v) -> float {
            float *slot = xch + (xp & 1) * 256;
            slot[h * 128 + r] = v;
            mbar_arrive(&pair_bar[g4]);
            ok = __all_sync(0xffffffffu, mbar_wait(&pair_bar[g4], (uint32_t)xp & 1u, abort_flag, p.err,
                                                   SRC_PREFILL)) && ok;
            ++xp;
            return slot[(h ^ 1) * 128 + r];
        };
        bool pend = false, pend_tiles = false;
        int64_t pend_qbase = 0;
        int pend_ntok = 0, pend_hkv = 0;
        float pend_l = 0.f, pend_m = 0.f;
        int itb = 0;          // CVT: ring items before this unit (the producer's order)
        uint32_t vpar = 0;    // CVT: per stage, parity of the V tiles read from it
        for (;; ++k) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&idx_full[k & 1], (uint32_t)(k >> 1) & 1u, abort_flag, p.err, SRC_PREFILL));
            if (!ok) break;
            const int u = unit_idx[k & 1];
            mbar_arrive(&idx_empty[k & 1]);
            if (u < 0) break;
            const PfUnit w = pf_unit_k<HALF>(p, u);
            const int t0 = w.t0A;
            const int nX = w.nA;
            const int tok = t0 + r / G;
            const int lim = p.causal ? min(tok + w.off, w.Lk - 1) : w.Lk - 1;
            // lane groups holding none of the unit's rows (a decode-like unit fills few
            // of the slot's 128) skip the softmax and only keep the barriers' phases;
            // with CVT their threads convert the V tiles, which all 256 threads do when
            // every lane group holds rows
            const int ngrp = (min(max(w.Lq - t0, 0), BM / G) * G + 31) / 32;
            float m_ref = -INFINITY;
            float l = 0.f;   // this half's share of d'
            if (g4 >= ngrp) {
                for (int j = 0; j < nX; ++j) {
                    const int t = cX + j;
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&s_full[0], (uint32_t)t & 1u, abort_flag, p.err, SRC_PREFILL));
                    if (!ok) break;
                    mbar_arrive(&s_free[0]);
                    if constexpr (CVT) {
                        const int itV = itb + 2 * j + 1, stV = itV % ST;   // K_j, V_j order
                        const uint32_t vph = (vpar >> stV) & 1u;
                        vpar ^= 1u << stV;
                        ok = __all_sync(0xffffffffu, mbar_wait(&full_v[stV], vph, abort_flag, p.err, SRC_PREFILL));
                        if (!ok) break;
                        v_tile_to_f16<D>(sRing + stV * S::kTileBytes, w.Lk - j * BN, p.err,
                                         (h * (4 - ngrp) + (g4 - ngrp)) * 32 + lane, (4 - ngrp) * 64);
                    }
                    // p_ready(t) only after p_ready(t - 1) has completed (PV(t - 1) done)
                    if (t > 0) {
                        ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[0], (uint32_t)(t - 1) & 1u, abort_flag,
                                                               p.err, SRC_PREFILL));
                        if (!ok) break;
                        tc_fence_after();
                    }
                    if (pend) {
                        pf_store_rows_half<D, OBOX>(p, &omap, tO, sP, pend_tiles, pend_qbase, pend_ntok, pend_hkv,
                                                    pend_l, pend_m, h);
                        pend = false;
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(&p_ready[0]);
                }
            } else
            for (int j = 0; j < nX; ++j) {
                const int t = cX + j;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&s_full[0], (uint32_t)t & 1u, abort_flag, p.err, SRC_PREFILL));
                if (!ok) break;
                tc_fence_after();
                float s[64];
                tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tc_wait_ld();
                tc_fence_before();
                mbar_arrive(&s_free[0]);
                const int key0 = j * BN + h * 64;
                if (key0 + 63 > lim) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (key0 + c > lim) s[c] = -INFINITY;
                }
                float mx8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    mx8[q] = max3f(s[q], s[q + 8], s[q + 16]);
                    mx8[q] = max3f(mx8[q], s[q + 24], s[q + 32]);
                    mx8[q] = max3f(mx8[q], s[q + 40], s[q + 48]);
                    mx8[q] = fmaxf(mx8[q], s[q + 56]);
                }
                const float mxh =
                    max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                const float mx = fmaxf(mxh, exchange(mxh));
                if (!ok) break;
                // the same inputs in both halves: the same reference, alpha and need
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool need = m_new > m_ref + 8.0f;
                float alpha = 1.f;
                if (need) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
                    m_ref = m_new;
                }
                l *= alpha;
                const float nref = ((m_ref == -INFINITY) ? 0.f : -m_ref) + 4.0f;
                float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x0, x1;
                    fma2(x0, x1, s[2 * i], s[2 * i + 1], sl2, sl2, nref, nref);
                    x0 = ex2(x0);
                    x1 = ex2(x1);
                    add2(la[i & 3], lb[i & 3], x0, x1);
                    pk[i] = pack_f16x2(x0, x1);
                }
                l += ((la[0] + lb[0]) + (la[1] + lb[1])) + ((la[2] + lb[2]) + (la[3] + lb[3]));
                if constexpr (CVT) {
                    // V tile j (bf16 as loaded) -> V' = fp16(V / 16) in place, before p_ready;
                    // rows past the sequence's last key are zeroed.  Every thread keeps the
                    // stage parities; these threads convert only when no lane group is idle.
                    const int itV = itb + 2 * j + 1, stV = itV % ST;   // K_j, V_j order
                    const uint32_t vph = (vpar >> stV) & 1u;
                    vpar ^= 1u << stV;
                    if (ngrp == 4) {
                        ok = __all_sync(0xffffffffu, mbar_wait(&full_v[stV], vph, abort_flag, p.err, SRC_PREFILL));
                        if (!ok) break;
                        v_tile_to_f16<D>(sRing + stV * S::kTileBytes, w.Lk - j * BN, p.err, threadIdx.x, 256);
                    }
                }
                if (t > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[0], (uint32_t)(t - 1) & 1u, abort_flag, p.err,
                                                           SRC_PREFILL));
                    if (!ok) break;
                    tc_fence_after();
                }
                if (pend) {
                    pf_store_rows_half<D, OBOX>(p, &omap, tO, sP, pend_tiles, pend_qbase, pend_ntok, pend_hkv, pend_l,
                                          pend_m, h);
                    pend = false;
                }
                if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int c = 2 * h; c < 2 * h + 2; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + (uint32_t)(c * 32), o);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + (uint32_t)(c * 32), o);
                    }
                    tc_wait_st();
                }
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(prow + ((ch ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&p_ready[0]);
            }
            if (!ok) break;
            const float ltot = g4 < ngrp ? l + exchange(l) : 0.f;   // the unit's d' over both halves
            if (!ok) break;
            if (pend) {   // no key tiles in this unit: store the previous unit's rows now
                if (cX > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[0], (uint32_t)(cX - 1) & 1u, abort_flag, p.err,
                                                           SRC_PREFILL));
                    if (!ok) break;
                    tc_fence_after();
                }
                pf_store_rows_half<D, OBOX>(p, &omap, tO, sP, pend_tiles, pend_qbase, pend_ntok, pend_hkv, pend_l, pend_m,
                                      h);
            }
            cX += nX;
            if constexpr (CVT) itb += 2 * w.n;
            pend = true;
            pend_tiles = nX > 0;
            pend_qbase = (int64_t)w.qs + t0;
            pend_ntok = min(max(w.Lq - t0, 0), BM / G);
            pend_hkv = w.hkv;
            pend_l = ltot;
            pend_m = m_ref;
        }
        if (ok && pend) {
            if (cX > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[0], (uint32_t)(cX - 1) & 1u, abort_flag, p.err,
                                                       SRC_PREFILL));
            if (ok) {
                tc_fence_after();
                pf_store_rows_half<D, OBOX>(p, &omap, tO, sP, pend_tiles, pend_qbase, pend_ntok, pend_hkv, pend_l, pend_m,
                                      h);
            }
        }
        if (lane == 0) bulk_wait_all();
    } else {
        // ================================================================ softmax (one row per thread)
        const int X = warp >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + (uint32_t)(X * 128) + lane_off;
        const uint32_t tO = tmem + 256u + (uint32_t)(X * D) + lane_off;
        uint8_t *prow = sP + X * kPBytes + r * 128;   // this row of P'_X in both 64-key panels
        const float sl2 = p.scale_log2;
        int cX = 0, k = 0;   // S tiles of this slot before this unit
        bool ok = true;
        // The rows of the previous unit are stored once its last PV is done: in
        // the first tile of the next unit, after the exponentials and before
        // P'_X(0) is published (so PV_X(0) cannot overwrite O_X before it is read).
        bool pend = false, pend_tiles = false;
        int64_t pend_qbase = 0;   // packed row of the slot's first token
        int pend_ntok = 0, pend_hkv = 0;
        float pend_l = 0.f, pend_m = 0.f;
        uint8_t *pslot = sP + X * kPBytes;
        for (;; ++k) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&idx_full[k & 1], (uint32_t)(k >> 1) & 1u, abort_flag, p.err, SRC_PREFILL));
            if (!ok) break;
            const int u = unit_idx[k & 1];
            mbar_arrive(&idx_empty[k & 1]);
            if (u < 0) break;
            const PfUnit w = pf_unit_k<HALF>(p, u);
            const int t0 = X ? w.t0B : w.t0A;
            const int nX = X ? w.nB : w.nA;
            const int tok = t0 + r / G;
            // last key this row may see (negative: none)
            const int lim = p.causal ? min(tok + w.off, w.Lk - 1) : w.Lk - 1;
            float m_ref = -INFINITY;   // reference max (log2 units) used for P
            float l = 0.f;             // proxy denominator d'
            for (int j = 0; j < nX; ++j) {
                const int t = cX + j;   // S tiles of this slot so far
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&s_full[X], (uint32_t)t & 1u, abort_flag, p.err, SRC_PREFILL));
                if (!ok) break;
                tc_fence_after();
                float s[BN];
                tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
                tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
                tc_wait_ld();
                // S_X is in registers: the tensor core may overwrite it with S_X(t+1)
                tc_fence_before();
                mbar_arrive(&s_free[X]);
                const int key0 = j * BN;
                if (key0 + BN - 1 > lim) {
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (key0 + c > lim) s[c] = -INFINITY;
                }
                // row max: eight independent chains (chain q takes columns q, q + 8, ...)
                float mx8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    mx8[q] = max3f(s[q], s[q + 8], s[q + 16]);
#pragma unroll
                    for (int kk = 3; kk < 15; kk += 2) mx8[q] = max3f(mx8[q], s[q + 8 * kk], s[q + 8 * kk + 8]);
                    mx8[q] = fmaxf(mx8[q], s[q + 120]);
                }
                const float mx =
                    max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool need = m_new > m_ref + 8.0f;
                float alpha = 1.f;
                if (need) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
                    m_ref = m_new;
                }
                l *= alpha;
                // P' = 2^(s*scale*log2e - m_ref + 4) = 16 P as fp16, and the row sum in
                // four paired accumulators
                const float nref = ((m_ref == -INFINITY) ? 0.f : -m_ref) + 4.0f;
                float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[BN / 2];
#pragma unroll
                for (int i = 0; i < BN / 2; ++i) {
                    float x0, x1;
                    fma2(x0, x1, s[2 * i], s[2 * i + 1], sl2, sl2, nref, nref);
                    x0 = ex2(x0);
                    x1 = ex2(x1);
                    add2(la[i & 3], lb[i & 3], x0, x1);
                    pk[i] = pack_f16x2(x0, x1);
                }
                l += ((la[0] + lb[0]) + (la[1] + lb[1])) + ((la[2] + lb[2]) + (la[3] + lb[3]));
                // PV_X(t-1) has read P'_X and written O_X
                if (t > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[X], (uint32_t)(t - 1) & 1u, abort_flag, p.err,
                                                           SRC_PREFILL));
                    if (!ok) break;
                    tc_fence_after();
                }
                if (pend) {   // j == 0: O_X holds the previous unit's result
                    pf_store_rows<D, OBOX>(p, &omap, tO, pslot, pend_tiles, pend_qbase, pend_ntok, pend_hkv, pend_l, pend_m);
                    pend = false;
                }
                // O *= alpha where the reference moved (O of tile 0 is written, not accumulated)
                if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + (uint32_t)(c * 32), o);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + (uint32_t)(c * 32), o);
                    }
                    tc_wait_st();
                }
                // P' row into the two 128-byte-swizzled 64-key panels (K-major A operand)
#pragma unroll
                for (int pn = 0; pn < 2; ++pn) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const int i = pn * 32 + ch * 4;
                        *reinterpret_cast<uint4 *>(prow + pn * kPPanelBytes + ((ch ^ (r & 7)) << 4)) =
                            make_uint4(pk[i], pk[i + 1], pk[i + 2], pk[i + 3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&p_ready[X]);
            }
            if (!ok) break;
            if (pend) {   // no key tiles for slot X in this unit: store the previous unit's rows now
                if (cX > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[X], (uint32_t)(cX - 1) & 1u, abort_flag, p.err,
                                                           SRC_PREFILL));
                    if (!ok) break;
                    tc_fence_after();
                }
                pf_store_rows<D, OBOX>(p, &omap, tO, pslot, pend_tiles, pend_qbase, pend_ntok, pend_hkv, pend_l, pend_m);
            }
            cX += nX;
            pend = true;
            pend_tiles = nX > 0;
            pend_qbase = (int64_t)w.qs + t0;
            pend_ntok = min(max(w.Lq - t0, 0), BM / G);
            pend_hkv = w.hkv;
            pend_l = l;
            pend_m = m_ref;
        }
        // the last unit's rows
        if (ok && pend) {
            if (cX > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[X], (uint32_t)(cX - 1) & 1u, abort_flag, p.err,
                                                       SRC_PREFILL));
            if (ok) {
                tc_fence_after();
                pf_store_rows<D, OBOX>(p, &omap, tO, pslot, pend_tiles, pend_qbase, pend_ntok, pend_hkv, pend_l, pend_m);
            }
        }
        if (lane == 0) bulk_wait_all();   // this warp's output stores are complete before it exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// cu_seqlens for the kv-cache entry: cu_q[b] = b * seqlen_q, cu_k = exclusive
// prefix sum of cache_seqlens (each clamped to [0, max_cache_seqlen]; a value
// outside is reported).  One CTA.
// ---------------------------------------------------------------------------
constexpr int kCuThreads = 1024;

__global__ void __launch_bounds__(kCuThreads)
    attn_kvcache_cu_kernel(const int32_t *cache_seqlens, int batch, int seqlen_q, int max_cache_seqlen,
                           int32_t *cu_q, int32_t *cu_k, uint32_t *err) {
    __shared__ int wsum[kCuThreads / 32];
    const int per = (batch + kCuThreads - 1) / kCuThreads;
    const int b0 = threadIdx.x * per, b1 = min(b0 + per, batch);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
        int v = cache_seqlens[b];
        if (v < 0 || v > max_cache_seqlen) {
            record_error(err, ERR_INDEX | SRC_PREFILL);
            v = min(max(v, 0), max_cache_seqlen);
        }
        sum += v;
    }
    // exclusive scan of the per-thread sums
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int w = wsum[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        wsum[lane] = wi - w;
    }
    __syncthreads();
    int run = wsum[wid] + incl - sum;
    for (int b = b0; b < b1; ++b) {
        cu_k[b] = run;
        cu_q[b] = b * seqlen_q;
        run += min(max(cache_seqlens[b], 0), max_cache_seqlen);
    }
    if (threadIdx.x == kCuThreads - 1) {
        cu_k[batch] = wsum[wid] + incl;
        cu_q[batch] = batch * seqlen_q;
    }
}

// cu_seqlens of a padded batch: sequence b owns rows [b * seqlen, (b + 1) * seqlen)
__global__ void attn_padded_cu_kernel(int batch, int seqlen_q, int seqlen_k, int32_t *cu_q, int32_t *cu_k) {
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b <= batch; b += gridDim.x * blockDim.x) {
        cu_q[b] = b * seqlen_q;
        cu_k[b] = b * seqlen_k;
    }
}

cudaError_t launch_padded_cu(int batch, int seqlen_q, int seqlen_k, int32_t *cu_q, int32_t *cu_k,
                             cudaStream_t stream) {
    attn_padded_cu_kernel<<<(batch + 256) / 256, 256, 0, stream>>>(batch, seqlen_q, seqlen_k, cu_q, cu_k);
    return cudaGetLastError();
}

cudaError_t launch_kvcache_cu(const int32_t *cache_seqlens, int batch, int seqlen_q, int max_cache_seqlen,
                              int32_t *cu_q, int32_t *cu_k, uint32_t *err, cudaStream_t stream) {
    attn_kvcache_cu_kernel<<<1, kCuThreads, 0, stream>>>(cache_seqlens, batch, seqlen_q, max_cache_seqlen, cu_q,
                                                         cu_k, err);
    return cudaGetLastError();
}

template <int D, bool EARLY, bool HALF = false, bool OBOX = true, bool CVT = false>
static cudaError_t launch_prefill_t(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                    const CUtensorMap &omap, const PrefillParams &p, cudaStream_t stream) {
    using S = PfSmem<D, HALF>;
    static std::once_flag attr_once[kMaxDev];
    static cudaError_t attr_err[kMaxDev];
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::call_once(attr_once[dev], [&] {
        attr_err[dev] =
            cudaFuncSetAttribute(attn_prefill_kernel<D, EARLY, HALF, OBOX, CVT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kBytes);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    // unit list and V' in one launch: grid row 0 holds the scheduler (dispatched
    // before the conversion CTAs); with a paged V' cache the scheduler alone
    const dim3 cgrid = (p.v16_paged || p.v_cvt) ? dim3(1, 1)
                                                : dim3((p.max_seqlen_k + kCvtKeys - 1) / kCvtKeys, p.batch + 1);
    attn_prefill_prep_kernel<<<cgrid, kCvtThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    main_kernel_event_before(stream);
    // a programmatic dependent launch: the kernel's prologue overlaps the pre-pass's end
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(p.num_ctas);
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = S::kBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_prefill_kernel<D, EARLY, HALF, OBOX, CVT>, qmap, kmap, vmap, omap, p);
    if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
        (void)cudaGetLastError();
        attn_prefill_kernel<D, EARLY, HALF, OBOX, CVT><<<p.num_ctas, kPfThreads, S::kBytes, stream>>>(qmap, kmap, vmap, omap,
                                                                                           p);
        e = cudaGetLastError();
    }
    main_kernel_event_after(stream);
    return e;
}

cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const CUtensorMap &omap, const PrefillParams &p, int head_dim, cudaStream_t stream) {
    // a group that does not divide 128: slots of 128 / G * G rows, output rows
    // written row by row (the next unit always taken early; with a V' cache a
    // one-slot launch takes the two-slot instance)
    if (kPrefillSlotRows % p.G != 0) {
        if (head_dim == 128)
            return p.v_cvt ? launch_prefill_t<128, true, true, false, true>(qmap, kmap, vmap, omap, p, stream)
                           : launch_prefill_t<128, true, false, false>(qmap, kmap, vmap, omap, p, stream);
        return launch_prefill_t<64, false, false, false>(qmap, kmap, vmap, omap, p, stream);
    }
    // every sequence fits one query slot: slot B's softmax warps share slot A's
    // tiles, and convert V tiles themselves unless a V' cache is read
    if (head_dim == 128 && p.one_slot)
        return p.v_cvt ? launch_prefill_t<128, true, true, true, true>(qmap, kmap, vmap, omap, p, stream)
                       : launch_prefill_t<128, true, true>(qmap, kmap, vmap, omap, p, stream);
    // the next unit taken a unit ahead when keys are short (each unit's K / V is
    // small, so its siblings gain little from sharing it through L2) or when every
    // sequence is one query pair (a unit has no siblings)
    if (head_dim == 128)
        return (p.max_seqlen_k <= kEarlyMaxKeys || p.max_pairs == 1)
                   ? launch_prefill_t<128, true>(qmap, kmap, vmap, omap, p, stream)
                   : launch_prefill_t<128, false>(qmap, kmap, vmap, omap, p, stream);
    return launch_prefill_t<64, false>(qmap, kmap, vmap, omap, p, stream);
}

}  // namespace attn
