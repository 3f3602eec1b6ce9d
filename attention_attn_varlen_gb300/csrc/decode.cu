// decode.cu -- decode through the paged KV cache: one query token per sequence
// ("从零实现 vLLM (1.3)：如何加速 Attention 计算", section "Decode":
// flash_attn_with_kvcache(q.unsqueeze(1), k_cache, v_cache, cache_seqlens,
// block_table, softmax_scale, causal=True)), or a few (seqlen_q = Sq > 1, the
// same call with q of shape [B, Sq, H, D] and the bottom-right causal mask:
// new token t of a sequence with L cached keys sees keys j <= L - Sq + t), as a
// split-KV pass plus an exact log-sum-exp combine.
//
// The work is HBM-bound: every cached K/V byte of a (sequence, KV head) is read
// once and serves all Sq x G query rows of the group (G = Hq/Hkv heads).
//
// attn_decode_split_kernel: one CTA per (split, column group, KV head, sequence).
//   warp 4 (lane 0)   TMA producer: 64-token K and V tiles of the split,
//                     addressed through the block table, into a 3-stage ring
//                     of 128-byte-swizzled shared-memory panels.
//   warps 0-3         consumers: each takes 16 of the 64 tokens of every tile
//                     and keeps its own online-softmax state (m, d', o') for
//                     its tokens ("减少遍历次数的“在线 Softmax”" and
//                     "FlashAttention 的最终实现": running max, proxy
//                     denominator, proxy output rescaled by 2^(m_old - m_new)).
//                     The reference m of a column moves only when a tile's
//                     max exceeds it by more than 8 (log2 units), so the
//                     rescale is rare and P stays <= 256; d', o' and the
//                     merges all use that reference, so the result is the same.
//                     S^T = K Q^T and O^T += V^T P^T run on mma.sync m16n8k16
//                     with the tokens (then head_dim) in M and the Sq x G
//                     query columns (token-major) in N: up to 16 per CTA
//                     (one or two n8 tiles); more columns are split into
//                     groups of 16 over adjacent CTAs that read the same K/V
//                     tiles (the repeats come from L2).  Each column masks the
//                     keys past its own causal limit.  P^T is moved into the B-operand layout
//                     with movmatrix.  The four warps' states are merged
//                     exactly at the end.
// attn_decode_combine_kernel: one warp per (query row, query head) merges the
//   split partials: lse = log2 sum_s 2^lse_s, O = sum_s 2^(lse_s - lse) O_s.
//   This merge is exact because the update is associative ("计算流程（1-Pass
//   算法与分块）": tiles may be folded in any grouping).  A split that holds no
//   key a row may see leaves lse_s = -inf and weight 0.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace attn {

constexpr int kDecThreads = 160;   // 4 consumer warps + 1 producer warp
constexpr int kDecTile = 64;       // tokens per ring stage
constexpr int kDecPrefetch = 3;   // tiles ahead of the loads that the L2 prefetch runs (two-stage ring)

// bulk prefetch of one tensor-map box into L2 (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// QS: the CTA's query columns live in shared memory (read by ldmatrix per tile)
// instead of in every consumer's registers, which lets three CTAs share an SM;
// each then keeps two ring stages instead of three
template <int D, bool QS = false>
struct DecSmem {
    static constexpr int kStages = QS ? 2 : 3;
    static constexpr int kPanels = D / 64;
    static constexpr int kPanelBytes = kDecTile * 128;             // 64 rows x 128 B
    static constexpr int kStageBytes = 2 * kPanels * kPanelBytes;  // K then V
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kQBytes = QS ? 16 * D * 2 : 0;            // 16 query columns x D bf16, swizzled
    static constexpr int kBytes = kRingBytes + kQBytes + 1024 /*align slack*/ + 64 /*barriers*/;
};


// VH: V tiles come from the fp16 V / 16 cache; PV then multiplies them by one fp16
// term P' = 16 P (11 significant bits) instead of P's bf16 hi + lo terms.
template <int D, int NT, bool VH, bool QS>
__global__ void __launch_bounds__(kDecThreads, QS ? 3 : 0) attn_decode_split_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using S = DecSmem<D, QS>;
    constexpr int kDecStages = S::kStages;
    static_assert(!QS || NT == 2, "query columns in shared memory: two n8 tiles");
    constexpr int KS = D / 16;       // k-steps of the QK^T product
    constexpr int NC = 8 * NT;       // query columns, padded to whole n8 tiles
    extern __shared__ uint8_t dsmem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = ring + S::kRingBytes;   // QS: [16 columns][D], 16-byte chunks XOR-swizzled by column
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + S::kRingBytes + S::kQBytes);
    uint64_t *empty = full + kDecStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kDecStages);

    // blockIdx.x = split * ncg + column group: the CTAs of one split's column groups
    // are adjacent, so the second and later read the split's K/V tiles from L2
    const int split = blockIdx.x / p.ncg, cgrp = blockIdx.x % p.ncg, hkv = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's columns: global column c0 + n (n < NQ) is query token (c0 + n) / G,
    // head hkv * G + (c0 + n) % G
    const int c0 = cgrp * NC;
    const int NQ = min(NC, p.Sq * p.G - c0);
    int L = __ldg(p.cache_seqlens + b);
    if (L < 0 || L > p.max_seqlen) {
        // outside [0, max_seqlen]: reported once, then clamped
        if (split == 0 && cgrp == 0 && threadIdx.x == 0) record_error(p.err, ERR_INDEX | SRC_DECODE);
        L = L < 0 ? 0 : p.max_seqlen;
    }
    const int s0 = split * p.split_tokens;
    if (s0 >= L) {
        // no tokens for this split.  With one split the output is written here.
        if (p.num_splits == 1 && split == 0) {
            for (int i = threadIdx.x; i < NQ * D; i += kDecThreads) {
                const int n = c0 + i / D, d = i % D;
                const int h = hkv * p.G + n % p.G;
                const int64_t row = (int64_t)b * p.Sq + n / p.G;
                p.out[row * p.out_row_stride + (int64_t)h * D + d] = __float2bfloat16(0.f);
                if (p.lse && d == 0) p.lse[row * p.lse_row_stride + (int64_t)h * p.lse_head_stride] = -INFINITY;
            }
        }
        return;
    }
    const int s1 = min(L, s0 + p.split_tokens);
    const int n_tiles = (s1 - s0 + kDecTile - 1) / kDecTile;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            const int rpb = p.rows_per_box;
            const int boxes = kDecTile / rpb;
            const uint32_t box_bytes = (uint32_t)rpb * 128u;
            const int32_t *bt = p.block_table + (int64_t)b * p.bt_stride;
            const int oob_row = (int)(p.num_blocks * p.block_size);   // one past the last row: zero-filled
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % kDecStages;
                const uint32_t ph = (uint32_t)(t / kDecStages) & 1u;
                if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.err, SRC_DECODE)) break;
                issued = t + 1;
                const int tok0 = s0 + t * kDecTile;
                int nb = 0;
                for (int i = 0; i < boxes; ++i)
                    if (tok0 + i * rpb < s1) ++nb;
                mbar_arrive_expect_tx(&full[st], (uint32_t)nb * box_bytes * 2u * S::kPanels);
                uint8_t *kbase = ring + st * S::kStageBytes;
                uint8_t *vbase = kbase + S::kPanels * S::kPanelBytes;
                for (int i = 0; i < nb; ++i) {
                    const int tok = tok0 + i * rpb;
                    int blk = __ldg(bt + tok / p.block_size);
                    int row;
                    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                        record_error(p.err, ERR_INDEX | SRC_DECODE);
                        row = oob_row;
                    } else {
                        row = blk * p.block_size + tok % p.block_size;
                    }
#pragma unroll
                    for (int pn = 0; pn < S::kPanels; ++pn) {
                        tma_load_3d(kbase + pn * S::kPanelBytes + i * box_bytes, &kmap, &full[st], pn * 64, hkv, row);
                        tma_load_3d(vbase + pn * S::kPanelBytes + i * box_bytes, &vmap, &full[st], pn * 64, hkv, row);
                    }
                }
                if constexpr (QS) {
                    // two ring stages hold less than the load latency covers here: the first
                    // column group's producer pulls the K / V boxes kDecPrefetch tiles ahead
                    // into L2, so those tiles' loads (its own and the other groups') hit L2
                    if (cgrp == 0) {
                        const int tp0 = s0 + (t + kDecPrefetch) * kDecTile;
                        for (int i = 0; i < boxes; ++i) {
                            const int tok = tp0 + i * rpb;
                            if (tok >= s1) break;
                            const int blk = __ldg(bt + tok / p.block_size);
                            if (blk < 0 || (int64_t)blk >= p.num_blocks) continue;   // reported by its load
                            const int row = blk * p.block_size + tok % p.block_size;
#pragma unroll
                            for (int pn = 0; pn < S::kPanels; ++pn) {
                                tma_prefetch_l2_3d(&kmap, pn * 64, hkv, row);
                                tma_prefetch_l2_3d(&vmap, pn * 64, hkv, row);
                            }
                        }
                    }
                }
            }
            // keep the CTA (and its shared memory) alive until every copy this
            // thread issued has landed, even if the consumers gave up
            for (int t = issued - kDecStages < 0 ? 0 : issued - kDecStages; t < issued; ++t)
                mbar_wait(&full[t % kDecStages], (uint32_t)(t / kDecStages) & 1u, nullptr, p.err, SRC_DECODE);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    // Q^T as B fragments of n-tile nt: b0 = Q[n=8nt+g][16ks + 2c .. +1], b1 = Q[8nt+g][16ks + 2c + 8 .. +9]
    uint32_t qf[QS ? 1 : NT][QS ? 1 : KS][2];
    if constexpr (QS) {
        // the CTA's 16 query columns into shared memory: row n (column c0 + n, zeros
        // past NQ) holds its D values, 16-byte chunk ch at chunk ch ^ (n & 7)
        for (int i = threadIdx.x; i < 16 * (D / 8); i += 128) {
            const int n = i / (D / 8), ch = i % (D / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (n < NQ) {
                const int gn = c0 + n;
                const uint32_t *src = reinterpret_cast<const uint32_t *>(
                    p.q + ((int64_t)b * p.Sq + gn / p.G) * p.q_row_stride + (int64_t)(hkv * p.G + gn % p.G) * D) +
                                      ch * 4;
                v = make_uint4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
            }
            *reinterpret_cast<uint4 *>(sQ + n * (D * 2) + ((ch ^ (n & 7)) << 4)) = v;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    // keys at or past kend[nt][j] are masked for this lane's column 8nt + 2c + j:
    // the end of the split and, causally, the bottom-right limit L - Sq + t + 1
    int kend[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        const bool valid = n < NQ;
        const int gn = c0 + n;
        if constexpr (!QS) {
            const int64_t qrow_idx = (int64_t)b * p.Sq + (valid ? gn / p.G : 0);
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                p.q + qrow_idx * p.q_row_stride + (int64_t)(hkv * p.G + (valid ? gn % p.G : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qf[nt][ks][0] = valid ? __ldg(qrow + ks * 8 + c) : 0u;
                qf[nt][ks][1] = valid ? __ldg(qrow + ks * 8 + 4 + c) : 0u;
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = nt * 8 + 2 * c + j;
            int e = s1;
            if (p.causal && col < NQ) e = min(e, L - p.Sq + (c0 + col) / p.G + 1);
            kend[nt][j] = e;
        }
    }
    float m[NT][2], l[NT][2];
    float o[NT][KS][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int i = 0; i < KS; ++i) o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
    }

    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % kDecStages;
        const uint32_t ph = (uint32_t)(t / kDecStages) & 1u;
        if (!mbar_wait(&full[st], ph, abort_flag, p.err, SRC_DECODE)) { ok = false; break; }
        const int tok0 = s0 + t * kDecTile;
        const int nvalid = s1 - tok0;   // >= 1
        const uint32_t kb = smem_u32(ring + st * S::kStageBytes);
        const uint32_t vb = kb + S::kPanels * S::kPanelBytes;
        const int r0 = warp * 16;
        if (r0 < nvalid) {
            const bool tail = r0 + 16 > nvalid;
            if (tail) {
                // rows past the sequence may hold anything (even NaN): zero this
                // warp's V rows there so P = 0 never meets a non-finite value
                uint8_t *vgen = ring + st * S::kStageBytes + S::kPanels * S::kPanelBytes;
                for (int i = lane; i < 16 * (D / 8); i += 32) {
                    const int r = r0 + i / (D / 8);
                    const int ch = i % (D / 8);
                    if (r >= nvalid)
                        *reinterpret_cast<uint4 *>(vgen + (ch / 8) * S::kPanelBytes + sw128_off(r, ch % 8)) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // S^T[16 tokens x 8 columns] = K[16 x D] * Q^T[D x 8], per n-tile
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            const int arow = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a0, a1, a2, a3;
                const uint32_t addr = kb + (ks / 4) * S::kPanelBytes + sw128_off(arow, (ks % 4) * 2 + (lane >> 4));
                ldsm_x4(addr, a0, a1, a2, a3);
                if constexpr (QS) {
                    // Q^T B fragments of both n8 tiles: matrix m = lane / 8 is column block
                    // m / 2, k half m % 2 of this k-step
                    const int qn = ((lane >> 4) << 3) + (lane & 7), qch = 2 * ks + ((lane >> 3) & 1);
                    uint32_t b00, b01, b10, b11;
                    ldsm_x4(smem_u32(sQ) + qn * (D * 2) + ((qch ^ (qn & 7)) << 4), b00, b01, b10, b11);
                    mma_bf16_16816(acc[0], a0, a1, a2, a3, b00, b01);
                    mma_bf16_16816(acc[1], a0, a1, a2, a3, b10, b11);
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(acc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
                }
            }
            const int key0 = tok0 + r0 + g, key1 = key0 + 8;
            uint32_t bp[NT][2], bl[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // scale into the log2 domain, mask keys past each column's end
                float s_0 = acc[nt][0] * sl2, s_1 = acc[nt][1] * sl2, s_2 = acc[nt][2] * sl2, s_3 = acc[nt][3] * sl2;
                if (key0 >= kend[nt][0]) s_0 = -INFINITY;
                if (key0 >= kend[nt][1]) s_1 = -INFINITY;
                if (key1 >= kend[nt][0]) s_2 = -INFINITY;
                if (key1 >= kend[nt][1]) s_3 = -INFINITY;
                // the reference of a column moves only when the tile's max exceeds it by
                // more than 8 (log2 units): P <= 256, and O is rarely rescaled.  Whether
                // any value of the warp does is one vote; the column maxima (over the
                // eight lanes sharing a column) are reduced only then.
                float mx0 = fmaxf(s_0, s_2), mx1 = fmaxf(s_1, s_3);
                if (__any_sync(0xffffffffu, mx0 > m[nt][0] + 8.f || mx1 > m[nt][1] + 8.f)) {
#pragma unroll
                    for (int sh = 4; sh < 32; sh <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
                    }
                    const bool nd0 = mx0 > m[nt][0] + 8.f, nd1 = mx1 > m[nt][1] + 8.f;
                    const float a_0 = !nd0 ? 1.f : (m[nt][0] == -INFINITY) ? 0.f : ex2(m[nt][0] - mx0);
                    const float a_1 = !nd1 ? 1.f : (m[nt][1] == -INFINITY) ? 0.f : ex2(m[nt][1] - mx1);
                    if (nd0) m[nt][0] = mx0;
                    if (nd1) m[nt][1] = mx1;
                    l[nt][0] *= a_0;
                    l[nt][1] *= a_1;
#pragma unroll
                    for (int i = 0; i < KS; ++i) {
                        o[nt][i][0] *= a_0;
                        o[nt][i][1] *= a_1;
                        o[nt][i][2] *= a_0;
                        o[nt][i][3] *= a_1;
                    }
                }
                const float ref0 = (m[nt][0] == -INFINITY) ? 0.f : m[nt][0];
                const float ref1 = (m[nt][1] == -INFINITY) ? 0.f : m[nt][1];
                const float p0 = ex2(s_0 - ref0), p2 = ex2(s_2 - ref0);
                const float p1 = ex2(s_1 - ref1), p3 = ex2(s_3 - ref1);
                l[nt][0] += p0 + p2;
                l[nt][1] += p1 + p3;
                // P^T into the B layout: rows = tokens, cols = query columns -> transpose.
                if constexpr (VH) {
                    // P' = 16 P as fp16 against V' = V / 16: the product is P V
                    bp[nt][0] = movmatrix_t(pack_f16x2(16.f * p0, 16.f * p1));
                    bp[nt][1] = movmatrix_t(pack_f16x2(16.f * p2, 16.f * p3));
                } else {
                    // P is carried as bf16 hi + lo terms (about 16 significant bits)
                    const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
                    bp[nt][0] = movmatrix_t(h01);
                    bp[nt][1] = movmatrix_t(h23);
                    bl[nt][0] = movmatrix_t(
                        pack_bf16x2(p0 - __uint_as_float(h01 << 16), p1 - __uint_as_float(h01 & 0xFFFF0000u)));
                    bl[nt][1] = movmatrix_t(
                        pack_bf16x2(p2 - __uint_as_float(h23 << 16), p3 - __uint_as_float(h23 & 0xFFFF0000u)));
                }
            }
            // O^T[D x 8] += V^T[D x 16 tokens] * P^T[16 x 8], per n-tile
            const int mi = lane >> 3;
            const int vrow = r0 + (lane & 7) + (mi >> 1) * 8;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int ch = 2 * mt + (mi & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vb + (ch / 8) * S::kPanelBytes + sw128_off(vrow, ch % 8), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if constexpr (VH) {
                        mma_f16_16816(o[nt][mt], a0, a1, a2, a3, bp[nt][0], bp[nt][1]);
                    } else {
                        mma_bf16_16816(o[nt][mt], a0, a1, a2, a3, bp[nt][0], bp[nt][1]);
                        mma_bf16_16816(o[nt][mt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
                    }
                }
            }
            if (tail) fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---------------------------------------------------------------- merge the four warps
    // full per-warp denominators
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], sh);
            l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], sh);
        }
    }
    // all consumer warps are past the ring: reuse stage memory for the merge
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (*abort_flag) ok = false;
    float *mo = reinterpret_cast<float *>(ring);          // [4][D][NC]
    float *mm = mo + 4 * D * NC;                          // [4][NC]
    float *ml = mm + 4 * NC;                              // [4][NC]
    if (ok) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int cc = nt * 8 + 2 * c;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int d = mt * 16 + g;
                mo[(warp * D + d) * NC + cc] = o[nt][mt][0];
                mo[(warp * D + d) * NC + cc + 1] = o[nt][mt][1];
                mo[(warp * D + d + 8) * NC + cc] = o[nt][mt][2];
                mo[(warp * D + d + 8) * NC + cc + 1] = o[nt][mt][3];
            }
            if (g == 0) {
                mm[warp * NC + cc] = m[nt][0];
                mm[warp * NC + cc + 1] = m[nt][1];
                ml[warp * NC + cc] = l[nt][0];
                ml[warp * NC + cc + 1] = l[nt][1];
            }
        }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (!ok) {
        // a bounded wait gave up (the error word says so): leave NaN, not the
        // previous contents of the output or of the split partials, so that a
        // result of this call can never look plausible
        for (int i = threadIdx.x; i < NQ * D; i += 128) {
            const int n = i / D, d = i % D;
            const int h = hkv * p.G + (c0 + n) % p.G;
            const int64_t row = (int64_t)b * p.Sq + (c0 + n) / p.G;
            if (p.num_splits == 1) {
                p.out[row * p.out_row_stride + (int64_t)h * D + d] = __float2bfloat16(NAN);
                if (p.lse && d == 0) p.lse[row * p.lse_row_stride + (int64_t)h * p.lse_head_stride] = NAN;
            } else {
                const int64_t prow = (row * p.Hq + h) * p.num_splits + split;
                p.o_part[prow * D + d] = NAN;
                if (d == 0) p.lse_part[prow] = NAN;
            }
        }
        return;
    }
    for (int i = threadIdx.x; i < NQ * D; i += 128) {
        const int n = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, mm[w * NC + n]);
        float Ls = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float mw = mm[w * NC + n];
                const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
                Ls += ml[w * NC + n] * f;
                O += mo[(w * D + d) * NC + n] * f;
            }
        }
        const int h = hkv * p.G + (c0 + n) % p.G;
        const int64_t row = (int64_t)b * p.Sq + (c0 + n) / p.G;
        const float on = Ls > 0.f ? O / Ls : 0.f;
        const float l2 = Ls > 0.f ? M + __log2f(Ls) : -INFINITY;
        if (p.num_splits == 1) {
            p.out[row * p.out_row_stride + (int64_t)h * D + d] = __float2bfloat16(on);
            if (p.lse && d == 0)
                p.lse[row * p.lse_row_stride + (int64_t)h * p.lse_head_stride] = l2 * 0.69314718055994531f;
        } else {
            const int64_t prow = (row * p.Hq + h) * p.num_splits + split;
            p.o_part[prow * D + d] = on;
            if (d == 0) p.lse_part[prow] = l2;
        }
    }
}

// One warp per (query row, query head): exact merge of the split partials.
template <int D>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(const DecodeParams p, int total_rows) {
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= total_rows) return;
    const int per_seq = p.Sq * p.Hq;
    const int b = w / per_seq, t = (w % per_seq) / p.Hq, h = w % p.Hq;
    int L = __ldg(p.cache_seqlens + b);
    L = L < 0 ? 0 : (L > p.max_seqlen ? p.max_seqlen : L);   // the split kernel's clamp
    int ns = L <= 0 ? 0 : (L + p.split_tokens - 1) / p.split_tokens;
    if (ns > p.num_splits) ns = p.num_splits;
    const int64_t row0 = (int64_t)w * p.num_splits;
    float la = lane < ns ? p.lse_part[row0 + lane] : -INFINITY;
    float lb = lane + 32 < ns ? p.lse_part[row0 + lane + 32] : -INFINITY;
    float M = fmaxf(la, lb);
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
    const float wa = (la == -INFINITY) ? 0.f : ex2(la - M);
    const float wb = (lb == -INFINITY) ? 0.f : ex2(lb - M);
    float Ls = wa + wb;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, sh);
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float ws = __shfl_sync(0xffffffffu, s < 32 ? wa : wb, s & 31);
        if (ws == 0.f) continue;   // warp-uniform; a split that saw no key of this row holds 0 partials
        const float *src = p.o_part + (row0 + s) * D + lane * PER;
        if (PER == 4) {
            const float4 v4 = *reinterpret_cast<const float4 *>(src);
            acc[0] += ws * v4.x;
            acc[1] += ws * v4.y;
            acc[2] += ws * v4.z;
            acc[3] += ws * v4.w;
        } else {
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[i] += ws * src[i];
        }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    const int64_t row = (int64_t)b * p.Sq + t;
    __nv_bfloat16 *dst = p.out + row * p.out_row_stride + (int64_t)h * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) dst[i] = __float2bfloat16(acc[i] * inv);
    if (p.lse && lane == 0)
        p.lse[row * p.lse_row_stride + (int64_t)h * p.lse_head_stride] =
            Ls > 0.f ? (M + __log2f(Ls)) * 0.69314718055994531f : -INFINITY;
}

template <int D, int NT, bool VH, bool QS = false>
static cudaError_t launch_decode_t(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                                   int batch, cudaStream_t stream) {
    using S = DecSmem<D, QS>;
    static std::once_flag attr_once[kMaxDev];
    static cudaError_t attr_err[kMaxDev];
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::call_once(attr_once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(attn_decode_split_kernel<D, NT, VH, QS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    dim3 grid(p.num_splits * p.ncg, p.Hkv, batch);
    main_kernel_event_before(stream);
    attn_decode_split_kernel<D, NT, VH, QS><<<grid, kDecThreads, S::kBytes, stream>>>(kmap, vmap, p);
    main_kernel_event_after(stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.num_splits == 1) return e;
    const int rows = batch * p.Sq * p.Hq;
    attn_decode_combine_kernel<D><<<(rows + 3) / 4, 128, 0, stream>>>(p, rows);
    return cudaGetLastError();
}

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p, int batch,
                          int head_dim, cudaStream_t stream) {
    const bool two = p.Sq * p.G > 8;
    // several column groups (more than 16 query columns per KV head): their CTAs
    // read the same tiles, and three per SM keep more consumer warps in flight
    const bool qs = p.ncg > 1;
    if (p.v16) {
        if (head_dim == 128)
            return two ? launch_decode_t<128, 2, true>(kmap, vmap, p, batch, stream)
                       : launch_decode_t<128, 1, true>(kmap, vmap, p, batch, stream);
        return two ? launch_decode_t<64, 2, true>(kmap, vmap, p, batch, stream)
                   : launch_decode_t<64, 1, true>(kmap, vmap, p, batch, stream);
    }
    if (head_dim == 128)
        return two ? (qs ? launch_decode_t<128, 2, false, true>(kmap, vmap, p, batch, stream)
                         : launch_decode_t<128, 2, false>(kmap, vmap, p, batch, stream))
                   : launch_decode_t<128, 1, false>(kmap, vmap, p, batch, stream);
    return two ? launch_decode_t<64, 2, false>(kmap, vmap, p, batch, stream)
               : launch_decode_t<64, 1, false>(kmap, vmap, p, batch, stream);
}

}  // namespace attn

namespace attn {

// ---------------------------------------------------------------------------
// Statically reserved scratch for attn_decode_paged_noalloc.
//
// Some callers cannot allocate device memory when they decode: a serving
// loop that has handed all free memory to its paged KV-cache pool at start-up,
// or code that must not call cudaMalloc on its hot path because it may
// synchronise the device and stall other streams.  For them the split
// partials live in this fixed array instead of a caller workspace.  It is
// part of the module image, so every GPU that loads the library holds these
// bytes until the process exits.  All calls share it: two calls that overlap
// on the GPU (different streams, no ordering between them) race on it.
// Nothing in it needs clearing between calls: every partial the combine
// kernel reads is written earlier by the same call (a split CTA whose bounded
// wait gave up writes NaN partials, so stale contents never reach the output).
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchBytes = 32ull << 20;   // 32 MiB
static __device__ __align__(256) float g_decode_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::once_flag g_scratch_once[kMaxDev];
float *g_scratch_ptr[kMaxDev];
cudaError_t g_scratch_err[kMaxDev];
}  // namespace

// Device address of the static scratch on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress, with that device current),
// once even if several host threads get there together; later calls reuse the
// cached address.
cudaError_t decode_noalloc_scratch(float **ptr, size_t *bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::call_once(g_scratch_once[dev], [&] {
        void *p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
        g_scratch_ptr[dev] = reinterpret_cast<float *>(p);
    });
    if (g_scratch_err[dev] != cudaSuccess) return g_scratch_err[dev];
    *ptr = g_scratch_ptr[dev];
    *bytes = kNoAllocScratchBytes;
    return cudaSuccess;
}

}  // namespace attn
