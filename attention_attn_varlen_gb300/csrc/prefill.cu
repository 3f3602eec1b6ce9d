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
// Work unit (one CTA): a sequence b, a KV head, and two query "slots" A and B
// of 128 rows each.  A slot packs 128/G consecutive tokens x the G query heads
// that share the KV head (row r = token_offset * G + g), so one K/V stream
// feeds 256 query rows.  Slot B holds the 128/G tokens after slot A.
//
// Roles (320 threads):
//   warps 0-3  softmax for slot A, one thread per row (TMEM lanes 0-127)
//   warps 4-7  softmax for slot B
//   warp 8     TMA producer: Q_A, Q_B once, then K_j, V_j tiles through a
//              4-stage ring (128 keys x head_dim, 128-byte swizzle)
//   warp 9     TMEM allocator and single-thread MMA issuer
// TMEM (512 columns): S_A [0,128), S_B [128,256) fp32; O_A, O_B after them.
// P is written back by the softmax threads over S: P_hi = bf16(P) in columns
// 0-63, P_lo = bf16(P - P_hi) in columns 64-127; PV runs on both terms.
//
// MMA order per key tile j:  S_A(j), PV_B(j-1), S_B(j), PV_A(j)
// so the tensor core works on one slot while the other slot's softmax runs.
// Because tcgen05 operations of one thread complete in order, the commit of
// S_X(j) also covers PV_X(j-1): a softmax thread that sees S_X(j) may rescale
// O_X safely.
//
// The rescale is lazy: the reference max of a row moves only when the tile
// max exceeds it by more than 8 (log2 units), so P stays <= 256 and O is
// rarely touched; the final O / d' uses the same reference, so the result is
// unchanged.
#include "common.cuh"
#include "kernels.h"

namespace attn {

constexpr int kPfThreads = 320;
constexpr int kPfStages = 4;
constexpr int BM = kPrefillSlotRows;   // 128 rows per slot
constexpr int BN = kPrefillKeyTile;    // 128 keys per tile

template <int D>
struct PfSmem {
    static constexpr int kPanels = D / 64;
    static constexpr int kPanelBytes = 128 * 128;            // 128 rows x 128 B
    static constexpr int kTileBytes = kPanels * kPanelBytes; // one Q slot, K tile or V tile
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBarOff = kRingOff + kPfStages * kTileBytes;
    static constexpr int kNumBars = 17;
    static constexpr int kBytes = kBarOff + kNumBars * 8 + 16 + 1024 /*align slack*/;
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

// O (+)= P_hi V + P_lo V.  P is carried as two bf16 terms (P_hi = bf16(P),
// P_lo = bf16(P - P_hi)) so the weights keep about 16 significant bits; a
// single bf16 P adds a weight-rounding error comparable to the bf16 output
// rounding itself.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_base, bool accumulate) {
    using S = PfSmem<D>;
    constexpr uint32_t idesc = idesc_bf16_f32(BM, D, 1);
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t vd = sw128_desc(v_base + kk * 16 * 128, S::kPanelBytes, 1024);
        tc_mma_ts(d_tmem, p_tmem + kk * 8, vd, idesc, (accumulate || kk > 0) ? 1u : 0u);
        tc_mma_ts(d_tmem, p_tmem + BN / 2 + kk * 8, vd, idesc, 1u);
    }
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    using S = PfSmem<D>;
    extern __shared__ uint8_t psmem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(psmem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = sm;
    uint8_t *sRing = sm + S::kRingOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = bars + 1 + kPfStages;
    uint64_t *s_full = bars + 1 + 2 * kPfStages;   // [2]
    uint64_t *p_ready = s_full + 2;                // [2]
    uint64_t *o_full = p_ready + 2;                // [2]
    uint64_t *fix_bar = o_full + 2;
    uint64_t *drain_bar = fix_bar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + S::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = p.num_pairs - 1 - (int)blockIdx.x;   // longest pairs first
    const int hkv = blockIdx.y, b = blockIdx.z;
    const int G = p.G, tps = BM / G;

    const int qs = __ldg(p.cu_q + b), qe = __ldg(p.cu_q + b + 1);
    const int ks0 = __ldg(p.cu_k + b), ke = __ldg(p.cu_k + b + 1);
    const int Lq = qe - qs, Lk = ke - ks0;
    if (qs < 0 || Lq < 0 || Lk < 0 || (int64_t)qe > p.total_q) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) record_error(p.err, ERR_INDEX | SRC_PREFILL);
        return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && (int64_t)Lq > (int64_t)p.num_pairs * 2 * tps)
        record_error(p.err, ERR_INDEX | SRC_PREFILL);   // longer than the stated max_seqlen_q
    const int t0A = pair * 2 * tps;
    if (t0A >= Lq) return;
    const int t0B = t0A + tps;
    const int off = Lk - Lq;
    auto tiles_for = [&](int t0) -> int {
        if (t0 >= Lq) return 0;
        const int t1 = min(t0 + tps, Lq);
        const int kend = p.causal ? min(max(t1 + off, 0), Lk) : Lk;
        return (kend + BN - 1) / BN;
    };
    const int nA = tiles_for(t0A), nB = tiles_for(t0B);
    const int n = max(nA, nB);
    const bool activeB = t0B < Lq;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kPfStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_ready[x], 128);
            mbar_init(&o_full[x], 1);
        }
        mbar_init(fix_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ================================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            if (n > 0) {
                mbar_arrive_expect_tx(q_full, (uint32_t)S::kTileBytes * (activeB ? 2u : 1u));
#pragma unroll
                for (int pn = 0; pn < S::kPanels; ++pn)
                    tma_load_3d(sQ + pn * S::kPanelBytes, &qmap, q_full, pn * 64, hkv * G, qs + t0A);
                if (activeB) {
#pragma unroll
                    for (int pn = 0; pn < S::kPanels; ++pn)
                        tma_load_3d(sQ + S::kTileBytes + pn * S::kPanelBytes, &qmap, q_full, pn * 64, hkv * G,
                                    qs + t0B);
                }
            }
        }
        const bool paged = p.block_table != nullptr;
        const int32_t *bt = paged ? p.block_table + (int64_t)b * p.bt_stride : nullptr;
        const int oob_row = paged ? (int)(p.num_blocks * p.block_size) : 0;
        int it = 0, fixc = 0;
        bool ok = true;
        for (int j = 0; j < n && ok; ++j) {
            for (int w = 0; w < 2; ++w) {   // 0: K tile, 1: V tile
                const int st = it % kPfStages;
                const uint32_t ph = (uint32_t)(it / kPfStages) & 1u;
                int got = 1;
                if (lane == 0) got = mbar_wait(&empty[st], ph ^ 1u, abort_flag, p.err, SRC_PREFILL);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) { ok = false; break; }
                uint8_t *dst = sRing + st * S::kTileBytes;
                const CUtensorMap *map = w ? &vmap : &kmap;
                const int key0 = j * BN;
                // paged V tile that runs past the sequence: rows past the end are
                // cache slots of unknown content (possibly NaN).  Land it on a
                // private barrier, zero those rows, then publish.
                const bool fix = paged && w == 1 && key0 + BN > Lk;
                uint64_t *bar = fix ? fix_bar : &full[st];
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar, (uint32_t)S::kTileBytes);
                    if (!paged) {
#pragma unroll
                        for (int pn = 0; pn < S::kPanels; ++pn)
                            tma_load_3d(dst + pn * S::kPanelBytes, map, bar, pn * 64, hkv, ks0 + key0);
                    } else {
                        const int rpb = p.rows_per_box;
                        for (int i = 0; i < BN / rpb; ++i) {
                            const int key = key0 + i * rpb;
                            int row = oob_row;   // past the end of the cache: zero-filled
                            if (key < Lk) {
                                const int blk = __ldg(bt + key / p.block_size);
                                if (blk < 0 || (int64_t)blk >= p.num_blocks)
                                    record_error(p.err, ERR_INDEX | SRC_PREFILL);
                                else
                                    row = blk * p.block_size + key % p.block_size;
                            }
#pragma unroll
                            for (int pn = 0; pn < S::kPanels; ++pn)
                                tma_load_3d(dst + pn * S::kPanelBytes + i * rpb * 128, map, bar, pn * 64, hkv, row);
                        }
                    }
                }
                if (fix) {
                    int got2 = 1;
                    if (lane == 0) got2 = mbar_wait(fix_bar, (uint32_t)fixc & 1u, abort_flag, p.err, SRC_PREFILL);
                    got2 = __shfl_sync(0xffffffffu, got2, 0);
                    ++fixc;
                    if (!got2) { ok = false; break; }
                    const int vr = Lk - key0;   // valid rows, >= 1
                    for (int idx = lane; idx < (BN - vr) * (D / 8); idx += 32) {
                        const int r = vr + idx / (D / 8), ch = idx % (D / 8);
                        *reinterpret_cast<uint4 *>(dst + (ch / 8) * S::kPanelBytes + sw128_off(r, ch % 8)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[st]);
                }
                ++it;
            }
        }
        if (lane == 0) {
            // every copy issued here lands before the CTA may exit
            for (int t = it - kPfStages < 0 ? 0 : it - kPfStages; t < it; ++t)
                mbar_wait(&full[t % kPfStages], (uint32_t)(t / kPfStages) & 1u, nullptr, p.err, SRC_PREFILL);
            if (n > 0) mbar_wait(q_full, 0, nullptr, p.err, SRC_PREFILL);
        }
    } else if (warp == 9) {
        // ================================================================ MMA issuer
        if (lane == 0 && n > 0) {
            bool ok = mbar_wait(q_full, 0, abort_flag, p.err, SRC_PREFILL);
            tc_fence_after();
            const uint32_t tS0 = tmem, tS1 = tmem + 128;
            const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + D;
            const uint32_t qA = smem_u32(sQ), qB = smem_u32(sQ + S::kTileBytes);
            const uint32_t ring = smem_u32(sRing);
            for (int j = 0; j <= n && ok; ++j) {
                const int itK = 2 * j, stK = itK % kPfStages;
                const int itV = 2 * j + 1, stV = itV % kPfStages;
                if (j < n) {
                    ok = mbar_wait(&full[stK], (uint32_t)(itK / kPfStages) & 1u, abort_flag, p.err, SRC_PREFILL);
                    if (!ok) break;
                    tc_fence_after();
                    if (j < nA) {
                        issue_qk<D>(tS0, qA, ring + stK * S::kTileBytes);
                        tc_commit(&s_full[0]);
                    }
                }
                if (j >= 1 && j - 1 < nB) {
                    const int jj = j - 1;
                    const int itP = 2 * jj + 1, stP = itP % kPfStages;
                    ok = mbar_wait(&full[stP], (uint32_t)(itP / kPfStages) & 1u, abort_flag, p.err, SRC_PREFILL) &&
                         mbar_wait(&p_ready[1], (uint32_t)jj & 1u, abort_flag, p.err, SRC_PREFILL);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv<D>(tO1, tS1, ring + stP * S::kTileBytes, jj > 0);
                    if (jj == nB - 1) tc_commit(&o_full[1]);
                    tc_commit(&empty[stP]);
                }
                if (j < n) {
                    if (j < nB) {
                        issue_qk<D>(tS1, qB, ring + stK * S::kTileBytes);
                        tc_commit(&s_full[1]);
                    }
                    tc_commit(&empty[stK]);
                    if (j < nA) {
                        ok = mbar_wait(&full[stV], (uint32_t)(itV / kPfStages) & 1u, abort_flag, p.err, SRC_PREFILL) &&
                             mbar_wait(&p_ready[0], (uint32_t)j & 1u, abort_flag, p.err, SRC_PREFILL);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv<D>(tO0, tS0, ring + stV * S::kTileBytes, j > 0);
                        if (j == nA - 1) tc_commit(&o_full[0]);
                        if (j >= nB) tc_commit(&empty[stV]);
                    }
                }
            }
            // no MMA may still run when TMEM is released
            tc_commit(drain_bar);
            mbar_wait(drain_bar, 0, nullptr, p.err, SRC_PREFILL);
        }
        __syncwarp();
    } else {
        // ================================================================ softmax (one row per thread)
        const int X = warp >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int t0 = X ? t0B : t0A;
        const int nX = X ? nB : nA;
        const int tok = t0 + r / G;
        const int head = hkv * G + r % G;
        const bool row_valid = tok < Lq;
        // last key this row may see (negative: none)
        const int lim = p.causal ? min(tok + off, Lk - 1) : Lk - 1;
        const uint32_t tS = tmem + (uint32_t)(X * 128) + lane_off;
        const uint32_t tO = tmem + 256u + (uint32_t)(X * D) + lane_off;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY;   // reference max (log2 units) used for P
        float l = 0.f;             // proxy denominator d'
        bool ok = true;
        for (int j = 0; j < nX; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[X], (uint32_t)j & 1u, abort_flag, p.err, SRC_PREFILL));
            if (!ok) break;
            tc_fence_after();
            float s[BN];
            tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
            tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
            tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
            tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
            tc_wait_ld();
            const int key0 = j * BN;
            if (key0 + BN - 1 > lim) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (key0 + c > lim) s[c] = -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; ++c) mx = fmaxf(mx, s[c]);
            const float m_new = fmaxf(m_ref, mx * sl2);
            const bool need = m_new > m_ref + 8.0f;
            float alpha = 1.f;
            if (need) {
                alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
                m_ref = m_new;
            }
            l *= alpha;
            const float nref = (m_ref == -INFINITY) ? 0.f : -m_ref;
            // P = 2^(s*scale*log2e - m_ref) as P_hi (columns 0-63 of S) and
            // P_lo = P - P_hi (columns 64-127), both bf16
#pragma unroll
            for (int c4 = 0; c4 < BN / 32; ++c4) {
                uint32_t pk[16], pl[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float x0 = ex2(fmaf(s[c4 * 32 + 2 * i], sl2, nref));
                    const float x1 = ex2(fmaf(s[c4 * 32 + 2 * i + 1], sl2, nref));
                    l += x0 + x1;
                    const uint32_t h = pack_bf16x2(x0, x1);
                    pk[i] = h;
                    pl[i] = pack_bf16x2(x0 - __uint_as_float(h << 16), x1 - __uint_as_float(h & 0xFFFF0000u));
                }
                tmem_st16(tS + (uint32_t)(c4 * 16), pk);
                tmem_st16(tS + (uint32_t)(BN / 2 + c4 * 16), pl);
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
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&p_ready[X]);
        }
        // ---------------------------------------------------------------- epilogue
        if (ok && nX > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&o_full[X], 0, abort_flag, p.err, SRC_PREFILL));
            tc_fence_after();
        }
        if (ok) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = p.out + (int64_t)(qs + (row_valid ? tok : 0)) * p.out_row_stride + (int64_t)head * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (nX > 0) {
                    tmem_ld32(tO + (uint32_t)(c * 32), o);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (row_valid) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            if (row_valid && p.lse)
                p.lse[(int64_t)head * p.total_q + qs + tok] =
                    l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
static cudaError_t launch_prefill_t(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                    const PrefillParams &p, cudaStream_t stream) {
    using S = PfSmem<D>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(attn_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    dim3 grid(p.num_pairs, p.Hkv, p.batch);
    attn_prefill_kernel<D><<<grid, kPfThreads, S::kBytes, stream>>>(qmap, kmap, vmap, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const PrefillParams &p, int head_dim, cudaStream_t stream) {
    if (head_dim == 128) return launch_prefill_t<128>(qmap, kmap, vmap, p, stream);
    return launch_prefill_t<64>(qmap, kmap, vmap, p, stream);
}

}  // namespace attn
