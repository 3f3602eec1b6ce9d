/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU statement of what the attention path computes.
 * It is the yardstick the CUDA kernels are compared against.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it;
 * the product library never links, loads or calls anything in this file, and
 * this file includes nothing from the product.
 *
 * Source of every definition here: the article
 *   "从零实现 vLLM (1.3)：如何加速 Attention 计算" (blog.xiaohansong.com),
 * cited below by its section headings.
 *
 * Inputs that are bf16 on the GPU arrive here as their raw 16-bit patterns and
 * are widened exactly (bf16 -> f32 -> f64 is exact).  All arithmetic is f64.
 *
 * Functions:
 *   oracle_softmax_naive_f32/f64  -- e^x / sum e^x, no max shift
 *                                    (section "安全 Softmax"的提出: the overflow it shows)
 *   oracle_softmax_safe           -- 3-pass safe softmax (same section)
 *   oracle_softmax_online         -- 2-pass online softmax with the d' recurrence
 *                                    (section 减少遍历次数的"在线 Softmax")
 *   oracle_softmax_rows           -- the safe softmax of every row of a matrix
 *                                    (section "安全 Softmax"), OpenMP over rows
 *   oracle_attn_tiled_row         -- 1-pass m, d', o' recurrence over key blocks
 *                                    (sections "FlashAttention 的最终实现" and
 *                                    "计算流程（1-Pass 算法与分块）")
 *   oracle_attn_varlen            -- three-step attention X = scale*QK^T, A = softmax(X),
 *                                    O = AV per query row (sections "标准实现方法",
 *                                    "图书馆例子跟实际矩阵计算的联系"), over varlen
 *                                    cu_seqlens packing and an optional paged cache
 *                                    (section "Prefill")
 *   oracle_decode_paged           -- one query token per sequence through the paged
 *                                    cache (section "Decode")
 *   oracle_store_kvcache          -- the slot_mapping scatter (section "Prefill")
 *
 * Readings where the article is silent (each is also listed in the design notes):
 *   - causal with Lq < Lk is bottom-right aligned: query i sees key j iff
 *     j <= Lk - Lq + i;
 *   - a row with no visible key outputs 0 and lse = -inf;
 *   - initial state of the recurrence m = -inf, d' = 0, o' = 0, and the
 *     rescale factor is taken as 0 while m is still -inf;
 *   - GQA: query head h reads KV head h / (Hq / Hkv);
 *   - slot_mapping holds flat slots block_id*block_size + offset into the
 *     cache viewed as [num_blocks*block_size, Hkv, D]; a negative slot skips
 *     the token.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Softmax variants (section "安全 Softmax"的提出 and the online section) */
/* ------------------------------------------------------------------ */

/* e^{x_i} / sum_j e^{x_j}, evaluated in float32 with no shift. */
void oracle_softmax_naive_f32(const float *x, int n, float *y)
{
    float sum = 0.0f;
    for (int i = 0; i < n; ++i) {
        y[i] = expf(x[i]);
        sum += y[i];
    }
    for (int i = 0; i < n; ++i) y[i] = y[i] / sum;
}

/* The same in float64. */
void oracle_softmax_naive_f64(const double *x, int n, double *y)
{
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
        y[i] = exp(x[i]);
        sum += y[i];
    }
    for (int i = 0; i < n; ++i) y[i] = y[i] / sum;
}

/* Safe softmax, three passes: m = max_j x_j; d = sum_j e^{x_j - m};
 * y_i = e^{x_i - m} / d. */
void oracle_softmax_safe(const double *x, int n, double *y)
{
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (x[i] > m) m = x[i];          /* pass 1 */
    double d = 0.0;
    for (int i = 0; i < n; ++i) d += exp(x[i] - m);               /* pass 2 */
    for (int i = 0; i < n; ++i) y[i] = exp(x[i] - m) / d;         /* pass 3 */
}

/* Row-wise softmax of a [rows, cols] matrix (row stride cols): every row
 * goes through oracle_softmax_safe, the plain definition. */
void oracle_softmax_rows(const double *x, int64_t rows, int cols, double *y, int nthreads)
{
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; ++r) oracle_softmax_safe(x + r * (int64_t)cols, cols, y + r * (int64_t)cols);
}

/* Online softmax, two passes.  Pass 1 runs the running maximum
 * m_i = max(m_{i-1}, x_i) together with the proxy denominator
 * d'_i = d'_{i-1} * e^{m_{i-1} - m_i} + e^{x_i - m_i}; pass 2 normalises with
 * the final m_N and d'_N.  m_trace / d_trace (nullable) receive m_i and d'_i. */
void oracle_softmax_online(const double *x, int n, double *y,
                           double *m_trace, double *d_trace)
{
    double m = -INFINITY, d = 0.0;
    for (int i = 0; i < n; ++i) {
        double m_new = x[i] > m ? x[i] : m;
        double carry = (m == -INFINITY) ? 0.0 : d * exp(m - m_new);
        d = carry + exp(x[i] - m_new);
        m = m_new;
        if (m_trace) m_trace[i] = m;
        if (d_trace) d_trace[i] = d;
    }
    for (int i = 0; i < n; ++i) y[i] = exp(x[i] - m) / d;
}

/* ------------------------------------------------------------------ */
/* 1-pass recurrence with key blocks (FlashAttention sections)          */
/* ------------------------------------------------------------------ */

/* One query row q[D] against keys K[Lk, D] and values V[Lk, D] (row-major
 * float64).  The keys are walked in blocks of `block` rows; inside a block the
 * state update is the article's per-key recurrence
 *     m_i  = max(m_{i-1}, x_i)
 *     d'_i = d'_{i-1} e^{m_{i-1}-m_i} + e^{x_i-m_i}
 *     o'_i = o'_{i-1} d'_{i-1} e^{m_{i-1}-m_i} / d'_i + e^{x_i-m_i} / d'_i * V[i,:]
 * with x_i = scale * q . K[i].  Keys with visible[i] == 0 (nullable: all
 * visible) are skipped.  Blocks only change the order in which whole blocks of
 * logits are formed before their keys are folded in, which is the point of
 * the tiling: the result must not depend on `block`.
 * Outputs o[D], *m_out and *d_out (the final m and d'). */
void oracle_attn_tiled_row(const double *q, const double *K, const double *V,
                           const unsigned char *visible, int Lk, int D,
                           double scale, int block, double *o,
                           double *m_out, double *d_out)
{
    double m = -INFINITY, d = 0.0;
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    if (block < 1) block = 1;
    double *x = (double *)malloc(sizeof(double) * (size_t)block);
    for (int j0 = 0; j0 < Lk; j0 += block) {
        int nb = Lk - j0 < block ? Lk - j0 : block;
        /* load the block and form its logits */
        for (int t = 0; t < nb; ++t) {
            const double *kr = K + (size_t)(j0 + t) * D;
            double s = 0.0;
            for (int c = 0; c < D; ++c) s += q[c] * kr[c];
            x[t] = scale * s;
        }
        /* fold the block's keys into (m, d', o') one at a time */
        for (int t = 0; t < nb; ++t) {
            int j = j0 + t;
            if (visible && !visible[j]) continue;
            double m_new = x[t] > m ? x[t] : m;
            double keep = (m == -INFINITY) ? 0.0 : d * exp(m - m_new); /* d'_{i-1} e^{m_{i-1}-m_i} */
            double e = exp(x[t] - m_new);
            double d_new = keep + e;
            const double *vr = V + (size_t)j * D;
            for (int c = 0; c < D; ++c) o[c] = o[c] * keep / d_new + e / d_new * vr[c];
            m = m_new;
            d = d_new;
        }
    }
    free(x);
    if (m_out) *m_out = m;
    if (d_out) *d_out = d;
}

/* ------------------------------------------------------------------ */
/* Three-step attention over varlen / paged inputs                       */
/* ------------------------------------------------------------------ */

/* Sequence b such that cu[b] <= t < cu[b+1]; -1 if none. */
static int find_seq(const int32_t *cu, int batch, int64_t t)
{
    int lo = 0, hi = batch - 1, ans = -1;
    while (lo <= hi) {
        int mid = (lo + hi) / 2;
        if ((int64_t)cu[mid] <= t) { ans = mid; lo = mid + 1; } else hi = mid - 1;
    }
    if (ans >= 0 && t >= (int64_t)cu[ans + 1]) {
        /* empty sequences share offsets: step forward to the one that holds t */
        while (ans < batch && t >= (int64_t)cu[ans + 1]) ++ans;
        if (ans >= batch) return -1;
    }
    return ans;
}

/* Row index into the K (or V) storage of logical key j of sequence b:
 * contiguous -> cu_k[b] + j; paged -> block_table[b][j / bs] * bs + j % bs. */
static int64_t key_row(int b, int j, const int32_t *cu_k,
                       const int32_t *block_table, int bt_stride, int block_size)
{
    if (!block_table) return (int64_t)cu_k[b] + j;
    int32_t blk = block_table[(int64_t)b * bt_stride + j / block_size];
    return (int64_t)blk * block_size + (j % block_size);
}

/* One output row by the three steps, with X materialised for the row.
 *   x[j] = scale * q . K_j                         (step 1, X = QK^T scaled)
 *   x[j] = -inf where the key is not visible        (mask)
 *   a = safe softmax(x)                             (step 2)
 *   o = sum_j a[j] V_j                              (step 3)
 * Returns 0, or -1 on an index outside the stated storage. */
static int attn_one_row(const uint16_t *qrow, const uint16_t *k, const uint16_t *v,
                        int b, int i, int Lq, int Lk, int hk, int Hkv, int D,
                        double scale, int causal, const int32_t *cu_k,
                        const int32_t *block_table, int bt_stride, int block_size,
                        int64_t k_rows, int64_t k_stride, int64_t v_stride,
                        double *xbuf, double *qbuf, double *o, double *lse)
{
    for (int c = 0; c < D; ++c) qbuf[c] = bf16_to_f64(qrow[c]);
    int n_vis = 0;
    double m = -INFINITY;
    for (int j = 0; j < Lk; ++j) {
        int vis = !causal || ((int64_t)j <= (int64_t)Lk - Lq + i);
        if (!vis) { xbuf[j] = -INFINITY; continue; }
        int64_t r = key_row(b, j, cu_k, block_table, bt_stride, block_size);
        if (r < 0 || r >= k_rows) return -1;
        const uint16_t *kr = k + r * k_stride + (int64_t)hk * D;
        double s = 0.0;
        for (int c = 0; c < D; ++c) s += qbuf[c] * bf16_to_f64(kr[c]);
        xbuf[j] = scale * s;
        if (xbuf[j] > m) m = xbuf[j];
        ++n_vis;
    }
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    if (n_vis == 0) { *lse = -INFINITY; return 0; }
    double den = 0.0;
    for (int j = 0; j < Lk; ++j) if (xbuf[j] != -INFINITY) den += exp(xbuf[j] - m);
    for (int j = 0; j < Lk; ++j) {
        if (xbuf[j] == -INFINITY) continue;
        double a = exp(xbuf[j] - m) / den;
        int64_t r = key_row(b, j, cu_k, block_table, bt_stride, block_size);
        const uint16_t *vr = v + r * v_stride + (int64_t)hk * D;
        for (int c = 0; c < D; ++c) o[c] += a * bf16_to_f64(vr[c]);
    }
    *lse = m + log(den);
    (void)Hkv;
    return 0;
}

/*
 * Varlen attention, three-step definition per query row.
 *   q      [total_q, Hq, D]  bf16 bits, token row stride q_stride (elements)
 *   k, v   contiguous: [total_k, Hkv, D], row strides k_stride / v_stride;
 *          paged (block_table != NULL): caches [num_blocks*block_size, Hkv, D]
 *   cu_q, cu_k  [batch+1] prefix offsets (cu_k counts logical keys when paged)
 *   rows   nullable list of row ids (token*Hq + head); NULL = every row
 *   out    [nrows, D] float64 (row order of `rows`, or token-major/head-minor)
 *   lse    [nrows] float64, natural-log log-sum-exp of the scaled logits
 * Returns 0 on success, -1 on an argument or index outside its storage.
 */
int oracle_attn_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *cu_q, const int32_t *cu_k, int batch,
                       int Hq, int Hkv, int D, double scale, int causal,
                       const int32_t *block_table, int bt_stride, int block_size,
                       int64_t num_blocks, int64_t q_stride, int64_t k_stride,
                       int64_t v_stride, const int64_t *rows, int64_t nrows,
                       double *out, double *lse, int nthreads)
{
    if (batch <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    int64_t total_q = cu_q[batch];
    int64_t k_rows = block_table ? num_blocks * (int64_t)block_size : (int64_t)cu_k[batch];
    int max_lk = 0;
    for (int b = 0; b < batch; ++b) {
        int lk = cu_k[b + 1] - cu_k[b];
        if (lk > max_lk) max_lk = lk;
    }
    int64_t n = rows ? nrows : total_q * Hq;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel reduction(| : err)
    {
        double *xbuf = (double *)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
        double *qbuf = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            int64_t id = rows ? rows[r] : r;
            int64_t t = id / Hq;
            int h = (int)(id % Hq);
            if (t < 0 || t >= total_q) { err |= 1; continue; }
            int b = find_seq(cu_q, batch, t);
            if (b < 0) { err |= 1; continue; }
            int i = (int)(t - cu_q[b]);
            int Lq = cu_q[b + 1] - cu_q[b];
            int Lk = cu_k[b + 1] - cu_k[b];
            int hk = h / G;
            if (attn_one_row(q + t * q_stride + (int64_t)h * D, k, v, b, i, Lq, Lk, hk, Hkv, D,
                             scale, causal, cu_k, block_table, bt_stride, block_size,
                             k_rows, k_stride, v_stride, xbuf, qbuf, out + r * D, lse + r))
                err |= 1;
        }
        free(xbuf);
        free(qbuf);
    }
    return err ? -1 : 0;
}

/*
 * Single-token decode through the paged cache (section "Decode"):
 *   q       [batch, Hq, D] bf16 bits (row stride q_stride elements per sequence)
 *   caches  [num_blocks*block_size, Hkv, D]
 *   cache_seqlens [batch]: keys 0..L_b-1 of sequence b, all visible to its one
 *           query (bottom-right causal with Lq = 1 sees every key)
 *   out     [batch, Hq, D] float64; lse [batch, Hq]
 */
int oracle_decode_paged(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *cache_seqlens, const int32_t *block_table,
                        int bt_stride, int batch, int Hq, int Hkv, int D, int block_size,
                        int64_t num_blocks, double scale, int64_t q_stride,
                        double *out, double *lse, int nthreads)
{
    if (batch <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    int max_lk = 0;
    for (int b = 0; b < batch; ++b) if (cache_seqlens[b] > max_lk) max_lk = cache_seqlens[b];
    int64_t row_stride = (int64_t)Hkv * D;
    int64_t k_rows = num_blocks * (int64_t)block_size;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel reduction(| : err)
    {
        double *xbuf = (double *)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
        double *qbuf = (double *)malloc(sizeof(double) * (size_t)D);
        /* cu_k is not used on the paged path; key_row only reads block_table */
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < (int64_t)batch * Hq; ++r) {
            int b = (int)(r / Hq), h = (int)(r % Hq);
            int Lk = cache_seqlens[b];
            if (Lk < 0) { err |= 1; continue; }
            if (attn_one_row(q + (int64_t)b * q_stride + (int64_t)h * D, k_cache, v_cache, b, 0,
                             1, Lk, h / G, Hkv, D, scale, 1, NULL, block_table, bt_stride,
                             block_size, k_rows, row_stride, row_stride, xbuf, qbuf,
                             out + r * D, lse + r))
                err |= 1;
        }
        free(xbuf);
        free(qbuf);
    }
    return err ? -1 : 0;
}

/*
 * store_kvcache (section "Prefill"): for every new token t with
 * slot = slot_mapping[t] >= 0, copy its Hkv*D elements of k into
 * k_cache[slot] and of v into v_cache[slot].  Plain element copy loop.
 * Returns -1 if a slot is >= num_slots (nothing is written for that token).
 */
int oracle_store_kvcache(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                         uint16_t *v_cache, const int64_t *slot_mapping, int64_t num_tokens,
                         int Hkv, int D, int64_t k_stride, int64_t v_stride, int64_t num_slots)
{
    int err = 0;
    int64_t row = (int64_t)Hkv * D;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { err = 1; continue; }
        for (int64_t e = 0; e < row; ++e) {
            k_cache[slot * row + e] = k[t * k_stride + e];
            v_cache[slot * row + e] = v[t * v_stride + e];
        }
    }
    return err ? -1 : 0;
}
