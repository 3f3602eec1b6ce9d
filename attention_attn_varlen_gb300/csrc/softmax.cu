// softmax.cu -- softmax of every row of a matrix with the online two-pass
// algorithm of "从零实现 vLLM (1.3)：如何加速 Attention 计算", section
// 减少遍历次数的“在线 Softmax”: pass 1 keeps the running maximum m and the proxy
// denominator d' = d' * e^(m_old - m_new) + e^(x - m_new); pass 2 writes
// y = e^(x - m) / d'.  The update runs on blocks of elements, the same
// recurrence in exact arithmetic: per 16-byte vector (its max first, then its
// terms) in the warp and two-pass kernels, and over all of a thread's elements
// at once (their max first, then one sum) where the row sits in registers.
// Partial (m, d') states of threads merge exactly:
//   m = max(m1, m2),  d' = d1 e^(m1 - m) + d2 e^(m2 - m).
//
// HBM-bound; every path below reads the matrix once and writes it once except
// the last.  Rows of up to 1024 fp32 / 2048 bf16 elements: one warp per row,
// the row held in registers.  Up to 16 KB: one CTA per row, rows streamed into a
// shared-memory ring by bulk copies.  Up to 64 KB: one CTA per row, the row held
// in registers across the CTA's threads; up to 512 KB: a thread-block cluster
// per row, each CTA holding a slice and the CTAs' (m, d') pairs exchanged
// through distributed shared memory.  Longer rows (or rows that are not 16-byte
// aligned): one CTA per row, pass 2 re-reads the row, which the CTAs in flight
// keep in L2.
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "kernels.h"

namespace attn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// error-word source bit of this file's kernels (beside SRC_STORE ... SRC_PREFILL)
constexpr uint32_t SRC_SOFTMAX = 1u << 12;

// thread-block cluster: this CTA's rank and the cluster's size (1 without a cluster)
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// store v into the shared-memory word of CTA `rank` of the cluster that sits at
// the address `local` has in this CTA
__device__ __forceinline__ void st_cluster_f32(const void *local, uint32_t rank, float v) {
    uint32_t a = smem_u32(local), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}
// every thread of every CTA of the cluster: stores before it are visible after it
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// untiled bulk copy global -> shared (16-byte aligned addresses, bytes a
// multiple of 16), completion on an mbarrier
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 16-byte vector of T as floats
template <typename T>
struct Vec;

template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const float *p, float (&f)[4]) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    __device__ static void from_bits(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ static void store(float *p, const float (&f)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
    __device__ static float one(const float *p) { return *p; }
    __device__ static void put(float *p, float f) { *p = f; }
    // the first `valid` (< 4) elements at p as raw bits; the rest are left 0
    __device__ static uint4 bits_partial(const float *p, int valid) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (valid > 0) v.x = __float_as_uint(p[0]);
        if (valid > 1) v.y = __float_as_uint(p[1]);
        if (valid > 2) v.z = __float_as_uint(p[2]);
        return v;
    }
};

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16 *p, float (&f)[8]) {
        from_bits(*reinterpret_cast<const uint4 *>(p), f);
    }
    __device__ static void from_bits(const uint4 &v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&f)[8]) {
        uint4 v;
        v.x = pack_bf16x2(f[0], f[1]);
        v.y = pack_bf16x2(f[2], f[3]);
        v.z = pack_bf16x2(f[4], f[5]);
        v.w = pack_bf16x2(f[6], f[7]);
        *reinterpret_cast<uint4 *>(p) = v;
    }
    __device__ static float one(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ static void put(__nv_bfloat16 *p, float f) { *p = __float2bfloat16_rn(f); }
    // the first `valid` (< 8) elements at p as raw bits; the rest are left 0
    __device__ static uint4 bits_partial(const __nv_bfloat16 *p, int valid) {
        const unsigned short *h = reinterpret_cast<const unsigned short *>(p);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 7; ++e)
            if (e < valid) w[e >> 1] |= (uint32_t)h[e] << ((e & 1) * 16);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// running state of the online recurrence (m in log2 units, d')
struct Online {
    float m = -INFINITY, d = 0.f;
    // fold k values (already scaled by log2 e)
    template <int K>
    __device__ void add(const float (&x)[K], int valid) {
        float vm = -INFINITY;
#pragma unroll
        for (int i = 0; i < K; ++i)
            if (i < valid) vm = fmaxf(vm, x[i]);
        if (vm == -INFINITY) return;
        if (vm > m) {
            d = (m == -INFINITY) ? 0.f : d * ex2(m - vm);
            m = vm;
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i)
            if (i < valid) s += ex2(x[i] - m);
        d += s;
    }
    __device__ void merge(float m2, float d2) {
        if (m2 == -INFINITY) return;
        if (m == -INFINITY) {
            m = m2;
            d = d2;
            return;
        }
        const float mn = fmaxf(m, m2);
        d = d * ex2(m - mn) + d2 * ex2(m2 - mn);
        m = mn;
    }
    __device__ void warp_merge() {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float d2 = __shfl_xor_sync(0xffffffffu, d, o);
            merge(m2, d2);
        }
    }
};

// ---------------------------------------------------------------------------
// one warp per row, NV vectors per lane held in registers (VEC: 16-byte
// accesses, and the warp's next row is loaded while it works on the current
// one; otherwise one element at a time, lane-strided)
// ---------------------------------------------------------------------------
template <typename T, int NV, bool VEC>
__global__ void __launch_bounds__(256) softmax_rows_warp_kernel(const T *x, T *y, int64_t rows, int cols,
                                                                int64_t xs, int64_t ys) {
    constexpr int N = VEC ? Vec<T>::N : 1;
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    uint4 next[NV];   // VEC: the whole 16-byte vectors of row r (then of the row after it)
    auto fetch = [&](int64_t row) {
        if constexpr (VEC) {
            const T *xr = x + row * xs;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int c0 = (i * 32 + lane) * N;
                if (c0 + N <= cols) next[i] = *reinterpret_cast<const uint4 *>(xr + c0);
            }
        }
    };
    if (r < rows) fetch(r);
    for (; r < rows; r += nw) {
        const T *xr = x + r * xs;
        T *yr = y + r * ys;
        uint4 cur[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) cur[i] = next[i];
        if (r + nw < rows) fetch(r + nw);
        float v[NV][N];
        Online st;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c0 = (i * 32 + lane) * N;
            int valid = cols - c0;
            valid = valid < 0 ? 0 : (valid > N ? N : valid);
            bool whole = false;
            if constexpr (VEC) {
                if (valid == N) {
                    Vec<T>::from_bits(cur[i], v[i]);
#pragma unroll
                    for (int e = 0; e < N; ++e) v[i][e] *= kLog2e;
                    whole = true;
                }
            }
            if (!whole) {
#pragma unroll
                for (int e = 0; e < N; ++e) v[i][e] = e < valid ? Vec<T>::one(xr + c0 + e) * kLog2e : -INFINITY;
            }
            st.add<N>(v[i], valid);
        }
        st.warp_merge();
        const float inv = 1.f / st.d;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c0 = (i * 32 + lane) * N;
            int valid = cols - c0;
            valid = valid < 0 ? 0 : (valid > N ? N : valid);
            float f[N];
#pragma unroll
            for (int e = 0; e < N; ++e) f[e] = ex2(v[i][e] - st.m) * inv;
            bool whole = false;
            if constexpr (VEC) {
                if (valid == N) {
                    Vec<T>::store(yr + c0, f);
                    whole = true;
                }
            }
            if (!whole) {
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (e < valid) Vec<T>::put(yr + c0 + e, f[e]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// one CTA per row, rows streamed through shared memory: thread 0 keeps the
// next `stages` rows of the CTA in flight with bulk copies (one per row, its
// whole 16-byte vectors; the few elements past the last one are read
// directly), so the bytes in flight are bounded by shared memory, not by
// registers.  Each thread copies its (at most KV) vectors of the landed row into
// registers, takes their maximum, sums e^(x - m) against it, and after the
// CTA's merge writes the normalised vectors from the same registers; a stage
// is refilled once every thread has passed the row's last barrier.  Every mbarrier wait is bounded: on a timeout the kernel records it
// in the error word, lets its copies in flight land (again bounded) and stops.
// ---------------------------------------------------------------------------
constexpr int kSmemMaxStages = 8;
constexpr int kSmemThreads = 128;
constexpr int kSmemVecs = 8;   // 16-byte vectors per thread: rows of up to 128 x 8 x 16 B = 16 KB

template <typename T, int NT, int KV>
__global__ void __launch_bounds__(NT, 2048 / NT / 2) softmax_rows_smem_kernel(const T *x, T *y, int64_t rows, int cols,
                                                               int64_t xs, int64_t ys, int stages, uint32_t slot,
                                                               uint32_t *err) {
    constexpr int N = Vec<T>::N;
    constexpr int NWARP = NT / 32;
    extern __shared__ __align__(128) uint8_t stage_mem[];
    __shared__ uint64_t full[kSmemMaxStages];
    __shared__ float sm_m[2][NWARP], sm_d[2][NWARP];
    __shared__ int abort_flag;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nwhole = cols / N;                        // 16-byte vectors in the bulk copy
    const int nvec = (cols + N - 1) / N;
    const uint32_t bulk = (uint32_t)nwhole * 16u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int s, int64_t row) {
        mbar_arrive_expect_tx(&full[s], bulk);
        bulk_load(stage_mem + (size_t)s * slot, x + row * xs, bulk, &full[s]);
    };
    if (threadIdx.x == 0)
        for (int s = 0; s < stages; ++s) {
            const int64_t row = blockIdx.x + (int64_t)s * gridDim.x;
            if (row < rows) issue(s, row);
        }
    int64_t it = 0;
    bool ok = true;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, ++it) {
        const int s = (int)(it % stages);
        const int par = (int)(it & 1);
        ok = mbar_wait(&full[s], (uint32_t)((it / stages) & 1), &abort_flag, err, SRC_SOFTMAX);
        const uint4 *sv = reinterpret_cast<const uint4 *>(stage_mem + (size_t)s * slot);
        const T *xr = x + r * xs;
        T *yr = y + r * ys;
        // the thread's vectors tid, tid + NT, ... (at most KV) into registers, as
        // floats when they fit in 32 registers (unpacked once), else as raw bits;
        // the partial vector past the bulk copy comes from global memory
        constexpr bool kAsFloat = KV * N <= 32;
        uint4 v[kAsFloat ? 1 : KV];
        float fv[kAsFloat ? KV : 1][N];
        auto elems = [&](int k, float (&f)[N]) {
            if constexpr (kAsFloat) {
#pragma unroll
                for (int e = 0; e < N; ++e) f[e] = fv[k][e];
            } else {
                Vec<T>::from_bits(v[k], f);
            }
        };
        float mx = -INFINITY;
        if (ok) {
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int i = (int)threadIdx.x + k * NT;
                uint4 bits = make_uint4(0u, 0u, 0u, 0u);
                if (i < nwhole)
                    bits = sv[i];
                else if (i < nvec)
                    bits = Vec<T>::bits_partial(xr + i * N, cols - i * N);
                const int valid = cols - i * N;
                float f[N];
                Vec<T>::from_bits(bits, f);
                if constexpr (kAsFloat) {
#pragma unroll
                    for (int e = 0; e < N; ++e) fv[k][e] = f[e];
                } else {
                    v[k] = bits;
                }
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (e < valid) mx = fmaxf(mx, f[e]);
            }
        }
        Online st;
        if (mx != -INFINITY) {
            st.m = mx * kLog2e;
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int valid = cols - ((int)threadIdx.x + k * NT) * N;
                float f[N];
                elems(k, f);
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (e < valid) st.d += ex2(fmaf(f[e], kLog2e, -st.m));
            }
        }
        st.warp_merge();
        if (lane == 0) {
            sm_m[par][wid] = st.m;
            sm_d[par][wid] = st.d;
        }
        // every thread agrees: all waits succeeded, or all stop here
        if (!__syncthreads_and(ok)) {
            ok = false;
            break;
        }
        Online t;
        if (lane < NWARP) {
            t.m = sm_m[par][lane];
            t.d = sm_d[par][lane];
        }
        t.warp_merge();
        const float m = t.m, inv = 1.f / t.d;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int i = (int)threadIdx.x + k * NT;
            if (i >= nvec) continue;
            float f[N];
            elems(k, f);
#pragma unroll
            for (int e = 0; e < N; ++e) f[e] = ex2(fmaf(f[e], kLog2e, -m)) * inv;
            if (i < nwhole) {
                Vec<T>::store(yr + i * N, f);
            } else {
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (i * N + e < cols) Vec<T>::put(yr + i * N + e, f[e]);
            }
        }
        __syncthreads();   // stage s has been read by every thread
        if (threadIdx.x == 0) {
            const int64_t nxt = r + (int64_t)stages * gridDim.x;
            if (nxt < rows) issue(s, nxt);
        }
    }
    if (!ok && threadIdx.x == 0) {
        // the copies issued for iterations it .. it + stages - 1 may still be in flight
        for (int j = 0; j < stages; ++j) {
            const int64_t jt = it + j;
            if (blockIdx.x + jt * gridDim.x < rows)
                mbar_wait(&full[jt % stages], (uint32_t)((jt / stages) & 1), nullptr, err, SRC_SOFTMAX);
        }
    }
}

// ---------------------------------------------------------------------------
// one CTA (or one cluster of CTAs) per row, the row held in registers.  CTA c of
// a cluster of C owns the row's slice of NT*KV 16-byte vectors starting at
// vector c*NT*KV; thread t holds vectors t, t + NT, ..., t + (KV-1) NT of the
// slice (coalesced loads), so pass 2 runs from registers and the row is read
// from HBM once.  Each CTA loads its next row while the current one is reduced
// and written.  A thread's elements are all in registers, so it takes their
// maximum first and sums e^(x - m) against it once; the (m, d') pairs of threads,
// warps, CTAs and cluster ranks then merge with the online rule.  Every thread
// writes only the vectors it read, so y may alias x.
// ---------------------------------------------------------------------------
constexpr int kMaxCluster = 8;

template <typename T, int KV, int NT>
__global__ void __launch_bounds__(NT) softmax_rows_cta_reg_kernel(const T *x, T *y, int64_t rows, int cols,
                                                                  int64_t xs, int64_t ys) {
    constexpr int N = Vec<T>::N;
    constexpr int NWARP = NT / 32;
    // (m, d') of each warp, and of each CTA of the cluster; two copies, by row
    // parity, so a row needs one barrier of each kind: a copy is rewritten only
    // after the next row's barrier, which every reader reaches after reading it
    __shared__ float sm_m[2][NWARP], sm_d[2][NWARP];
    __shared__ float cl_m[2][kMaxCluster], cl_d[2][kMaxCluster];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const uint32_t crank = cluster_ctarank(), csize = cluster_nctarank();
    const int base = (int)crank * NT * KV * N;
    uint4 next[KV];
    auto fetch = [&](int64_t row) {
        const T *xr = x + row * xs;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int c0 = base + (k * NT + (int)threadIdx.x) * N;
            if (c0 + N <= cols)
                next[k] = *reinterpret_cast<const uint4 *>(xr + c0);
            else if (c0 < cols)
                next[k] = Vec<T>::bits_partial(xr + c0, cols - c0);
            else
                next[k] = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // every CTA of a cluster walks the same rows, so all reach each cluster barrier
    const int64_t rstep = gridDim.x / csize;
    int64_t r = blockIdx.x / csize;
    if (r < rows) fetch(r);
    for (int par = 0; r < rows; r += rstep, par ^= 1) {
        uint4 cur[KV];
#pragma unroll
        for (int k = 0; k < KV; ++k) cur[k] = next[k];
        if (r + rstep < rows) fetch(r + rstep);
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int valid = cols - (base + (k * NT + (int)threadIdx.x) * N);
            float f[N];
            Vec<T>::from_bits(cur[k], f);
#pragma unroll
            for (int e = 0; e < N; ++e)
                if (e < valid) mx = fmaxf(mx, f[e]);
        }
        Online st;
        if (mx != -INFINITY) {
            st.m = mx * kLog2e;
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int valid = cols - (base + (k * NT + (int)threadIdx.x) * N);
                float f[N];
                Vec<T>::from_bits(cur[k], f);
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (e < valid) st.d += ex2(fmaf(f[e], kLog2e, -st.m));
            }
        }
        st.warp_merge();
        if (lane == 0) {
            sm_m[par][wid] = st.m;
            sm_d[par][wid] = st.d;
        }
        __syncthreads();
        Online t;
        if (lane < NWARP) {
            t.m = sm_m[par][lane];
            t.d = sm_d[par][lane];
        }
        t.warp_merge();
        if (csize > 1) {
            if (threadIdx.x < csize) {
                st_cluster_f32(&cl_m[par][crank], threadIdx.x, t.m);
                st_cluster_f32(&cl_d[par][crank], threadIdx.x, t.d);
            }
            cluster_sync();
            t = Online();
            if (lane < (int)csize) {
                t.m = cl_m[par][lane];
                t.d = cl_d[par][lane];
            }
            t.warp_merge();
        }
        const float m = t.m, inv = 1.f / t.d;
        T *yr = y + r * ys;
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int c0 = base + (k * NT + (int)threadIdx.x) * N;
            if (c0 >= cols) continue;
            float f[N];
            Vec<T>::from_bits(cur[k], f);
#pragma unroll
            for (int e = 0; e < N; ++e) f[e] = ex2(fmaf(f[e], kLog2e, -m)) * inv;
            if (c0 + N <= cols) {
                Vec<T>::store(yr + c0, f);
            } else {
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (c0 + e < cols) Vec<T>::put(yr + c0 + e, f[e]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// one CTA per row, two passes over the row (rows past 512 KB, or not 16-byte
// aligned)
// ---------------------------------------------------------------------------
// NT threads per CTA: 256 for rows of up to 32 KB (more rows in flight per SM),
// 512 beyond
template <typename T, bool VEC, int NT>
__global__ void __launch_bounds__(NT) softmax_rows_cta_kernel(const T *x, T *y, int64_t rows, int cols,
                                                                       int64_t xs, int64_t ys) {
    constexpr int N = VEC ? Vec<T>::N : 1;
    __shared__ float sm_m[NT / 32], sm_d[NT / 32];
    __shared__ float fin[2];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nvec = (cols + N - 1) / N;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const T *xr = x + r * xs;
        T *yr = y + r * ys;
        Online st;
        for (int i = threadIdx.x; i < nvec; i += NT) {
            const int c0 = i * N;
            const int valid = min(N, cols - c0);
            float f[N];
            bool whole = false;
            if constexpr (VEC) {
                if (valid == N) {
                    Vec<T>::load(xr + c0, f);
#pragma unroll
                    for (int e = 0; e < N; ++e) f[e] *= kLog2e;
                    whole = true;
                }
            }
            if (!whole) {
#pragma unroll
                for (int e = 0; e < N; ++e) f[e] = e < valid ? Vec<T>::one(xr + c0 + e) * kLog2e : -INFINITY;
            }
            st.add<N>(f, valid);
        }
        st.warp_merge();
        if (lane == 0) {
            sm_m[wid] = st.m;
            sm_d[wid] = st.d;
        }
        __syncthreads();
        if (wid == 0) {
            Online t;
            if (lane < NT / 32) {
                t.m = sm_m[lane];
                t.d = sm_d[lane];
            }
            t.warp_merge();
            if (lane == 0) {
                fin[0] = t.m;
                fin[1] = 1.f / t.d;
            }
        }
        __syncthreads();
        const float m = fin[0], inv = fin[1];
        for (int i = threadIdx.x; i < nvec; i += NT) {
            const int c0 = i * N;
            const int valid = min(N, cols - c0);
            float f[N];
            bool whole = false;
            if constexpr (VEC) {
                if (valid == N) {
                    Vec<T>::load(xr + c0, f);
#pragma unroll
                    for (int e = 0; e < N; ++e) f[e] = ex2(f[e] * kLog2e - m) * inv;
                    Vec<T>::store(yr + c0, f);
                    whole = true;
                }
            }
            if (!whole) {
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (e < valid) Vec<T>::put(yr + c0 + e, ex2(Vec<T>::one(xr + c0 + e) * kLog2e - m) * inv);
            }
        }
        __syncthreads();   // fin[] is rewritten for the next row
    }
}

template <typename T, int NV, bool VEC>
cudaError_t launch_warp(const T *x, T *y, int64_t rows, int cols, int64_t xs, int64_t ys, int sms,
                        cudaStream_t stream) {
    const int64_t blocks = (rows + 7) / 8;
    const int grid = (int)(blocks < (int64_t)sms * 8 ? blocks : (int64_t)sms * 8);
    softmax_rows_warp_kernel<T, NV, VEC><<<grid, 256, 0, stream>>>(x, y, rows, cols, xs, ys);
    return cudaGetLastError();
}

// A register-row kernel over rows split into `csize` slices (csize CTAs per
// cluster; 1: no cluster).  The grid is as many rows (clusters) as fit on the
// GPU at once, asked of the runtime once per instance and cluster size; returns
// cudaErrorNotSupported when no cluster of that size fits.
template <typename T, int KV, int NT>
cudaError_t launch_cta_reg(const T *x, T *y, int64_t rows, int cols, int64_t xs, int64_t ys, int sms, int csize,
                           cudaStream_t stream) {
    static std::once_flag once[kMaxCluster + 1];
    static int resident[kMaxCluster + 1];   // CTAs per SM (csize 1) or clusters per GPU
    auto kern = softmax_rows_cta_reg_kernel<T, KV, NT>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(NT);
    cfg.stream = stream;
    if (csize > 1) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    std::call_once(once[csize], [&] {
        int n = 0;
        cudaError_t e;
        if (csize == 1) {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NT, 0);
        } else {
            cfg.gridDim = dim3(csize);
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        }
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            n = csize == 1 ? 1 : 0;
        }
        resident[csize] = n;
    });
    int64_t cap = csize == 1 ? (int64_t)sms * resident[csize] : (int64_t)resident[csize];
    if (cap <= 0) return cudaErrorNotSupported;
    const int64_t units = rows < cap ? rows : cap;
    cfg.gridDim = dim3((unsigned)(units * csize));
    return cudaLaunchKernelEx(&cfg, kern, x, y, rows, cols, xs, ys);
}

// Rows of `row_bytes` bytes through the shared-memory ring: stages and CTAs per
// SM chosen so that about 200 KB of each SM's shared memory holds rows.
// cudaErrorNotSupported when no CTA of that size fits on an SM.
template <typename T, int KV>
cudaError_t launch_smem_kv(const T *x, T *y, int64_t rows, int cols, int64_t xs, int64_t ys, int sms, uint32_t *err,
                           cudaStream_t stream) {
    constexpr int NT = kSmemThreads;
    constexpr int kMaxDyn = 200 * 1024;
    static std::once_flag once;
    static bool attr_ok = false;
    auto kern = softmax_rows_smem_kernel<T, NT, KV>;
    std::call_once(once, [&] {
        attr_ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDyn) == cudaSuccess;
        if (!attr_ok) (void)cudaGetLastError();
    });
    if (!attr_ok) return cudaErrorNotSupported;
    if ((cols + Vec<T>::N - 1) / Vec<T>::N > NT * KV) return cudaErrorNotSupported;
    const uint32_t bulk = (uint32_t)(cols / Vec<T>::N) * 16u;
    const uint32_t slot = (bulk + 127u) & ~127u;
    // as many CTAs per SM as the threads allow (each row's reductions take a
    // fixed latency that other CTAs' rows hide), each with the stages that share
    // the SM's ~200 KB among them (at least two: one row read while the next lands)
    constexpr int kCtasPerSm = 2048 / NT;
    int stages = (int)(kMaxDyn / ((size_t)kCtasPerSm * slot));
    stages = stages < 2 ? 2 : (stages > kSmemMaxStages ? kSmemMaxStages : stages);
    const size_t dyn = (size_t)stages * slot;
    if (slot == 0 || dyn > (size_t)kMaxDyn) return cudaErrorNotSupported;
    // CTAs per SM for this shared-memory size, asked once per size
    static std::mutex mu;
    static std::unordered_map<size_t, int> per_sm_of;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto f = per_sm_of.find(dyn);
        if (f != per_sm_of.end()) {
            per_sm = f->second;
        } else {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, dyn) != cudaSuccess) {
                (void)cudaGetLastError();
                per_sm = 0;
            }
            per_sm_of[dyn] = per_sm;
        }
    }
    if (per_sm <= 0) return cudaErrorNotSupported;
    const int64_t cap = (int64_t)sms * per_sm;
    const int grid = (int)(rows < cap ? rows : cap);
    kern<<<grid, NT, dyn, stream>>>(x, y, rows, cols, xs, ys, stages, slot, err);
    return cudaGetLastError();
}

// the ring kernel with as few vectors per thread as the row needs (4 or 8): the
// unused ones would still cost their instructions
template <typename T>
cudaError_t launch_smem(const T *x, T *y, int64_t rows, int cols, int64_t xs, int64_t ys, int sms, uint32_t *err,
                        cudaStream_t stream) {
    const int nvec = (cols + Vec<T>::N - 1) / Vec<T>::N;
    if (nvec <= kSmemThreads * 4) return launch_smem_kv<T, 4>(x, y, rows, cols, xs, ys, sms, err, stream);
    return launch_smem_kv<T, kSmemVecs>(x, y, rows, cols, xs, ys, sms, err, stream);
}

template <typename T, bool VEC>
cudaError_t launch_t(const T *x, T *y, int64_t rows, int cols, int64_t xs, int64_t ys, int sms, uint32_t *err,
                     cudaStream_t stream) {
    constexpr int N = VEC ? Vec<T>::N : 1;
    // a warp per row while the row fits in 8 accesses per lane (1024 fp32 or
    // 2048 bf16 elements with 16-byte accesses, 256 elements otherwise); longer
    // rows hold too many registers for enough warps per SM
    const int per_lane = (cols + 32 * N - 1) / (32 * N);
    if (per_lane <= 1) return launch_warp<T, 1, VEC>(x, y, rows, cols, xs, ys, sms, stream);
    if (per_lane <= 2) return launch_warp<T, 2, VEC>(x, y, rows, cols, xs, ys, sms, stream);
    if (per_lane <= 4) return launch_warp<T, 4, VEC>(x, y, rows, cols, xs, ys, sms, stream);
    if (per_lane <= 8) return launch_warp<T, 8, VEC>(x, y, rows, cols, xs, ys, sms, stream);
    const int64_t row_bytes = (int64_t)cols * (int64_t)sizeof(T);
    if constexpr (VEC) {
        // up to 16 KB: a CTA of 128 threads per row, 16 CTAs per SM, rows
        // streamed through shared memory (short rows need many rows in flight at
        // once).  Beyond, the row in registers: one CTA of 256 threads (32 KB
        // slice) up to 32 KB, of 512 threads (64 KB) up to 64 KB, a cluster of up
        // to 8 of the 256-thread CTAs up to 256 KB, of the 512-thread ones up to
        // 512 KB
        constexpr int64_t kSlice256 = 256 * 8 * 16, kSlice512 = 512 * 8 * 16;
        cudaError_t e = cudaErrorNotSupported;
        if (row_bytes <= 16384)
            e = launch_smem<T>(x, y, rows, cols, xs, ys, sms, err, stream);
        else if (row_bytes <= kSlice256)
            e = launch_cta_reg<T, 8, 256>(x, y, rows, cols, xs, ys, sms, 1, stream);
        else if (row_bytes <= kSlice512)
            e = launch_cta_reg<T, 8, 512>(x, y, rows, cols, xs, ys, sms, 1, stream);
        else if (row_bytes <= kMaxCluster * kSlice256)
            e = launch_cta_reg<T, 8, 256>(x, y, rows, cols, xs, ys, sms,
                                          (int)((row_bytes + kSlice256 - 1) / kSlice256), stream);
        else if (row_bytes <= kMaxCluster * kSlice512)
            e = launch_cta_reg<T, 8, 512>(x, y, rows, cols, xs, ys, sms,
                                          (int)((row_bytes + kSlice512 - 1) / kSlice512), stream);
        if (e != cudaErrorNotSupported) return e;
    }
    if (row_bytes <= 32768) {
        const int grid = (int)(rows < (int64_t)sms * 8 ? rows : (int64_t)sms * 8);
        softmax_rows_cta_kernel<T, VEC, 256><<<grid, 256, 0, stream>>>(x, y, rows, cols, xs, ys);
    } else {
        const int grid = (int)(rows < (int64_t)sms * 4 ? rows : (int64_t)sms * 4);
        softmax_rows_cta_kernel<T, VEC, 512><<<grid, 512, 0, stream>>>(x, y, rows, cols, xs, ys);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_rows(const void *x, void *y, int64_t rows, int cols, int64_t x_row_stride,
                                int64_t y_row_stride, int bf16, int sms, uint32_t *err, cudaStream_t stream) {
    const size_t es = bf16 ? 2 : 4;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                     ((size_t)x_row_stride * es) % 16 == 0 && ((size_t)y_row_stride * es) % 16 == 0;
    if (bf16) {
        const auto *xb = reinterpret_cast<const __nv_bfloat16 *>(x);
        auto *yb = reinterpret_cast<__nv_bfloat16 *>(y);
        return vec ? launch_t<__nv_bfloat16, true>(xb, yb, rows, cols, x_row_stride, y_row_stride, sms, err, stream)
                   : launch_t<__nv_bfloat16, false>(xb, yb, rows, cols, x_row_stride, y_row_stride, sms, err, stream);
    }
    const auto *xf = reinterpret_cast<const float *>(x);
    auto *yf = reinterpret_cast<float *>(y);
    return vec ? launch_t<float, true>(xf, yf, rows, cols, x_row_stride, y_row_stride, sms, err, stream)
               : launch_t<float, false>(xf, yf, rows, cols, x_row_stride, y_row_stride, sms, err, stream);
}

}  // namespace attn
