// softmax.cu -- softmax of every row of a matrix with the online two-pass
// algorithm of "从零实现 vLLM (1.3)：如何加速 Attention 计算", section
// 减少遍历次数的“在线 Softmax”: pass 1 keeps the running maximum m and the proxy
// denominator d' = d' * e^(m_old - m_new) + e^(x - m_new); pass 2 writes
// y = e^(x - m) / d'.  The update runs on 16-byte vectors (the vector's max
// first, then its terms), which is the same recurrence over blocks of 4 or 8
// elements.  Partial (m, d') states of threads merge exactly:
//   m = max(m1, m2),  d' = d1 e^(m1 - m) + d2 e^(m2 - m).
//
// HBM-bound.  Rows of up to 1024 fp32 / 2048 bf16 elements: one warp per row,
// the row held in registers (one read, one write).  Longer rows: one CTA per row; pass 2
// re-reads the row, which the CTAs in flight keep in L2.
#include "common.cuh"
#include "kernels.h"

namespace attn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

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
// one CTA per row, two passes over the row
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

template <typename T, bool VEC>
cudaError_t launch_t(const T *x, T *y, int64_t rows, int cols, int64_t xs, int64_t ys, int sms,
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
    if ((int64_t)cols * (int64_t)sizeof(T) <= 32768) {
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
                                int64_t y_row_stride, int bf16, int sms, cudaStream_t stream) {
    const size_t es = bf16 ? 2 : 4;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                     ((size_t)x_row_stride * es) % 16 == 0 && ((size_t)y_row_stride * es) % 16 == 0;
    if (bf16) {
        const auto *xb = reinterpret_cast<const __nv_bfloat16 *>(x);
        auto *yb = reinterpret_cast<__nv_bfloat16 *>(y);
        return vec ? launch_t<__nv_bfloat16, true>(xb, yb, rows, cols, x_row_stride, y_row_stride, sms, stream)
                   : launch_t<__nv_bfloat16, false>(xb, yb, rows, cols, x_row_stride, y_row_stride, sms, stream);
    }
    const auto *xf = reinterpret_cast<const float *>(x);
    auto *yf = reinterpret_cast<float *>(y);
    return vec ? launch_t<float, true>(xf, yf, rows, cols, x_row_stride, y_row_stride, sms, stream)
               : launch_t<float, false>(xf, yf, rows, cols, x_row_stride, y_row_stride, sms, stream);
}

}  // namespace attn
