// conv1d.cu -- the depthwise causal convolution that produces the scan input
// u in the Mamba block (width d_conv, the "local convolution width" of the
// pages' usage examples: "Mamba: Selective State Space Models" README,
// "Quick Start"; "What are State Space Models (SSMs)?", "Getting Started"),
// followed by the optional SiLU, and its single-token decode step.
//
//     y_t = bias[d] + sum_{k=0}^{W-1} w[d][k] * x_{t-(W-1)+k}
//     out_t = silu(y_t)  (when requested)
//
// x_s for s < 0 comes from a carried state (the W-1 inputs before the
// sequence, oldest first) or is zero.
//
// The forward pass is a streaming kernel bound by HBM (one read of x and one
// write of out per element): a thread owns a 16-byte vector of channels (8
// bf16 or 4 float32) over a tile of TT consecutive steps and keeps the W-1
// previous inputs of each channel in registers, so consecutive threads move
// consecutive 16-byte pieces of each (batch, step) row.  Rows whose length
// or alignment does not allow 16-byte vectors take a one-channel-per-thread
// version of the same kernel.
#include <cuda_bf16.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

#include "ssm_internal.cuh"

namespace ssm {

namespace {

constexpr int kConvTile = 128;     // steps per thread (64: 0.479 ms on 1 x 131072 x 5120, 128: 0.442 ms)
constexpr int kConvThreads = 128;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// silu(y) = y * sigmoid(y): (y/2)(1 + tanh(y/2)) with the hardware tanh for
// bf16 outputs (absolute error below the output's rounding), the accurate
// library exponential for float32 outputs.
template <bool kFast>
__device__ __forceinline__ float conv_silu(float y) {
    if constexpr (kFast) {
        const float hy = 0.5f * y;
        float t;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hy));
        return fmaf(hy, t, hy);
    } else {
        return y / (1.f + expf(-y));
    }
}

template <typename T, int V>
struct Vec {
    T e[V];
};

template <typename T, int V>
__device__ __forceinline__ Vec<T, V> ld_vec(const T* p) {
    Vec<T, V> v;
    if constexpr (V * sizeof(T) == 16) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(p));
        memcpy(&v, &q, 16);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) v.e[i] = p[i];
    }
    return v;
}

template <typename T, int V>
__device__ __forceinline__ void st_vec(T* p, const Vec<T, V>& v) {
    if constexpr (V * sizeof(T) == 16) {
        uint4 q;
        memcpy(&q, &v, 16);
        __stcs(reinterpret_cast<uint4*>(p), q);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) p[i] = v.e[i];
    }
}

// One thread: channels c0 .. c0+V-1 of batch row b, steps t0 .. t0+TT-1.
template <typename T, int V, int W, bool kSilu, bool kFast>
__global__ void __launch_bounds__(kConvThreads)
conv1d_fwd_kernel(const T* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
                  const float* __restrict__ state_in, T* __restrict__ out, int64_t L, int64_t dim, int64_t nvec,
                  int64_t ntile) {
    const int64_t gid = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;
    const int64_t vi = gid % nvec, tile = gid / nvec;
    if (tile >= ntile) return;
    const int64_t b = blockIdx.y;
    const int64_t c0 = vi * V;
    const int64_t t0 = tile * kConvTile;
    const int64_t t1 = min(t0 + kConvTile, L);

    float wr[V][W], br[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const bool ok = c0 + i < dim;
#pragma unroll
        for (int k = 0; k < W; ++k) wr[i][k] = ok ? w[(c0 + i) * W + k] : 0.f;
        br[i] = (bias && ok) ? bias[c0 + i] : 0.f;
    }
    // the W-1 inputs before t0, oldest first
    float win[W > 1 ? W - 1 : 1][V];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
        const int64_t s = t0 - (W - 1) + j;
        if (s >= 0) {
            const Vec<T, V> v = ld_vec<T, V>(x + (b * L + s) * dim + c0);
#pragma unroll
            for (int i = 0; i < V; ++i) win[j][i] = to_f(v.e[i]);
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i)
                win[j][i] = (state_in && c0 + i < dim) ? state_in[((b * dim) + c0 + i) * (W - 1) + (W - 1) + s] : 0.f;
        }
    }
    const T* xp = x + (b * L + t0) * dim + c0;
    T* op = out + (b * L + t0) * dim + c0;
    auto step = [&](const Vec<T, V>& xv, T* o) {
        Vec<T, V> ov;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const float xc = to_f(xv.e[i]);
            float acc = br[i];
#pragma unroll
            for (int k = 0; k < W - 1; ++k) acc = fmaf(wr[i][k], win[k][i], acc);
            acc = fmaf(wr[i][W - 1], xc, acc);
            if constexpr (kSilu) acc = conv_silu<kFast>(acc);
            ov.e[i] = from_f<T>(acc);
#pragma unroll
            for (int k = 0; k + 1 < W - 1; ++k) win[k][i] = win[k + 1][i];
            if constexpr (W > 1) win[W - 2][i] = xc;
        }
        st_vec<T, V>(o, ov);
    };
    if constexpr (V * sizeof(T) == 16) {
        // 16-byte rows: each thread streams its column through a private ring of
        // kRing steps in shared memory, filled by asynchronous copies kGroup
        // steps at a time, so kRing * 16 bytes per thread are in flight without
        // holding registers (the kernel is bound by bytes in flight).
        constexpr int kGroup = 4, kRing = 16, kGroups = kRing / kGroup;
        __shared__ __align__(16) unsigned char ring[kRing][kConvThreads][16];
        const int nst = (int)(t1 - t0);
        auto issue = [&](int g) {
            if (g * kGroup < nst) {
#pragma unroll
                for (int u = 0; u < kGroup; ++u) {
                    const int s = g * kGroup + u;
                    if (s < nst) {
                        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&ring[s % kRing][threadIdx.x][0]);
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(xp + (int64_t)s * dim)
                                     : "memory");
                    }
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
#pragma unroll
        for (int g = 0; g < kGroups; ++g) issue(g);
        for (int g = 0; g * kGroup < nst; ++g) {
            asm volatile("cp.async.wait_group %0;" ::"n"(kGroups - 1) : "memory");
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int s = g * kGroup + u;
                if (s < nst) {
                    Vec<T, V> xv;
                    memcpy(&xv, &ring[s % kRing][threadIdx.x][0], 16);
                    step(xv, op + (int64_t)s * dim);
                }
            }
            issue(g + kGroups);   // into the slots just read
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
        for (int64_t t = t0; t < t1; ++t, xp += dim, op += dim) step(ld_vec<T, V>(xp), op);
    }
}

// state_out[b][d][k] = x_{L-(W-1)+k} (from the carried state when L < W-1);
// every value is read before any is written, so state_out may be state_in.
template <typename T, int W>
__global__ void conv1d_state_kernel(const T* __restrict__ x, const float* state_in, float* state_out, int64_t L,
                                    int64_t dim, int64_t batch) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= batch * dim) return;
    const int64_t b = i / dim, d = i % dim;
    float v[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
        const int64_t s = L - (W - 1) + k;
        v[k] = s >= 0 ? to_f(x[(b * L + s) * dim + d])
                      : (state_in ? state_in[i * (W - 1) + (W - 1) + s] : 0.f);
    }
#pragma unroll
    for (int k = 0; k < W - 1; ++k) state_out[i * (W - 1) + k] = v[k];
}

// One decode step per (batch, channel): window = state (oldest first) then x.
template <typename T, int W, bool kSilu, bool kFast>
__global__ void conv1d_update_kernel(float* __restrict__ state, const T* __restrict__ x, const float* __restrict__ w,
                                     const float* __restrict__ bias, T* __restrict__ out, int64_t dim,
                                     int64_t total) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int64_t d = i % dim;
    float* st = state + i * (W - 1);
    float s[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int k = 0; k < W - 1; ++k) s[k] = st[k];
    const float xc = to_f(x[i]);
    float acc = bias ? bias[d] : 0.f;
#pragma unroll
    for (int k = 0; k < W - 1; ++k) acc = fmaf(w[d * W + k], s[k], acc);
    acc = fmaf(w[d * W + W - 1], xc, acc);
    if constexpr (kSilu) acc = conv_silu<kFast>(acc);
    out[i] = from_f<T>(acc);
#pragma unroll
    for (int k = 0; k + 1 < W - 1; ++k) st[k] = s[k + 1];
    if constexpr (W > 1) st[W - 2] = xc;
}

template <typename T, int V, int W, bool kSilu>
cudaError_t launch_fwd_v(const ConvArgs& a, cudaStream_t s) {
    constexpr bool kFast = !std::is_same<T, float>::value;
    const int64_t nvec = (a.dim + V - 1) / V;
    const int64_t ntile = (a.seqlen + kConvTile - 1) / kConvTile;
    const int64_t blocks = (nvec * ntile + kConvThreads - 1) / kConvThreads;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    conv1d_fwd_kernel<T, V, W, kSilu, kFast><<<dim3((unsigned)blocks, (unsigned)a.batch), kConvThreads, 0, s>>>(
        static_cast<const T*>(a.x), a.w, a.bias, a.state_in, static_cast<T*>(a.out), a.seqlen, a.dim, nvec, ntile);
    return cudaGetLastError();
}

template <typename T, int W>
cudaError_t launch_fwd_t(const ConvArgs& a, cudaStream_t s) {
    constexpr int V = 16 / (int)sizeof(T);
    const bool vec = a.dim % V == 0 && (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.out) % 16) == 0;
    cudaError_t e;
    if (vec)
        e = a.silu ? launch_fwd_v<T, V, W, true>(a, s) : launch_fwd_v<T, V, W, false>(a, s);
    else
        e = a.silu ? launch_fwd_v<T, 1, W, true>(a, s) : launch_fwd_v<T, 1, W, false>(a, s);
    if (e != cudaSuccess || !a.state_out || W == 1) return e;
    const int64_t n = a.batch * a.dim;
    conv1d_state_kernel<T, W><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
        static_cast<const T*>(a.x), a.state_in, a.state_out, a.seqlen, a.dim, a.batch);
    return cudaGetLastError();
}

template <typename T, int W>
cudaError_t launch_update_t(const ConvArgs& a, cudaStream_t s) {
    constexpr bool kFast = !std::is_same<T, float>::value;
    const int64_t n = a.batch * a.dim;
    const unsigned grid = (unsigned)((n + 255) / 256);
    if (a.silu)
        conv1d_update_kernel<T, W, true, kFast><<<grid, 256, 0, s>>>(a.state_out, static_cast<const T*>(a.x), a.w,
                                                                       a.bias, static_cast<T*>(a.out), a.dim, n);
    else
        conv1d_update_kernel<T, W, false, kFast><<<grid, 256, 0, s>>>(a.state_out, static_cast<const T*>(a.x), a.w,
                                                                        a.bias, static_cast<T*>(a.out), a.dim, n);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_fwd(const ConvArgs& a, cudaStream_t s) {
    switch (a.width) {
        case 1: return launch_fwd_t<T, 1>(a, s);
        case 2: return launch_fwd_t<T, 2>(a, s);
        case 3: return launch_fwd_t<T, 3>(a, s);
        case 4: return launch_fwd_t<T, 4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t dispatch_update(const ConvArgs& a, cudaStream_t s) {
    switch (a.width) {
        case 1: return launch_update_t<T, 1>(a, s);
        case 2: return launch_update_t<T, 2>(a, s);
        case 3: return launch_update_t<T, 3>(a, s);
        case 4: return launch_update_t<T, 4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_conv1d_fwd(const ConvArgs& a, DType dt, cudaStream_t s) {
    return dt == DType::BF16 ? dispatch_fwd<__nv_bfloat16>(a, s) : dispatch_fwd<float>(a, s);
}

cudaError_t launch_conv1d_update(const ConvArgs& a, DType dt, cudaStream_t s) {
    return dt == DType::BF16 ? dispatch_update<__nv_bfloat16>(a, s) : dispatch_update<float>(a, s);
}

}  // namespace ssm
