// state_update.cu -- single-token recurrent update of the selective SSM
// ("Efficient Scan", item 2 of the Mamba README: sequential scan for
// inference, constant memory).
//
// Per (batch, channel) the float32 state h[0..N) is read once and written
// once, in place:
//     Delta = softplus(dt + dt_bias)
//     h[n]  = exp(Delta A[n]) h[n] + Delta B[n] x
//     out   = (C . h + D x) * silu(z)
//
// The step is bound by HBM traffic on the state (2 * 4 * N bytes per
// channel).  The state is walked as 16-byte quads (four states): quad i is
// state words 4i..4i+3, i.e. channel i / Q, states 4 (i % Q) .. +3, with
// Q = N / 4.  Thread t of a block handles quads base + j * THREADS + t for
// j < J, so every warp-wide access touches 512 contiguous bytes; all J
// quads (and their per-channel inputs) are loaded before any arithmetic so
// J * 16 bytes of state per thread are in flight.  The Q lanes of a channel
// are adjacent and add their partial C . h with xor shuffles.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int kThreads = 256;
constexpr int kQuadsPerThread = 4;

template <typename T>
struct Quad;  // four consecutive activations of B or C
template <>
struct Quad<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ float4 f(type v) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
};
template <>
struct Quad<float> {
    using type = float4;
    static __device__ __forceinline__ float4 f(type v) { return v; }
};

template <typename T, int N, bool kFast, bool kVecBC>
__global__ void __launch_bounds__(kThreads)
state_update_kernel(UpdateArgs p) {
    static_assert(N % 4 == 0, "d_state must be a multiple of 4");
    constexpr int Q = N / 4;
    constexpr int J = kQuadsPerThread;
    const int64_t total = p.batch * p.dim * Q;
    const int64_t base = (int64_t)blockIdx.x * (kThreads * J) + threadIdx.x;
    const int q = threadIdx.x % Q;  // same for every j (kThreads is a multiple of Q)

    float4 s[J], a[J], bv[J], cv[J];
    float xv[J], dl[J], zv[J], dd[J];
    bool act[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int64_t i = base + (int64_t)j * kThreads;
        act[j] = i < total;
        const int64_t ii = act[j] ? i : 0;   // inactive quads read quad 0 and store nothing
        const int64_t bd = ii / Q;
        const int64_t b = bd / p.dim, d = bd - b * p.dim;
        s[j] = reinterpret_cast<const float4*>(p.state)[ii];
        a[j] = reinterpret_cast<const float4*>(p.A)[d * Q + q];
        const T* Bp = static_cast<const T*>(p.B) + b * N + 4 * q;
        const T* Cp = static_cast<const T*>(p.C) + b * N + 4 * q;
        if constexpr (kVecBC) {
            bv[j] = Quad<T>::f(*reinterpret_cast<const typename Quad<T>::type*>(Bp));
            cv[j] = Quad<T>::f(*reinterpret_cast<const typename Quad<T>::type*>(Cp));
        } else {
            bv[j] = make_float4(to_f32(Bp[0]), to_f32(Bp[1]), to_f32(Bp[2]), to_f32(Bp[3]));
            cv[j] = make_float4(to_f32(Cp[0]), to_f32(Cp[1]), to_f32(Cp[2]), to_f32(Cp[3]));
        }
        xv[j] = to_f32(static_cast<const T*>(p.x)[bd]);
        dl[j] = to_f32(static_cast<const T*>(p.dt)[bd]) + (p.dt_bias ? p.dt_bias[d] : 0.f);
        zv[j] = p.z ? to_f32(static_cast<const T*>(p.z)[bd]) : 0.f;
        dd[j] = p.D ? p.D[d] : 0.f;
    }

#pragma unroll
    for (int j = 0; j < J; ++j) {
        const float dlt = p.softplus ? softplus_f<kFast>(dl[j]) : dl[j];
        const float du = dlt * xv[j];
        const float d2 = dlt * kLog2e;
        const float hs[4] = {s[j].x, s[j].y, s[j].z, s[j].w};
        const float av[4] = {a[j].x, a[j].y, a[j].z, a[j].w};
        const float bb[4] = {bv[j].x, bv[j].y, bv[j].z, bv[j].w};
        const float cc[4] = {cv[j].x, cv[j].y, cv[j].z, cv[j].w};
        float h[4], y = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float dA = decay_exp2<kFast>(d2 * av[k]);
            h[k] = fmaf(dA, hs[k], du * bb[k]);
            y = fmaf(cc[k], h[k], y);
        }
#pragma unroll
        for (int m = Q / 2; m >= 1; m >>= 1) y += __shfl_xor_sync(0xffffffffu, y, m);
        const int64_t i = base + (int64_t)j * kThreads;
        if (act[j]) {
            reinterpret_cast<float4*>(p.state)[i] = make_float4(h[0], h[1], h[2], h[3]);
            if (q == 0) {
                const float gate = p.z ? silu_f<kFast>(zv[j]) : 1.f;
                static_cast<T*>(p.out)[i / Q] = from_f32<T>((y + dd[j] * xv[j]) * gate);
            }
        }
    }
}

template <typename T, int N, bool kVec>
cudaError_t launch_v(const UpdateArgs& a, cudaStream_t s) {
    constexpr bool kFast = !std::is_same<T, float>::value;
    const int64_t total = a.batch * a.dim * (N / 4);
    const int64_t per_block = (int64_t)kThreads * kQuadsPerThread;
    const int64_t blocks = (total + per_block - 1) / per_block;
    state_update_kernel<T, N, kFast, kVec><<<(unsigned)blocks, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_n(const UpdateArgs& a, cudaStream_t s) {
    // one vector load per quad of B / C needs both rows aligned to 4 elements
    const uintptr_t al = 4 * sizeof(T);
    const bool vec = (reinterpret_cast<uintptr_t>(a.B) % al) == 0 && (reinterpret_cast<uintptr_t>(a.C) % al) == 0;
    if (vec) return launch_v<T, N, true>(a, s);
    return launch_v<T, N, false>(a, s);
}

template <typename T>
cudaError_t launch_t(const UpdateArgs& a, cudaStream_t s) {
    switch (a.dstate) {
        case 4: return launch_n<T, 4>(a, s);
        case 8: return launch_n<T, 8>(a, s);
        case 16: return launch_n<T, 16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_state_update(const UpdateArgs& a, DType dt, cudaStream_t s) {
    if (dt == DType::F32) return launch_t<float>(a, s);
    return launch_t<__nv_bfloat16>(a, s);
}

}  // namespace ssm
