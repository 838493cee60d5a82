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
// channel).  One thread owns one channel and all N of its states: N/4
// independent 16-byte loads are in flight per thread, the per-channel terms
// (softplus, silu, D x) are evaluated once, and y needs no cross-lane sum.
// Consecutive threads take consecutive channels, so x/dt/z/out accesses are
// coalesced and every byte of a warp's 32 * 4N-byte state block is used.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int kThreads = 256;

template <typename T, int N, bool kFast, bool kVecBC>
__global__ void __launch_bounds__(kThreads)
state_update_kernel(UpdateArgs p) {
    static_assert(N % 4 == 0, "d_state must be a multiple of 4");
    const int64_t bd = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (bd >= p.batch * p.dim) return;
    const int64_t b = bd / p.dim, d = bd - b * p.dim;

    float4* sp = reinterpret_cast<float4*>(p.state) + bd * (N / 4);
    float4 s4[N / 4];
#pragma unroll
    for (int q = 0; q < N / 4; ++q) s4[q] = sp[q];

    const float xv = to_f32(static_cast<const T*>(p.x)[bd]);
    float dl = to_f32(static_cast<const T*>(p.dt)[bd]);
    if (p.dt_bias) dl += p.dt_bias[d];
    if (p.softplus) dl = softplus_f<kFast>(dl);
    const float gate = p.z ? silu_f<kFast>(to_f32(static_cast<const T*>(p.z)[bd])) : 1.f;
    const float skip = p.D ? p.D[d] * xv : 0.f;
    const float du = dl * xv;
    const float dl2 = dl * kLog2e;

    float Bv[N], Cv[N];
    const T* Bp = static_cast<const T*>(p.B) + b * N;
    const T* Cp = static_cast<const T*>(p.C) + b * N;
    if constexpr (kVecBC) {
        constexpr int kPer = 16 / sizeof(T);  // elements per 16-byte load
#pragma unroll
        for (int q = 0; q < N / kPer; ++q) {
            const uint4 rb = reinterpret_cast<const uint4*>(Bp)[q];
            const uint4 rc = reinterpret_cast<const uint4*>(Cp)[q];
            const T* eb = reinterpret_cast<const T*>(&rb);
            const T* ec = reinterpret_cast<const T*>(&rc);
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                Bv[q * kPer + j] = to_f32(eb[j]);
                Cv[q * kPer + j] = to_f32(ec[j]);
            }
        }
    } else {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            Bv[n] = to_f32(Bp[n]);
            Cv[n] = to_f32(Cp[n]);
        }
    }

    const float4* ap = reinterpret_cast<const float4*>(p.A) + d * (N / 4);
    float y = 0.f;
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
        const float4 a = ap[q];
        float h[4] = {s4[q].x, s4[q].y, s4[q].z, s4[q].w};
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float dA = decay_exp2<kFast>(dl2 * av[j]);
            h[j] = fmaf(dA, h[j], du * Bv[4 * q + j]);
            y = fmaf(Cv[4 * q + j], h[j], y);
        }
        s4[q] = make_float4(h[0], h[1], h[2], h[3]);
    }
#pragma unroll
    for (int q = 0; q < N / 4; ++q) sp[q] = s4[q];
    static_cast<T*>(p.out)[bd] = from_f32<T>((y + skip) * gate);
}

template <typename T, int N, bool kVec>
cudaError_t launch_v(const UpdateArgs& a, cudaStream_t s) {
    constexpr bool kFast = !std::is_same<T, float>::value;
    const int64_t total = a.batch * a.dim;
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    state_update_kernel<T, N, kFast, kVec><<<(unsigned)blocks, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_n(const UpdateArgs& a, cudaStream_t s) {
    // 16-byte loads of a batch row's B and C need both rows 16-byte aligned.
    const bool vec = (N * sizeof(T)) % 16 == 0 &&
                     (reinterpret_cast<uintptr_t>(a.B) % 16) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.C) % 16) == 0;
    if constexpr ((N * sizeof(T)) % 16 == 0) {
        if (vec) return launch_v<T, N, true>(a, s);
    }
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
