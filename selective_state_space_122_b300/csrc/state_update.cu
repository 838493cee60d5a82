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
// channel).  The state is read and written as 16-byte quads by L = N / 4
// adjacent lanes per channel, so every warp load or store of the state is one
// contiguous, fully used 512-byte run (a thread owning a channel's 64 bytes
// would touch half of every 32-byte sector per instruction).  A thread serves
// its quad of the channel in L consecutive batch rows; lane g of a channel
// computes that channel's per-(row, channel) terms -- softplus, Delta x, D x,
// silu(z) -- for row g only, and the channel's lanes exchange them by
// shuffle, so none of it is computed twice.  Row addresses advance by fixed
// strides from the group's first row (the channel's B/C group is divided out
// once per thread, not per row).  Per row: the states are updated
// with one SFU exp2 each, C . h is summed over the channel's lanes by
// shuffle, and the lane that owns the row writes the output.  A block covers
// 32 * 4 / L channels x 2 L batch rows; each row of A is loaded once per
// thread and reused over its rows.  State loads use the default cache
// policy, state stores the streaming (evict-first) one.  Measured on a B300
// (256 x 5120 x 16, CUDA events): 34.8 us with a clean L2 (5.1 TB/s for
// 178.6 MB), 38.9 us when L2 first holds dirty lines, against 38.9 / 43.0 us
// with default stores; streaming loads as well were slower (45.0 / 49.2 us).
// Five blocks of 256 threads per SM: more residency (fewer registers) ran
// slower (41.0 us at six blocks, 61.4 us at eight).
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int kThreads = 128;   // 4 warps
constexpr int kRowsY = 2;       // row groups (of L rows) per block

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

// Block: kThreads lanes = 32 * 4 / L channels x L lanes (lane g of a channel
// owns states 4g .. 4g+3), times kRowsY groups of L batch rows in y.
template <typename T, int N, bool kFast, bool kVecBC>
__global__ void __launch_bounds__(kThreads * kRowsY, 5)
state_update_kernel(UpdateArgs p) {
    static_assert(N % 4 == 0, "d_state must be a multiple of 4");
    constexpr int L = N / 4;                   // lanes (and rows) per channel
    constexpr int CPB = kThreads / L;          // channels per block
    const int g = threadIdx.x % L;
    const int64_t d = (int64_t)blockIdx.x * CPB + threadIdx.x / L;
    const int64_t b0 = ((int64_t)blockIdx.y * kRowsY + threadIdx.y) * L;
    const bool d_ok = d < p.dim;
    const int lane = threadIdx.x & 31;
    const int base = lane - g;                 // lane 0 of this channel's group

    // per-channel constants (the channel's lanes read the same words)
    const float4 a = d_ok ? __ldg(reinterpret_cast<const float4*>(p.A) + d * L + g) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float dd = (p.D && d_ok) ? __ldg(p.D + d) : 0.f;
    const float bias = (p.dt_bias && d_ok) ? __ldg(p.dt_bias + d) : 0.f;

    // this lane's row (b0 + g): the per-(row, channel) terms
    const int64_t bg = b0 + g;
    const bool own_ok = d_ok && bg < p.batch;
    const int64_t bdg = bg * p.dim + d;
    float xg = 0.f, dlg = 0.f, zg = 0.f;
    if (own_ok) {
        xg = to_f32(static_cast<const T*>(p.x)[bdg]);
        dlg = to_f32(static_cast<const T*>(p.dt)[bdg]) + bias;
        if (p.z) zg = to_f32(static_cast<const T*>(p.z)[bdg]);
    }
    // row b0's state quad, B/C quad and output; the next row is dim * L
    // quads, ngroups * N activations and dim outputs further (hoisted: no
    // per-row division or 64-bit index products)
    float4* st0 = reinterpret_cast<float4*>(p.state) + (b0 * p.dim + d) * L + g;
    const int64_t st_row = p.dim * L;
    const int64_t grp = d_ok ? (int64_t)((uint32_t)d / (uint32_t)p.gch) : 0;
    const T* B0 = static_cast<const T*>(p.B) + (b0 * p.ngroups + grp) * N + 4 * g;
    const T* C0 = static_cast<const T*>(p.C) + (b0 * p.ngroups + grp) * N + 4 * g;
    const int64_t bc_row = p.ngroups * N;
    T* out0 = static_cast<T*>(p.out) + b0 * p.dim + d;
    const int nrow = d_ok ? (p.batch - b0 < L ? (int)(p.batch - b0) : L) : 0;   // valid rows of this group
    // the states of all L rows, loaded before any arithmetic (L loads in flight)
    float4 s[L];
#pragma unroll
    for (int r = 0; r < L; ++r) s[r] = r < nrow ? st0[r * st_row] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.softplus) dlg = softplus_f<kFast>(dlg);
    const float dxg = dlg * xg;
    const float gate = p.z ? silu_f<kFast>(zg) : 1.f;
    const float2 a01 = make_float2(a.x * kLog2e, a.y * kLog2e), a23 = make_float2(a.z * kLog2e, a.w * kLog2e);

#pragma unroll
    for (int r = 0; r < L; ++r) {
        const bool row_ok = r < nrow;
        // row r's Delta and Delta x, from the lane that owns row r
        const float dl = __shfl_sync(0xffffffffu, dlg, base + r);
        const float dx = __shfl_sync(0xffffffffu, dxg, base + r);
        float4 bv = make_float4(0.f, 0.f, 0.f, 0.f), cv = bv;
        if (row_ok) {
            const T* Bp = B0 + r * bc_row;
            const T* Cp = C0 + r * bc_row;
            if constexpr (kVecBC) {
                bv = Quad<T>::f(*reinterpret_cast<const typename Quad<T>::type*>(Bp));
                cv = Quad<T>::f(*reinterpret_cast<const typename Quad<T>::type*>(Cp));
            } else {
                bv = make_float4(to_f32(Bp[0]), to_f32(Bp[1]), to_f32(Bp[2]), to_f32(Bp[3]));
                cv = make_float4(to_f32(Cp[0]), to_f32(Cp[1]), to_f32(Cp[2]), to_f32(Cp[3]));
            }
        }
        const float2 dl2 = splat2(dl), dx2 = splat2(dx);
        const float2 e0 = mul2(dl2, a01), e1 = mul2(dl2, a23);
        const float2 h0 = fma2(make_float2(decay_exp2<kFast>(e0.x), decay_exp2<kFast>(e0.y)),
                               make_float2(s[r].x, s[r].y), mul2(dx2, make_float2(bv.x, bv.y)));
        const float2 h1 = fma2(make_float2(decay_exp2<kFast>(e1.x), decay_exp2<kFast>(e1.y)),
                               make_float2(s[r].z, s[r].w), mul2(dx2, make_float2(bv.z, bv.w)));
        const float2 c2 = fma2(make_float2(cv.z, cv.w), h1, mul2(make_float2(cv.x, cv.y), h0));
        float y = c2.x + c2.y;
#pragma unroll
        for (int o = 1; o < L; o <<= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
        if (row_ok) {
            __stcs(st0 + r * st_row, make_float4(h0.x, h0.y, h1.x, h1.y));
            // the owner of row r has its D x and gate
            if (g == r) out0[r * p.dim] = from_f32<T>((y + dd * xg) * gate);
        }
    }
}

template <typename T, int N, bool kVec>
cudaError_t launch_v(const UpdateArgs& a, cudaStream_t s) {
    constexpr bool kFast = !std::is_same<T, float>::value;
    constexpr int L = N / 4, CPB = kThreads / L;
    const int64_t rows = kRowsY * L;
    const dim3 grid((unsigned)((a.dim + CPB - 1) / CPB), (unsigned)((a.batch + rows - 1) / rows));
    state_update_kernel<T, N, kFast, kVec><<<grid, dim3(kThreads, kRowsY), 0, s>>>(a);
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
    if (a.batch > 65535LL * kRowsY) return cudaErrorInvalidValue;
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
