// scan_bwd.cu -- the backward of the selective scan: every input's gradient
// given dout = dL/d out (the training half of the pages' "Efficient Scan":
// "Mamba: Selective State Space Models" README).
//
// With x_t = delta_raw_t + bias, Delta_t = softplus(x_t) (or x_t),
// a_t[n] = exp(Delta_t A[n]), h_t = a_t h_{t-1} + Delta_t B_t u_t,
// y_t = C_t . h_t + D u_t, out_t = y_t silu(z_t), the adjoint state
// lambda_t = dL/dh_t runs backwards in time,
//     dy_t = dout_t silu(z_t),   lambda_t = C_t dy_t + a_{t+1} lambda_{t+1},
// and the gradients are sums of per-step terms:
//     dC_t[n] = sum_d dy_t h_t[n]          dB_t[n] = sum_d lambda_t[n] Delta_t u_t
//     du_t    = D dy_t + sum_n lambda_t[n] Delta_t B_t[n]
//     dDelta_t = sum_n lambda_t[n] (A[n] a_t[n] h_{t-1}[n] + B_t[n] u_t)
//     dA[n]   = sum_{b,t} lambda_t[n] Delta_t a_t[n] h_{t-1}[n]
//     dD = sum dy_t u_t,   dz_t = dout_t y_t silu'(z_t),
//     ddelta_raw_t = dDelta_t softplus'(x_t),   dbias = sum ddelta_raw_t.
//
// Work decomposition: a CTA owns CC channels of one batch row (one lane per
// (channel, state): N lanes per channel, 8 warps) and the whole sequence.
//   pass 1: the forward recurrence, storing the state entering every K-step
//           chunk in the workspace;
//   pass 2: the chunks in reverse order: per chunk, stage u, delta_raw, z,
//           dout and B, C in shared memory, evaluate the per-(t, d) terms once,
//           recompute the chunk's states from its checkpoint into registers,
//           then run the adjoint backwards over the chunk; sums over a
//           channel's states are warp shuffles; sums over the CTA's channels
//           (dB, dC) are warp shuffles into per-warp shared-memory partials,
//           added up and flushed to global memory once per chunk.
// dA, dB, dC, dD and dbias accumulate with atomics across CTAs and batch rows
// (the launcher zeroes them first).
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "ssm_internal.cuh"

namespace ssm {

namespace {

constexpr int kBwdThreads = 256;   // 8 warps

// steps per chunk (the staged tiles and the per-warp dB/dC partials fit the
// 48 KB of static shared memory for every state count)
__host__ __device__ constexpr int bwd_chunk(int) { return 16; }

template <typename T>
__device__ __forceinline__ float bw_ld(const T* p, int64_t i) {
    if constexpr (std::is_same<T, float>::value) return p[i];
    else return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void bw_st(T* p, int64_t i, float v) {
    if constexpr (std::is_same<T, float>::value) p[i] = v;
    else p[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float bw_sigmoid(float v) { return 1.f / (1.f + expf(-v)); }
__device__ __forceinline__ float bw_softplus(float v) { return fmaxf(v, 0.f) + log1pf(expf(-fabsf(v))); }

// sum over the N lanes of one channel (lanes n = 0 .. N-1 of a group)
template <int N>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = N / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T, int N>
__global__ void __launch_bounds__(kBwdThreads, 2)
scan_bwd_kernel(const BwdArgs p, float* __restrict__ ckpt) {
    constexpr int K = bwd_chunk(N);
    constexpr int CPW = 32 / N;                  // channels per warp
    constexpr int CC = CPW * (kBwdThreads / 32); // channels per CTA
    __shared__ float s_u[K][CC], s_dl[K][CC], s_dy[K][CC], s_y[K][CC], s_du[K][CC], s_dd[K][CC];
    __shared__ float s_x[K][CC], s_z[K][CC], s_do[K][CC];
    __shared__ float s_B[N][K], s_C[N][K];
    __shared__ float s_pB[kBwdThreads / 32][N][K], s_pC[kBwdThreads / 32][N][K];   // per-warp partials
    __shared__ float s_dD[CC], s_db[CC];

    const T* u = static_cast<const T*>(p.u);
    const T* dr = static_cast<const T*>(p.delta);
    const T* Bg = static_cast<const T*>(p.B);
    const T* Cg = static_cast<const T*>(p.C);
    const T* zg = static_cast<const T*>(p.z);
    const T* dout = static_cast<const T*>(p.dout);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = lane % N;
    const int cl = warp * CPW + lane / N;        // channel within the CTA
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * CC;
    const int64_t d = d0 + cl;
    const bool ch_ok = d < p.dim;
    const int64_t L = p.seqlen, dim = p.dim;
    const int64_t nch = (L + K - 1) / K;
    const float An = ch_ok ? p.A[d * N + n] : 0.f;
    const float Dd = (p.D && ch_ok) ? p.D[d] : 0.f;

    for (int i = tid; i < CC; i += kBwdThreads) s_dD[i] = s_db[i] = 0.f;

    // per-(t, d) loads and terms of chunk c into shared memory
    auto stage = [&](int64_t c, bool backward) {
        const int64_t t0 = c * K;
        for (int i = tid; i < K * CC; i += kBwdThreads) {
            const int k = i / CC, cc = i % CC;
            const int64_t t = t0 + k, dd = d0 + cc;
            const bool ok = t < L && dd < dim;
            const int64_t gi = (b * L + t) * dim + dd;
            const float xr = ok ? bw_ld(dr, gi) + (p.delta_bias ? p.delta_bias[dd] : 0.f) : 0.f;
            const float dl = ok ? (p.softplus ? bw_softplus(xr) : xr) : 0.f;
            s_u[k][cc] = ok ? bw_ld(u, gi) : 0.f;
            s_dl[k][cc] = dl;
            if (backward) {
                const float zv = (ok && zg) ? bw_ld(zg, gi) : 0.f;
                const float dov = ok ? bw_ld(dout, gi) : 0.f;
                s_x[k][cc] = xr;
                s_z[k][cc] = zv;
                s_do[k][cc] = dov;
                s_dy[k][cc] = zg ? dov * zv * bw_sigmoid(zv) : dov;
            }
        }
        for (int i = tid; i < N * K; i += kBwdThreads) {
            const int nn = i / K, k = i % K;
            const int64_t t = t0 + k;
            const bool ok = t < L;
            s_B[nn][k] = ok ? bw_ld(Bg, (b * N + nn) * L + t) : 0.f;
            if (backward) s_C[nn][k] = ok ? bw_ld(Cg, (b * N + nn) * L + t) : 0.f;
        }
        __syncthreads();
    };

    // ---- pass 1: forward, checkpoint the state entering each chunk
    float h = 0.f;
    for (int64_t c = 0; c < nch; ++c) {
        stage(c, false);
        if (ch_ok) ckpt[((b * dim + d) * nch + c) * N + n] = h;
#pragma unroll 8
        for (int k = 0; k < K; ++k) h = expf(s_dl[k][cl] * An) * h + s_dl[k][cl] * s_B[n][k] * s_u[k][cl];
        __syncthreads();
    }

    // ---- pass 2: chunks in reverse
    float lam = 0.f, anext = 0.f, dA_acc = 0.f;
    for (int64_t c = nch - 1; c >= 0; --c) {
        stage(c, true);
        const int64_t t0 = c * K;
        const float h_in = ch_ok ? ckpt[((b * dim + d) * nch + c) * N + n] : 0.f;
        float hk[K];
        float hc = h_in;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            hc = expf(s_dl[k][cl] * An) * hc + s_dl[k][cl] * s_B[n][k] * s_u[k][cl];
            hk[k] = hc;
            const float yp = group_sum<N>(s_C[n][k] * hc);
            if (n == 0) s_y[k][cl] = yp + Dd * s_u[k][cl];
        }
#pragma unroll
        for (int k = K - 1; k >= 0; --k) {
            const float dl = s_dl[k][cl], uu = s_u[k][cl], dy = s_dy[k][cl];
            const float a = expf(dl * An);
            const float hprev = k > 0 ? hk[k - 1] : h_in;
            lam = s_C[n][k] * dy + anext * lam;
            // dC, dB terms summed over the warp's channels (lanes n, n+N, ...)
            float pc = dy * hk[k], pb = lam * dl * uu;
#pragma unroll
            for (int o = N; o < 32; o <<= 1) {
                pc += __shfl_xor_sync(0xffffffffu, pc, o);
                pb += __shfl_xor_sync(0xffffffffu, pb, o);
            }
            if (lane < N) {
                s_pC[warp][n][k] = pc;
                s_pB[warp][n][k] = pb;
            }
            const float dup = group_sum<N>(lam * dl * s_B[n][k]);
            const float ddp = group_sum<N>(lam * (An * a * hprev + s_B[n][k] * uu));
            if (n == 0) {
                s_du[k][cl] = Dd * dy + dup;
                s_dd[k][cl] = ddp;
            }
            dA_acc += lam * dl * a * hprev;
            anext = a;
        }
        __syncthreads();
        // per-(t, d) outputs of the chunk
        for (int i = tid; i < K * CC; i += kBwdThreads) {
            const int k = i / CC, cc = i % CC;
            const int64_t t = t0 + k, dd = d0 + cc;
            if (t >= L || dd >= dim) continue;
            const int64_t gi = (b * L + t) * dim + dd;
            const float ddl = s_dd[k][cc];
            const float dx = p.softplus ? ddl * bw_sigmoid(s_x[k][cc]) : ddl;
            bw_st(static_cast<T*>(p.du), gi, s_du[k][cc]);
            bw_st(static_cast<T*>(p.ddelta), gi, dx);
            atomicAdd(&s_db[cc], dx);
            atomicAdd(&s_dD[cc], s_dy[k][cc] * s_u[k][cc]);
            if (zg && p.dz) {
                const float zv = s_z[k][cc], sg = bw_sigmoid(zv);
                bw_st(static_cast<T*>(p.dz), gi, s_do[k][cc] * s_y[k][cc] * sg * (1.f + zv * (1.f - sg)));
            }
        }
        // dB, dC of the chunk: the warps' partials summed, one global atomic
        // per (state, step)
        for (int i = tid; i < N * K; i += kBwdThreads) {
            const int nn = i / K, k = i % K;
            const int64_t t = t0 + k;
            if (t >= L) continue;
            float sb = 0.f, sc = 0.f;
#pragma unroll
            for (int w = 0; w < kBwdThreads / 32; ++w) {
                sb += s_pB[w][nn][k];
                sc += s_pC[w][nn][k];
            }
            atomicAdd(p.dB + (b * N + nn) * L + t, sb);
            atomicAdd(p.dC + (b * N + nn) * L + t, sc);
        }
        __syncthreads();
    }
    if (ch_ok) atomicAdd(p.dA + d * N + n, dA_acc);
    for (int i = tid; i < CC; i += kBwdThreads) {
        if (d0 + i >= dim) continue;
        if (p.dD) atomicAdd(p.dD + d0 + i, s_dD[i]);
        if (p.dbias) atomicAdd(p.dbias + d0 + i, s_db[i]);
    }
}

template <typename T, int N>
cudaError_t launch_bwd_t(const BwdArgs& a, float* ckpt, cudaStream_t s) {
    constexpr int CC = (32 / N) * (kBwdThreads / 32);
    dim3 grid((unsigned)((a.dim + CC - 1) / CC), (unsigned)a.batch);
    scan_bwd_kernel<T, N><<<grid, kBwdThreads, 0, s>>>(a, ckpt);
    return cudaGetLastError();
}

}  // namespace

int64_t bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate) {
    const int k = bwd_chunk(dstate);
    return batch * dim * ((seqlen + k - 1) / k) * dstate * 4;
}

cudaError_t launch_scan_bwd(const BwdArgs& a, DType dt, void* workspace, cudaStream_t s) {
    // the accumulated gradients start from zero
    const int64_t N = a.dstate;
    cudaError_t e = cudaMemsetAsync(a.dA, 0, a.dim * N * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dB, 0, a.batch * N * a.seqlen * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dC, 0, a.batch * N * a.seqlen * 4, s);
    if (e == cudaSuccess && a.dD) e = cudaMemsetAsync(a.dD, 0, a.dim * 4, s);
    if (e == cudaSuccess && a.dbias) e = cudaMemsetAsync(a.dbias, 0, a.dim * 4, s);
    if (e != cudaSuccess) return e;
    float* ck = static_cast<float*>(workspace);
    const bool bf = dt == DType::BF16;
    switch (a.dstate) {
        case 4: return bf ? launch_bwd_t<__nv_bfloat16, 4>(a, ck, s) : launch_bwd_t<float, 4>(a, ck, s);
        case 8: return bf ? launch_bwd_t<__nv_bfloat16, 8>(a, ck, s) : launch_bwd_t<float, 8>(a, ck, s);
        case 16: return bf ? launch_bwd_t<__nv_bfloat16, 16>(a, ck, s) : launch_bwd_t<float, 16>(a, ck, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
