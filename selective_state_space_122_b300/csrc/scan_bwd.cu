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
// Work decomposition: a CTA owns CC channels of one batch row (four states
// per lane: N/4 lanes per channel, 4 warps) and the whole sequence.
//   pass 1: the forward recurrence, storing the state entering every K-step
//           chunk in the workspace;
//   pass 2: the chunks in reverse order: per chunk, stage u, delta_raw, z,
//           dout and B, C in shared memory, evaluate the per-(t, d) terms once,
//           recompute the chunk's states from its checkpoint into registers,
//           with their decays, then run the adjoint backwards over the chunk;
//           sums over a channel's states are in-lane sums plus warp shuffles
//           over its N/4 lanes; each lane's dB and dC terms go to its own
//           shared-memory slots, summed over the CTA's channels with 16-byte
//           loads and added to global memory once per chunk.
// dA, dB, dC, dD and dbias accumulate with atomics across CTAs and batch rows
// (the launcher zeroes them first).
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "device_memo.h"
#include "ssm_internal.cuh"

namespace ssm {

namespace {

constexpr int kBwdThreads = 128;   // 4 warps

// Layout of one CTA: four states per lane (G), R = N / 4 lanes per channel,
// 32 / R channels per warp, four warps; K steps per chunk.
template <int N>
struct BwdCfg {
    static constexpr int G = 4;
    static constexpr int R = N / G;
    static constexpr int CPW = 32 / R;
    static constexpr int CC = CPW * (kBwdThreads / 32);   // channels per CTA
    static constexpr int K = 8;
    // dynamic shared memory, float offsets
    static constexpr int T_CH = K * CC;                    // one per-(t, d) array
    static constexpr int O_U = 0, O_DL = T_CH, O_DY = 2 * T_CH, O_Y = 3 * T_CH, O_DU = 4 * T_CH, O_DD = 5 * T_CH;
    static constexpr int O_X = 6 * T_CH, O_Z = 7 * T_CH, O_DO = 8 * T_CH;
    static constexpr int O_B = 9 * T_CH, O_C = O_B + N * K;
    static constexpr int O_P = O_C + N * K;                // [K][lanes of the CTA][8]: dC (4), dB (4)
    static constexpr int O_DD_CH = O_P + K * kBwdThreads * 8;
    static constexpr int O_DB_CH = O_DD_CH + CC;
    static constexpr int FLOATS = O_DB_CH + CC;
    static constexpr int SMEM = FLOATS * 4;
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

// steps per chunk (the workspace holds the state entering every chunk)
__host__ __device__ constexpr int bwd_chunk(int) { return 8; }

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

// exp(x): the SFU exp2 for bf16 activations (relative error ~2^-22, far below
// the bf16 output rounding), the accurate library exp for float32.
template <bool kFast>
__device__ __forceinline__ float bw_exp(float x) {
    if constexpr (kFast) {
        float y;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
        return y;
    } else {
        return expf(x);
    }
}

// sum over the R lanes of one channel
template <int R>
__device__ __forceinline__ float chan_sum(float v) {
#pragma unroll
    for (int o = R / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// kTight: a register budget for four CTAs per SM (at most 128 registers a
// thread, a few hundred bytes of spills), taken when the grid would not fit
// the GPU in one wave otherwise; small grids keep every register.
template <typename T, int N, bool kTight>
__global__ void __launch_bounds__(kBwdThreads, kTight ? 4 : 1)
scan_bwd_kernel(const BwdArgs p, float* __restrict__ ckpt) {
    using CF = BwdCfg<N>;
    constexpr int K = CF::K, R = CF::R, CPW = CF::CPW, CC = CF::CC, G = CF::G;
    constexpr bool kFast = !std::is_same<T, float>::value;
    extern __shared__ __align__(16) float sm[];
    float* s_u = sm + CF::O_U;
    float* s_dl = sm + CF::O_DL;
    float* s_dy = sm + CF::O_DY;
    float* s_y = sm + CF::O_Y;
    float* s_du = sm + CF::O_DU;
    float* s_dd = sm + CF::O_DD;
    float* s_x = sm + CF::O_X;
    float* s_z = sm + CF::O_Z;
    float* s_do = sm + CF::O_DO;
    float* s_B = sm + CF::O_B;      // [K][N]
    float* s_C = sm + CF::O_C;
    float* s_P = sm + CF::O_P;      // [K][kBwdThreads][8]
    float* s_dDc = sm + CF::O_DD_CH;
    float* s_dbc = sm + CF::O_DB_CH;

    const T* u = static_cast<const T*>(p.u);
    const T* dr = static_cast<const T*>(p.delta);
    const T* Bg = static_cast<const T*>(p.B);
    const T* Cg = static_cast<const T*>(p.C);
    const T* zg = static_cast<const T*>(p.z);
    const T* dout = static_cast<const T*>(p.dout);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane % R;                       // states 4g .. 4g+3
    const int cl = warp * CPW + lane / R;         // channel within the CTA
    const int64_t b = blockIdx.y;
    // CTA -> (B/C group, block of CC channels within it): the CTAs of a group
    // cover its channels [grp * gch, dend) only, so every CTA reads and adds
    // to one B/C block
    // (channel indices stay below 2^31: the host rejects larger dims)
    const int gch = (int)p.gch;
    const int bpg = (gch + CC - 1) / CC;
    const int grp = (int)blockIdx.x / bpg;
    const int d0 = grp * gch + ((int)blockIdx.x - grp * bpg) * CC;
    const int dend = d0 + min(CC, (grp + 1) * gch - d0);
    const int64_t blk = b * p.ngroups + grp;
    const int64_t d = d0 + cl;
    const bool ch_ok = d < dend;
    const int64_t L = p.seqlen, dim = p.dim;
    const int64_t nch = (L + K - 1) / K;
    float An[G];
#pragma unroll
    for (int j = 0; j < G; ++j) An[j] = ch_ok ? p.A[d * N + G * g + j] : 0.f;
    const float Dd = (p.D && ch_ok) ? p.D[d] : 0.f;

    for (int i = tid; i < CC; i += kBwdThreads) s_dDc[i] = s_dbc[i] = 0.f;

    // A chunk's inputs are fetched into registers one chunk ahead (their
    // global-memory latency overlaps the previous chunk's work), then turned
    // into the per-(t, d) terms in shared memory.
    constexpr int IT = (K * CC + kBwdThreads - 1) / kBwdThreads;   // (t, d) items per thread
    constexpr int BT = (N * K + kBwdThreads - 1) / kBwdThreads;    // (n, t) items per thread
    struct Pre {
        float u[IT], xr[IT], z[IT], dov[IT], Bv[BT], Cv[BT];
        bool ok[IT];
    };
    auto fetch = [&](int64_t c, bool backward, Pre& r) {
        const int64_t t0 = c * K;
#pragma unroll
        for (int q = 0; q < IT; ++q) {
            const int i = tid + q * kBwdThreads;
            const int k = i / CC, cc = i % CC;
            const int64_t t = t0 + k, dd = d0 + cc;
            const bool ok = i < K * CC && t < L && dd < dend;
            const int64_t gi = (b * L + t) * dim + dd;
            r.ok[q] = ok;
            r.xr[q] = ok ? bw_ld(dr, gi) + (p.delta_bias ? p.delta_bias[dd] : 0.f) : 0.f;
            r.u[q] = ok ? bw_ld(u, gi) : 0.f;
            r.z[q] = (backward && ok && zg) ? bw_ld(zg, gi) : 0.f;
            r.dov[q] = (backward && ok) ? bw_ld(dout, gi) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < BT; ++q) {
            const int i = tid + q * kBwdThreads;
            const int nn = i / K, k = i % K;
            const int64_t t = t0 + k;
            const bool ok = i < N * K && t < L;
            r.Bv[q] = ok ? bw_ld(Bg, (blk * N + nn) * L + t) : 0.f;
            r.Cv[q] = (backward && ok) ? bw_ld(Cg, (blk * N + nn) * L + t) : 0.f;
        }
    };
    auto commit = [&](const Pre& r, bool backward) {
#pragma unroll
        for (int q = 0; q < IT; ++q) {
            const int i = tid + q * kBwdThreads;
            if (i >= K * CC) continue;
            const float xr = r.xr[q];
            s_u[i] = r.u[q];
            s_dl[i] = r.ok[q] ? (p.softplus ? bw_softplus(xr) : xr) : 0.f;
            if (backward) {
                s_x[i] = xr;
                s_z[i] = r.z[q];
                s_do[i] = r.dov[q];
                s_dy[i] = zg ? r.dov[q] * r.z[q] * bw_sigmoid(r.z[q]) : r.dov[q];
            }
        }
#pragma unroll
        for (int q = 0; q < BT; ++q) {
            const int i = tid + q * kBwdThreads;
            if (i >= N * K) continue;
            const int nn = i / K, k = i % K;
            s_B[k * N + nn] = r.Bv[q];
            if (backward) s_C[k * N + nn] = r.Cv[q];
        }
        __syncthreads();
    };

    // ---- pass 1: forward from h_{-1} (the given state, else zero),
    // checkpoint the state entering each chunk
    const float2 A01 = make_float2(An[0], An[1]), A23 = make_float2(An[2], An[3]);
    float2 h01 = make_float2(0.f, 0.f), h23 = make_float2(0.f, 0.f);
    if (p.h0 && ch_ok) {
        const float4 v = *reinterpret_cast<const float4*>(p.h0 + (b * dim + d) * N + G * g);
        h01 = make_float2(v.x, v.y);
        h23 = make_float2(v.z, v.w);
    }
    Pre pre;
    fetch(0, false, pre);
    for (int64_t c = 0; c < nch; ++c) {
        commit(pre, false);
        if (c + 1 < nch) fetch(c + 1, false, pre);
        if (ch_ok)
            *reinterpret_cast<float4*>(ckpt + ((b * dim + d) * nch + c) * N + G * g) =
                make_float4(h01.x, h01.y, h23.x, h23.y);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float dl = s_dl[k * CC + cl];
            const float2 dl2 = splat2(dl), du2 = splat2(dl * s_u[k * CC + cl]);
            const float4 Bq = *reinterpret_cast<const float4*>(s_B + k * N + G * g);
            const float2 e01 = mul2(dl2, A01), e23 = mul2(dl2, A23);
            h01 = fma2(make_float2(bw_exp<kFast>(e01.x), bw_exp<kFast>(e01.y)), h01, mul2(du2, make_float2(Bq.x, Bq.y)));
            h23 = fma2(make_float2(bw_exp<kFast>(e23.x), bw_exp<kFast>(e23.y)), h23, mul2(du2, make_float2(Bq.z, Bq.w)));
        }
        __syncthreads();
    }

    // ---- pass 2: chunks in reverse.  The adjoint "after" the last step is
    // dL/d last_state (zero when absent), carried into step L-1 with weight 1.
    float2 lam01 = make_float2(0.f, 0.f), lam23 = lam01, dA01 = lam01, dA23 = lam01;
    float2 an01 = make_float2(1.f, 1.f), an23 = an01;
    if (p.dlast && ch_ok) {
        const float4 v = *reinterpret_cast<const float4*>(p.dlast + (b * dim + d) * N + G * g);
        lam01 = make_float2(v.x, v.y);
        lam23 = make_float2(v.z, v.w);
    }
    fetch(nch - 1, true, pre);
    for (int64_t c = nch - 1; c >= 0; --c) {
        commit(pre, true);
        if (c > 0) fetch(c - 1, true, pre);
        const int64_t t0 = c * K;
        float2 hin01, hin23;
        {
            const float4 v = ch_ok ? *reinterpret_cast<const float4*>(ckpt + ((b * dim + d) * nch + c) * N + G * g)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            hin01 = make_float2(v.x, v.y);
            hin23 = make_float2(v.z, v.w);
        }
        // recompute the chunk's states and decays (pairs of states per packed
        // operation); y_t for dz
        float2 hk01[K], hk23[K], ak01[K], ak23[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float dl = s_dl[k * CC + cl], uu = s_u[k * CC + cl];
            const float2 dl2 = splat2(dl), du2 = splat2(dl * uu);
            const float4 Bq = *reinterpret_cast<const float4*>(s_B + k * N + G * g);
            const float4 Cq = *reinterpret_cast<const float4*>(s_C + k * N + G * g);
            const float2 e01 = mul2(dl2, A01), e23 = mul2(dl2, A23);
            ak01[k] = make_float2(bw_exp<kFast>(e01.x), bw_exp<kFast>(e01.y));
            ak23[k] = make_float2(bw_exp<kFast>(e23.x), bw_exp<kFast>(e23.y));
            hk01[k] = fma2(ak01[k], k > 0 ? hk01[k - 1] : hin01, mul2(du2, make_float2(Bq.x, Bq.y)));
            hk23[k] = fma2(ak23[k], k > 0 ? hk23[k - 1] : hin23, mul2(du2, make_float2(Bq.z, Bq.w)));
            const float2 yv = fma2(make_float2(Cq.z, Cq.w), hk23[k], mul2(make_float2(Cq.x, Cq.y), hk01[k]));
            const float yp = chan_sum<R>(yv.x + yv.y);
            if (g == 0) s_y[k * CC + cl] = yp + Dd * uu;
        }
        // the adjoint, backwards over the chunk
#pragma unroll
        for (int k = K - 1; k >= 0; --k) {
            const float dl = s_dl[k * CC + cl], uu = s_u[k * CC + cl], dy = s_dy[k * CC + cl];
            const float2 dl2 = splat2(dl), uu2 = splat2(uu), dy2 = splat2(dy);
            const float4 Bq = *reinterpret_cast<const float4*>(s_B + k * N + G * g);
            const float4 Cq = *reinterpret_cast<const float4*>(s_C + k * N + G * g);
            const float2 B01 = make_float2(Bq.x, Bq.y), B23 = make_float2(Bq.z, Bq.w);
            const float2 hp01 = k > 0 ? hk01[k - 1] : hin01, hp23 = k > 0 ? hk23[k - 1] : hin23;
            lam01 = fma2(an01, lam01, mul2(make_float2(Cq.x, Cq.y), dy2));
            lam23 = fma2(an23, lam23, mul2(make_float2(Cq.z, Cq.w), dy2));
            const float2 ld01 = mul2(lam01, dl2), ld23 = mul2(lam23, dl2);       // lambda Delta
            const float2 pc01 = mul2(dy2, hk01[k]), pc23 = mul2(dy2, hk23[k]);   // dC terms
            const float2 pb01 = mul2(ld01, uu2), pb23 = mul2(ld23, uu2);         // dB terms
            const float2 duv = fma2(ld23, B23, mul2(ld01, B01));
            // A a h_{t-1} + B u, per state
            const float2 t01 = fma2(mul2(A01, ak01[k]), hp01, mul2(B01, uu2));
            const float2 t23 = fma2(mul2(A23, ak23[k]), hp23, mul2(B23, uu2));
            const float2 ddv = fma2(lam23, t23, mul2(lam01, t01));
            dA01 = fma2(mul2(ld01, ak01[k]), hp01, dA01);
            dA23 = fma2(mul2(ld23, ak23[k]), hp23, dA23);
            an01 = ak01[k];
            an23 = ak23[k];
            float4* pp = reinterpret_cast<float4*>(s_P + ((size_t)k * kBwdThreads + tid) * 8);
            pp[0] = make_float4(pc01.x, pc01.y, pc23.x, pc23.y);
            pp[1] = make_float4(pb01.x, pb01.y, pb23.x, pb23.y);
            const float dup = chan_sum<R>(duv.x + duv.y);
            const float ddp = chan_sum<R>(ddv.x + ddv.y);
            if (g == 0) {
                s_du[k * CC + cl] = fmaf(Dd, dy, dup);
                s_dd[k * CC + cl] = ddp;
            }
        }
        __syncthreads();
        // per-(t, d) outputs of the chunk
        for (int i = tid; i < K * CC; i += kBwdThreads) {
            const int k = i / CC, cc = i % CC;
            const int64_t t = t0 + k, dd = d0 + cc;
            if (t >= L || dd >= dend) continue;
            const int64_t gi = (b * L + t) * dim + dd;
            const float ddl = s_dd[i];
            const float dx = p.softplus ? ddl * bw_sigmoid(s_x[i]) : ddl;
            bw_st(static_cast<T*>(p.du), gi, s_du[i]);
            bw_st(static_cast<T*>(p.ddelta), gi, dx);
            atomicAdd(&s_dbc[cc], dx);
            atomicAdd(&s_dDc[cc], s_dy[i] * s_u[i]);
            if (zg && p.dz) {
                const float zv = s_z[i], sg = bw_sigmoid(zv);
                bw_st(static_cast<T*>(p.dz), gi, s_do[i] * s_y[i] * sg * (1.f + zv * (1.f - sg)));
            }
        }
        // dB, dC of the chunk: every (step, state quad, B-or-C) summed over the
        // CTA's channels (parts of the channel range per thread when there are
        // fewer such sums than threads), then added to global memory
        {
            constexpr int SUMS = K * R * 2;
            constexpr int PARTS = SUMS >= kBwdThreads ? 1 : kBwdThreads / SUMS;
            constexpr int CPP = CC / PARTS;
            for (int i = tid; i < SUMS * PARTS; i += kBwdThreads) {
                const int part = i / SUMS, sidx = i % SUMS;
                const int k = sidx / (2 * R), gq = (sidx / 2) % R, which = sidx % 2;
                const int64_t t = t0 + k;
                if (t >= L) continue;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int cc = part * CPP; cc < (part + 1) * CPP; ++cc) {
                    // the lane of channel cc holding state quad gq
                    const int ln = (cc / CPW) * 32 + (cc % CPW) * R + gq;
                    const float4 v = reinterpret_cast<const float4*>(s_P + ((size_t)k * kBwdThreads + ln) * 8)[which];
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
                float* dst = (which ? p.dB : p.dC) + (blk * N + G * gq) * L + t;
                atomicAdd(dst, acc.x);
                atomicAdd(dst + L, acc.y);
                atomicAdd(dst + 2 * L, acc.z);
                atomicAdd(dst + 3 * L, acc.w);
            }
        }
        __syncthreads();
    }
    // h_0 = a_0 h_{-1} + ...: the adjoint of the initial state is a_0 lambda_0
    if (p.dh0 && ch_ok)
        *reinterpret_cast<float4*>(p.dh0 + (b * dim + d) * N + G * g) =
            make_float4(an01.x * lam01.x, an01.y * lam01.y, an23.x * lam23.x, an23.y * lam23.y);
    if (ch_ok) {
        float* da = p.dA + d * N + G * g;
        atomicAdd(da, dA01.x);
        atomicAdd(da + 1, dA01.y);
        atomicAdd(da + 2, dA23.x);
        atomicAdd(da + 3, dA23.y);
    }
    for (int i = tid; i < CC; i += kBwdThreads) {
        if (d0 + i >= dend) continue;
        if (p.dD) atomicAdd(p.dD + d0 + i, s_dDc[i]);
        if (p.dbias) atomicAdd(p.dbias + d0 + i, s_dbc[i]);
    }
}

template <typename T, int N>
cudaError_t launch_bwd_t(const BwdArgs& a, float* ckpt, int sms, cudaStream_t s) {
    using CF = BwdCfg<N>;
    // shared-memory size of both instantiations, set once per device
    static DeviceMemo memo;
    int dev = 0, set = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    cudaError_t err = cudaSuccess;
    if (!memo.get(dev, [&](int& r) {
            err = cudaFuncSetAttribute(scan_bwd_kernel<T, N, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       CF::SMEM);
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(scan_bwd_kernel<T, N, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           CF::SMEM);
            r = 1;
            return err == cudaSuccess;
        }, &set))
        return err;
    const int64_t gx = a.ngroups * ((a.gch + CF::CC - 1) / CF::CC);
    if (gx > 0x7fffffff) return cudaErrorInvalidValue;
    dim3 grid((unsigned)gx, (unsigned)a.batch);
    // with every register a thread, about two CTAs fit an SM
    if ((int64_t)grid.x * grid.y > 2 * (int64_t)sms)
        scan_bwd_kernel<T, N, true><<<grid, kBwdThreads, CF::SMEM, s>>>(a, ckpt);
    else
        scan_bwd_kernel<T, N, false><<<grid, kBwdThreads, CF::SMEM, s>>>(a, ckpt);
    return cudaGetLastError();
}

}  // namespace

int64_t bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate) {
    const int k = bwd_chunk(dstate);
    return batch * dim * ((seqlen + k - 1) / k) * dstate * 4;
}

cudaError_t launch_scan_bwd(const BwdArgs& a, DType dt, void* workspace, int sms, cudaStream_t s) {
    // the accumulated gradients start from zero
    const int64_t N = a.dstate;
    cudaError_t e = cudaMemsetAsync(a.dA, 0, a.dim * N * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dB, 0, a.batch * a.ngroups * N * a.seqlen * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dC, 0, a.batch * a.ngroups * N * a.seqlen * 4, s);
    if (e == cudaSuccess && a.dD) e = cudaMemsetAsync(a.dD, 0, a.dim * 4, s);
    if (e == cudaSuccess && a.dbias) e = cudaMemsetAsync(a.dbias, 0, a.dim * 4, s);
    if (e != cudaSuccess) return e;
    float* ck = static_cast<float*>(workspace);
    const bool bf = dt == DType::BF16;
    switch (a.dstate) {
        case 4: return bf ? launch_bwd_t<__nv_bfloat16, 4>(a, ck, sms, s) : launch_bwd_t<float, 4>(a, ck, sms, s);
        case 8: return bf ? launch_bwd_t<__nv_bfloat16, 8>(a, ck, sms, s) : launch_bwd_t<float, 8>(a, ck, sms, s);
        case 16: return bf ? launch_bwd_t<__nv_bfloat16, 16>(a, ck, sms, s) : launch_bwd_t<float, 16>(a, ck, sms, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
