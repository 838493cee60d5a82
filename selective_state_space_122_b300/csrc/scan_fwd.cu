// scan_fwd.cu -- full-sequence selective scan for sm_103a.
//
// Computes, per (batch, channel), the recurrence of the Mamba selective SSM
// ("Mamba: Selective State Space Models" README: "State Space Model",
// "Selective Mechanism", "Efficient Scan"):
//     Delta_t = softplus(delta_raw_t + delta_bias)
//     h_t     = exp(Delta_t A) * h_{t-1} + Delta_t B_t u_t
//     out_t   = (C_t . h_t + D u_t) * silu(z_t)
//
// Work layout (one CTA = CW consecutive channels of one batch row, walking
// the whole sequence chunk by chunk; the state never leaves the chip):
//   * lane = (c, g): channel c of the CTA and state group g (G consecutive
//     states; the R = N / G lanes of a channel are adjacent lanes);
//   * a chunk of TC = S * K steps is cut into S sub-chunks of K steps, one
//     per warp;
//   * S == 1: the lane walks every step of the chunk with its states in
//     registers (the sequential scan of "Efficient Scan");
//   * S > 1: each warp first runs its sub-chunk from a zero state, keeping
//     exp(Delta A) and Delta B u of every step in registers, and publishes
//     the sub-chunk summary (prod exp(Delta A), local end state).  Each lane
//     then folds the summaries of the earlier sub-chunks into the chunk's
//     incoming state with the associative operator
//         (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2)
//     ("Efficient Scan", parallel scan) and reruns its sub-chunk from the
//     true incoming state over the stored values.  No exponential is
//     evaluated twice; the last warp's final state is the next chunk's
//     incoming state.
//   * per (t, d) work (softplus, Delta u, D u, silu(z)) is done once per
//     (t, d) into shared memory; the raw activations and B/C of chunk k+1
//     are fetched into registers while chunk k is computed;
//   * y_t = sum over the R lanes of a channel: each lane keeps K partial
//     sums and a transposed butterfly leaves K / R finished sums per lane;
//   * the inner loop uses packed f32x2 multiplies / FMAs (two states per
//     instruction) and one SFU ex2 per (t, state).
//
// Shared-memory layouts (chosen so warp-wide accesses stay at one wavefront
// per 128 bytes): Delta / Delta u and D u / silu(z) as [channel][t] float2
// rows (one 16-byte load = two steps); B and C as float rows, one per state,
// t-contiguous, with the state of row j * R + g being g * G + j so the R
// lanes of a channel read rows in distinct bank groups.
#include <cstdint>
#include <type_traits>

#include "device_memo.h"
#include "ssm_internal.cuh"

namespace ssm {
namespace {

template <bool kFast>
__device__ __forceinline__ float2 exp2_2(float2 x) {
    return make_float2(decay_exp2<kFast>(x.x), decay_exp2<kFast>(x.y));
}

// ------------------------------------------------------------- configuration

template <typename T, int N_, int G_, int S_, int K_>
struct Cfg {
    static constexpr int N = N_, G = G_, S = S_, K = K_;
    static constexpr int R = N / G;                 // lanes per channel
    static constexpr int CW = 32 / R;               // channels per CTA
    static constexpr int THREADS = 32 * S;
    static constexpr int TC = S * K;                // steps per chunk
    static constexpr bool kSplit = S > 1;
    static constexpr int V = 16 / (int)sizeof(T);   // elements per 16-byte vector
    static constexpr int PAIRS = TC * CW / 2;       // (t, channel pair) prologue items per chunk
    static constexpr int PAIRS_PT = (PAIRS + THREADS - 1) / THREADS;
    static constexpr int BCV = 2 * N * TC / V;      // 16-byte vectors of B and C per chunk
    static constexpr int BCV_PT = (BCV + THREADS - 1) / THREADS;
    static constexpr int KR = K / R;                // finished sums per lane
    // row strides (floats): TCD for the float2 [c][t] rows, TCB for B/C rows
    static constexpr int TCD = 2 * TC + 4;
    static constexpr int TCB = TC + 4;
    static_assert(G % 4 == 0, "states per lane come in 16-byte groups");
    static_assert(N % G == 0 && R <= 16, "lane layout");
    static_assert(K % 4 == 0 && K % R == 0 && (R == 1 || KR % 2 == 0), "steps per lane");
    static_assert(TC % V == 0, "B/C chunk rows are whole vectors");
    // shared memory, in floats
    static constexpr int OFF_DD = 0;                       // [CW][TCD]  (Delta, Delta u) per t
    static constexpr int OFF_SG = OFF_DD + CW * TCD;       // [CW][TCD]  (D u, silu z) per t
    static constexpr int OFF_B = OFF_SG + CW * TCD;        // [N][TCB]
    static constexpr int OFF_C = OFF_B + N * TCB;          // [N][TCB]
    static constexpr int OFF_P = OFF_C + N * TCB;          // [S][CW][N]   sub-chunk decay products
    static constexpr int OFF_H = OFF_P + (kSplit ? S * CW * N : 0);    // [S][CW][N] local end states
    static constexpr int OFF_CAR = OFF_H + (kSplit ? S * CW * N : 0);  // [2][CW][N] chunk carries
    static constexpr int OFF_OUT = OFF_CAR + (kSplit ? 2 * CW * N : 0);  // T [TC][CW]
    static constexpr int SMEM_FLOATS = OFF_OUT + (TC * CW * (int)sizeof(T) + 15) / 16 * 4;
    static constexpr size_t SMEM_BYTES = sizeof(float) * SMEM_FLOATS;
    // B/C row of state n
    static __device__ __forceinline__ int brow(int n) { return (n % G) * R + n / G; }
};

// Per-launch facts the kernel needs beyond ScanArgs.
struct Geo {
    int vec_x;   // u/delta/z/out rows allow paired (2-element) accesses
    int vec_bc;  // B/C rows allow 16-byte accesses
    int64_t bpg; // CTAs per channel group (B/C block): the CTAs of a group
                 // cover its channels only, so every CTA reads one B/C block
};

template <typename T>
struct Pair;  // two consecutive elements
template <>
struct Pair<__nv_bfloat16> {
    using type = __nv_bfloat162;
    static __device__ __forceinline__ float2 f(type v) { return __bfloat1622float2(v); }
    static __device__ __forceinline__ type make(float a, float b) { return __floats2bfloat162_rn(a, b); }
};
template <>
struct Pair<float> {
    using type = float2;
    static __device__ __forceinline__ float2 f(type v) { return v; }
    static __device__ __forceinline__ type make(float a, float b) { return make_float2(a, b); }
};

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// kGrouped: B and C per channel group (the CTAs of a group cover its channels
// only); without it the CTA's channels are a plain block of the row.
template <typename CF, typename T, bool kFast, bool kGrouped>
struct ScanKernel {
    using PT = typename Pair<T>::type;
    static constexpr int N = CF::N, G = CF::G, R = CF::R, CW = CF::CW, K = CF::K;
    [[maybe_unused]] static constexpr int S = CF::S;
    static constexpr int TC = CF::TC, V = CF::V, TCD = CF::TCD, TCB = CF::TCB, KR = CF::KR;
    static constexpr int THREADS = CF::THREADS;

    // ---- raw inputs of one chunk, held in registers between fetch and use
    struct Regs {
        PT u[CF::PAIRS_PT], dl[CF::PAIRS_PT], z[CF::PAIRS_PT];
        uint4 bc[CF::BCV_PT];
    };

    // Per-thread constants of the prologue's channel pair (a thread handles
    // the same pair in every chunk because THREADS is a multiple of CW / 2).
    struct PairConst {
        float2 bias, dsk;
        bool ok0, ok1;
    };

    // channels [.., dend) of row `row` (row stride dim)
    static __device__ __forceinline__ PT load_pair(const T* base, int64_t row, int64_t d, int64_t dim,
                                                   int64_t dend, int64_t L, bool vec) {
        if (row < L && d + 1 < dend && vec) return *reinterpret_cast<const PT*>(base + row * dim + d);
        float a = 0.f, b = 0.f;
        if (row < L) {
            if (d < dend) a = to_f32(base[row * dim + d]);
            if (d + 1 < dend) b = to_f32(base[row * dim + d + 1]);
        }
        return Pair<T>::make(a, b);
    }

    // blk: the B/C block (batch row * ngroups + group) of the CTA's channels
    static __device__ __forceinline__ void fetch(Regs& r, const ScanArgs& p, const Geo& geo, int64_t b,
                                                 int64_t blk, int64_t d0, int64_t dend, int64_t t0, int tid) {
        const int64_t L = p.seqlen, dim = p.dim;
        const T* u = static_cast<const T*>(p.u) + b * L * dim;
        const T* dl = static_cast<const T*>(p.delta) + b * L * dim;
        const T* zp = p.z ? static_cast<const T*>(p.z) + b * L * dim : nullptr;
#pragma unroll
        for (int k = 0; k < CF::PAIRS_PT; ++k) {
            const int idx = tid + k * THREADS;
            if (CF::PAIRS % THREADS == 0 || idx < CF::PAIRS) {
                const int t = idx / (CW / 2), cp = idx % (CW / 2);
                const int64_t row = t0 + t, d = d0 + 2 * cp;
                r.u[k] = load_pair(u, row, d, dim, dend, L, geo.vec_x);
                r.dl[k] = load_pair(dl, row, d, dim, dend, L, geo.vec_x);
                r.z[k] = zp ? load_pair(zp, row, d, dim, dend, L, geo.vec_x) : Pair<T>::make(0.f, 0.f);
            }
        }
        const T* Bb = static_cast<const T*>(p.B) + blk * N * L;
        const T* Cb = static_cast<const T*>(p.C) + blk * N * L;
#pragma unroll
        for (int k = 0; k < CF::BCV_PT; ++k) {
            const int idx = tid + k * THREADS;
            if (CF::BCV % THREADS == 0 || idx < CF::BCV) {
                const int which = idx / (N * TC / V);
                const int rem = idx % (N * TC / V);
                const int n = rem / (TC / V), tv = rem % (TC / V);
                const T* src = (which ? Cb : Bb) + (int64_t)n * L;
                const int64_t t = t0 + (int64_t)tv * V;
                if (geo.vec_bc && t + V <= L) {
                    r.bc[k] = *reinterpret_cast<const uint4*>(src + t);
                } else {
                    union {
                        uint4 v;
                        T e[V];
                    } w;
#pragma unroll
                    for (int j = 0; j < V; ++j) w.e[j] = (t + j < L) ? src[t + j] : from_f32<T>(0.f);
                    r.bc[k] = w.v;
                }
            }
        }
    }

    // ---- per-(t, d) prologue from registers into shared memory
    static __device__ __forceinline__ void prologue(const Regs& r, const PairConst& pc, float* sm,
                                                    const ScanArgs& p, int64_t t0, int tid) {
        float* s_dd = sm + CF::OFF_DD;
        float* s_sg = sm + CF::OFF_SG;
#pragma unroll
        for (int k = 0; k < CF::PAIRS_PT; ++k) {
            const int idx = tid + k * THREADS;
            if (CF::PAIRS % THREADS == 0 || idx < CF::PAIRS) {
                const int t = idx / (CW / 2), cp = idx % (CW / 2);
                const bool row_ok = t0 + t < p.seqlen;
                const float2 uv = Pair<T>::f(r.u[k]);
                const float2 zv = Pair<T>::f(r.z[k]);
                const float2 x = add2(Pair<T>::f(r.dl[k]), pc.bias);
                float2 dlt = p.softplus ? softplus_f2<kFast>(x) : x;
                // padded steps / channels: Delta = 0 leaves the state unchanged
                dlt.x = (row_ok && pc.ok0) ? dlt.x : 0.f;
                dlt.y = (row_ok && pc.ok1) ? dlt.y : 0.f;
                const float2 du = mul2(dlt, uv);
                const float2 skip = mul2(pc.dsk, uv);
                const float2 gate = p.z ? silu_f2<kFast>(zv) : splat2(1.f);
                const int c = 2 * cp;
                *reinterpret_cast<float2*>(s_dd + c * TCD + 2 * t) = make_float2(dlt.x, du.x);
                *reinterpret_cast<float2*>(s_dd + (c + 1) * TCD + 2 * t) = make_float2(dlt.y, du.y);
                *reinterpret_cast<float2*>(s_sg + c * TCD + 2 * t) = make_float2(skip.x, gate.x);
                *reinterpret_cast<float2*>(s_sg + (c + 1) * TCD + 2 * t) = make_float2(skip.y, gate.y);
            }
        }
        float* s_B = sm + CF::OFF_B;
        float* s_C = sm + CF::OFF_C;
#pragma unroll
        for (int k = 0; k < CF::BCV_PT; ++k) {
            const int idx = tid + k * THREADS;
            if (CF::BCV % THREADS == 0 || idx < CF::BCV) {
                const int which = idx / (N * TC / V);
                const int rem = idx % (N * TC / V);
                const int n = rem / (TC / V), tv = rem % (TC / V);
                float* dst = (which ? s_C : s_B) + CF::brow(n) * TCB + tv * V;
                union {
                    uint4 v;
                    T e[V];
                } w;
                w.v = r.bc[k];
#pragma unroll
                for (int j = 0; j < V; j += 4)
                    st4(dst + j, make_float4(to_f32(w.e[j]), to_f32(w.e[j + 1]), to_f32(w.e[j + 2]),
                                             to_f32(w.e[j + 3])));
            }
        }
    }

    // ---- out tile (shared) -> global, pairs of channels per access
    static __device__ __forceinline__ void store_out(const float* sm, const ScanArgs& p, const Geo& geo,
                                                     int64_t b, int64_t d0, int64_t dend, int64_t t0, int tid) {
        const T* s_out = reinterpret_cast<const T*>(sm + CF::OFF_OUT);
        T* out = static_cast<T*>(p.out) + b * p.seqlen * p.dim;
#pragma unroll
        for (int k = 0; k < CF::PAIRS_PT; ++k) {
            const int idx = tid + k * THREADS;
            if (CF::PAIRS % THREADS == 0 || idx < CF::PAIRS) {
                const int t = idx / (CW / 2), cp = idx % (CW / 2);
                const int64_t row = t0 + t, d = d0 + 2 * cp;
                if (row < p.seqlen) {
                    const PT v = *reinterpret_cast<const PT*>(s_out + t * CW + 2 * cp);
                    if (geo.vec_x && d + 1 < dend) {
                        *reinterpret_cast<PT*>(out + row * p.dim + d) = v;
                    } else {
                        const float2 f = Pair<T>::f(v);
                        if (d < dend) out[row * p.dim + d] = from_f32<T>(f.x);
                        if (d + 1 < dend) out[row * p.dim + d + 1] = from_f32<T>(f.y);
                    }
                }
            }
        }
    }

    // ---- y: transposed butterfly over the R lanes of a channel.  After all
    // levels v[0..K/R) of lane g hold the full sums of steps g*K/R + r.
    template <int M, int LEN>
    static __device__ __forceinline__ void reduce_level(float (&v)[K], int g) {
        if constexpr (M >= 1) {
            const bool upper = (g & M) != 0;
#pragma unroll
            for (int r = 0; r < LEN / 2; ++r) {
                const float send = upper ? v[r] : v[r + LEN / 2];
                const float keep = upper ? v[r + LEN / 2] : v[r];
                v[r] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            reduce_level<M / 2, LEN / 2>(v, g);
        }
    }

    // ---- finished sums -> gated outputs in the shared out tile
    static __device__ __forceinline__ void write_y(const float (&v)[K], float* sm, int t_first, int c) {
        const float* s_sg = sm + CF::OFF_SG + c * TCD;
        T* s_out = reinterpret_cast<T*>(sm + CF::OFF_OUT);
#pragma unroll
        for (int r = 0; r < KR; r += 2) {
            const int t = t_first + r;
            const float4 sg = ld4(s_sg + 2 * t);  // (skip_t, gate_t, skip_t+1, gate_t+1)
            const float2 y = mul2(add2(make_float2(v[r], v[r + 1]), make_float2(sg.x, sg.z)),
                                  make_float2(sg.y, sg.w));
            s_out[t * CW + c] = from_f32<T>(y.x);
            s_out[(t + 1) * CW + c] = from_f32<T>(y.y);
        }
    }

    // ---- one direct sweep over steps [t_first, t_first + K) from state h,
    // producing the partial y sums of this lane's states in v.  B and C are
    // read SW steps at a time (one 8- or 16-byte load per state and array).
    static constexpr int SW = G <= 8 ? 4 : 2;
    using VecSW = typename std::conditional<SW == 4, float4, float2>::type;

    static __device__ __forceinline__ void sweep_direct(float2 (&h)[G / 2], const float2 (&A2)[G / 2],
                                                        const float* sm, int c, int g, float (&v)[K]) {
        const float* s_dd = sm + CF::OFF_DD + c * TCD;
        const float* s_B = sm + CF::OFF_B;
        const float* s_C = sm + CF::OFF_C;
#pragma unroll
        for (int i0 = 0; i0 < K; i0 += SW) {
            VecSW bq[G], cq[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                bq[j] = *reinterpret_cast<const VecSW*>(s_B + (j * R + g) * TCB + i0);
                cq[j] = *reinterpret_cast<const VecSW*>(s_C + (j * R + g) * TCB + i0);
            }
#pragma unroll
            for (int i2 = 0; i2 < SW; i2 += 2) {
                const float4 dd = ld4(s_dd + 2 * (i0 + i2));  // (Delta, Delta u) x two steps
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    const float2 dA = exp2_2<kFast>(mul2(splat2(dd.x), A2[j]));
                    const float2 bv = make_float2(comp(bq[2 * j], i2), comp(bq[2 * j + 1], i2));
                    h[j] = fma2(dA, h[j], mul2(splat2(dd.y), bv));
                    acc0 = fma2(make_float2(comp(cq[2 * j], i2), comp(cq[2 * j + 1], i2)), h[j], acc0);
                }
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    const float2 dA = exp2_2<kFast>(mul2(splat2(dd.z), A2[j]));
                    const float2 bv = make_float2(comp(bq[2 * j], i2 + 1), comp(bq[2 * j + 1], i2 + 1));
                    h[j] = fma2(dA, h[j], mul2(splat2(dd.w), bv));
                    acc1 = fma2(make_float2(comp(cq[2 * j], i2 + 1), comp(cq[2 * j + 1], i2 + 1)), h[j], acc1);
                }
                const float2 pr = add2(make_float2(acc0.x, acc1.x), make_float2(acc0.y, acc1.y));
                v[i0 + i2] = pr.x;
                v[i0 + i2 + 1] = pr.y;
            }
        }
    }

    // ---- split layouts, pass 1: local scan of this warp's sub-chunk from a
    // zero state, keeping exp(Delta A) and Delta B u; returns sum of Delta.
    static __device__ __forceinline__ float sweep_local(float2 (&dA)[K][G / 2], float2 (&dBu)[K][G / 2],
                                                        float2 (&hl)[G / 2], const float2 (&A2)[G / 2],
                                                        const float* sm, int tf, int c, int g) {
        const float* s_dd = sm + CF::OFF_DD + c * TCD;
        const float* s_B = sm + CF::OFF_B;
        float2 sdl = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < G / 2; ++j) hl[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i0 = 0; i0 < K; i0 += 4) {
            float4 bq[G];
#pragma unroll
            for (int j = 0; j < G; ++j) bq[j] = ld4(s_B + (j * R + g) * TCB + tf + i0);
#pragma unroll
            for (int i2 = 0; i2 < 4; i2 += 2) {
                const float4 dd = ld4(s_dd + 2 * (tf + i0 + i2));
                sdl = add2(sdl, make_float2(dd.x, dd.z));
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int i = i0 + i2 + s;
                    const float dlt = s ? dd.z : dd.x, du = s ? dd.w : dd.y;
#pragma unroll
                    for (int j = 0; j < G / 2; ++j) {
                        dA[i][j] = exp2_2<kFast>(mul2(splat2(dlt), A2[j]));
                        dBu[i][j] = mul2(splat2(du),
                                         make_float2(comp(bq[2 * j], i2 + s), comp(bq[2 * j + 1], i2 + s)));
                        hl[j] = fma2(dA[i][j], hl[j], dBu[i][j]);
                    }
                }
            }
        }
        return sdl.x + sdl.y;
    }

    // ---- split layouts, pass 2: rerun the sub-chunk from its true incoming
    // state h over the stored values, producing the partial y sums.
    static __device__ __forceinline__ void sweep_replay(const float2 (&dA)[K][G / 2],
                                                        const float2 (&dBu)[K][G / 2], float2 (&h)[G / 2],
                                                        const float* sm, int tf, int g, float (&v)[K]) {
        const float* s_C = sm + CF::OFF_C;
#pragma unroll
        for (int i0 = 0; i0 < K; i0 += 4) {
            float4 cq[G];
#pragma unroll
            for (int j = 0; j < G; ++j) cq[j] = ld4(s_C + (j * R + g) * TCB + tf + i0);
#pragma unroll
            for (int i1 = 0; i1 < 4; i1 += 2) {
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    h[j] = fma2(dA[i0 + i1][j], h[j], dBu[i0 + i1][j]);
                    acc0 = fma2(make_float2(comp(cq[2 * j], i1), comp(cq[2 * j + 1], i1)), h[j], acc0);
                }
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    h[j] = fma2(dA[i0 + i1 + 1][j], h[j], dBu[i0 + i1 + 1][j]);
                    acc1 = fma2(make_float2(comp(cq[2 * j], i1 + 1), comp(cq[2 * j + 1], i1 + 1)), h[j], acc1);
                }
                const float2 pr = add2(make_float2(acc0.x, acc1.x), make_float2(acc0.y, acc1.y));
                v[i0 + i1] = pr.x;
                v[i0 + i1 + 1] = pr.y;
            }
        }
    }

    static __device__ void run(const ScanArgs& p, const Geo& geo) {
        extern __shared__ __align__(16) float sm[];
        const int tid = threadIdx.x;
        const int warp = tid >> 5, lane = tid & 31;
        const int g = lane % R;
        const int c = lane / R;
        const int64_t b = blockIdx.y;
        // CTA -> (channel group, block of CW channels within the group); the
        // host keeps dim below 2^31, so channel indices fit 32 bits
        int64_t d0, dend, blk;
        if constexpr (kGrouped) {
            const int gch = (int)p.gch, bpg = (int)geo.bpg;
            const int grp = (int)blockIdx.x / bpg;
            const int c0 = grp * gch + ((int)blockIdx.x - grp * bpg) * CW;
            d0 = c0;
            dend = c0 + min(CW, (grp + 1) * gch - c0);
            blk = b * p.ngroups + grp;
        } else {
            d0 = (int64_t)blockIdx.x * CW;
            dend = p.dim;
            blk = b;
        }
        const int64_t d = d0 + c;
        const bool valid = d < dend;
        const int64_t L = p.seqlen;
        const int64_t nchunks = (L + TC - 1) / TC;

        // decay exponents A * log2(e) of this lane's states g*G + (2j, 2j+1)
        float2 A2[G / 2];
#pragma unroll
        for (int j = 0; j < G / 2; ++j) {
            const float a0 = valid ? p.A[d * N + g * G + 2 * j] : 0.f;
            const float a1 = valid ? p.A[d * N + g * G + 2 * j + 1] : 0.f;
            A2[j] = make_float2(a0 * kLog2e, a1 * kLog2e);
        }

        PairConst pc;
        {
            const int cp = tid % (CW / 2);
            const int64_t dp = d0 + 2 * cp;
            pc.ok0 = dp < dend;
            pc.ok1 = dp + 1 < dend;
            pc.bias = make_float2((p.delta_bias && pc.ok0) ? p.delta_bias[dp] : 0.f,
                                  (p.delta_bias && pc.ok1) ? p.delta_bias[dp + 1] : 0.f);
            pc.dsk = make_float2((p.D && pc.ok0) ? p.D[dp] : 0.f, (p.D && pc.ok1) ? p.D[dp + 1] : 0.f);
        }

        // state before the first step: the caller's initial state, else zero
        float2 h[G / 2];
#pragma unroll
        for (int j = 0; j < G / 2; ++j) {
            const float* h0 = p.h0 + (b * p.dim + d) * N + g * G + 2 * j;
            h[j] = (p.h0 && valid) ? make_float2(h0[0], h0[1]) : make_float2(0.f, 0.f);
        }
        if constexpr (CF::kSplit) {
            float* s_car = sm + CF::OFF_CAR;
            for (int i = tid; i < CW * N; i += THREADS) {
                const int64_t dc = d0 + i / N;
                s_car[i] = (p.h0 && dc < dend) ? p.h0[(b * p.dim + dc) * N + i % N] : 0.f;
            }
        }

        Regs rg;
        fetch(rg, p, geo, b, blk, d0, dend, 0, tid);
        prologue(rg, pc, sm, p, 0, tid);
        if (nchunks > 1) fetch(rg, p, geo, b, blk, d0, dend, TC, tid);
        __syncthreads();

        for (int64_t ch = 0; ch < nchunks; ++ch) {
            float v[K];
            if constexpr (!CF::kSplit) {
                sweep_direct(h, A2, sm, c, g, v);
            } else {
                const int tf = warp * K;  // this warp's sub-chunk
                float2 dA[K][G / 2], dBu[K][G / 2], hl[G / 2];
                const float sd = sweep_local(dA, dBu, hl, A2, sm, tf, c, g);
                // sub-chunk summary (prod_i exp(Delta_i A), local end state)
                float* s_P = sm + CF::OFF_P + (warp * CW + c) * N + g * G;
                float* s_H = sm + CF::OFF_H + (warp * CW + c) * N + g * G;
#pragma unroll
                for (int j = 0; j < G / 2; j += 2) {
                    const float2 P0 = exp2_2<kFast>(mul2(splat2(sd), A2[j]));
                    const float2 P1 = exp2_2<kFast>(mul2(splat2(sd), A2[j + 1]));
                    st4(s_P + 2 * j, make_float4(P0.x, P0.y, P1.x, P1.y));
                    st4(s_H + 2 * j, make_float4(hl[j].x, hl[j].y, hl[j + 1].x, hl[j + 1].y));
                }
                __syncthreads();
                // incoming state: the chunk carry folded through sub-chunks 0 .. warp-1
                const int par = (int)(ch & 1);
                const float* s_car = sm + CF::OFF_CAR + par * CW * N + c * N + g * G;
#pragma unroll
                for (int j = 0; j < G / 2; j += 2) {
                    const float4 cr = ld4(s_car + 2 * j);
                    h[j] = make_float2(cr.x, cr.y);
                    h[j + 1] = make_float2(cr.z, cr.w);
                }
                for (int s = 0; s < warp; ++s) {
                    const float* sp = sm + CF::OFF_P + (s * CW + c) * N + g * G;
                    const float* sh = sm + CF::OFF_H + (s * CW + c) * N + g * G;
#pragma unroll
                    for (int j = 0; j < G / 2; j += 2) {
                        const float4 P = ld4(sp + 2 * j), H = ld4(sh + 2 * j);
                        h[j] = fma2(make_float2(P.x, P.y), h[j], make_float2(H.x, H.y));
                        h[j + 1] = fma2(make_float2(P.z, P.w), h[j + 1], make_float2(H.z, H.w));
                    }
                }
                sweep_replay(dA, dBu, h, sm, tf, g, v);
                // the last sub-chunk's final state is the next chunk's carry
                if (warp == S - 1) {
                    float* s_nc = sm + CF::OFF_CAR + (par ^ 1) * CW * N + c * N + g * G;
#pragma unroll
                    for (int j = 0; j < G / 2; j += 2)
                        st4(s_nc + 2 * j, make_float4(h[j].x, h[j].y, h[j + 1].x, h[j + 1].y));
                }
            }
            reduce_level<R / 2, K>(v, g);
            write_y(v, sm, (CF::kSplit ? warp * K : 0) + g * KR, c);
            __syncthreads();
            store_out(sm, p, geo, b, d0, dend, ch * TC, tid);
            if (ch + 1 < nchunks) {
                prologue(rg, pc, sm, p, (ch + 1) * TC, tid);
                if (ch + 2 < nchunks) fetch(rg, p, geo, b, blk, d0, dend, (ch + 2) * TC, tid);
            }
            __syncthreads();
        }

        if (p.last_state && valid) {
            float* ls = p.last_state + (b * p.dim + d) * N + g * G;
            if constexpr (!CF::kSplit) {
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    ls[2 * j] = h[j].x;
                    ls[2 * j + 1] = h[j].y;
                }
            } else if (warp == 0) {
                // after the last chunk the final state sits in the carry slot
                const float* s_car = sm + CF::OFF_CAR + (int)(nchunks & 1) * CW * N + c * N + g * G;
#pragma unroll
                for (int j = 0; j < G; ++j) ls[j] = s_car[j];
            }
        }
    }
};

template <typename CF, typename T, bool kFast, bool kGrouped>
__global__ void __launch_bounds__(CF::THREADS) scan_fwd_kernel(ScanArgs p, Geo geo) {
    ScanKernel<CF, T, kFast, kGrouped>::run(p, geo);
}

template <typename T, int N, int G, int S, int K>
cudaError_t launch_cfg(const ScanArgs& a, cudaStream_t s) {
    using CF = Cfg<T, N, G, S, K>;
    constexpr bool kFast = !std::is_same<T, float>::value;
    auto kern = a.ngroups == 1 ? scan_fwd_kernel<CF, T, kFast, false> : scan_fwd_kernel<CF, T, kFast, true>;
    if (CF::SMEM_BYTES > 48 * 1024) {
        // once per kernel instantiation and device
        static DeviceMemo memo[2];
        const int gi = a.ngroups == 1 ? 0 : 1;
        int dev = 0, set = 0;
        if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
        cudaError_t err = cudaSuccess;
        if (!memo[gi].get(dev, [&](int& r) {
                err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CF::SMEM_BYTES);
                r = 1;
                return err == cudaSuccess;
            }, &set))
            return err;
    }
    const size_t es = sizeof(T);
    Geo geo;
    // paired accesses need even channel indices: an even row length and,
    // with groups, an even group size (every CTA starts at a group boundary)
    geo.vec_x = (a.dim % 2 == 0) && (a.gch % 2 == 0) && (reinterpret_cast<uintptr_t>(a.u) % (2 * es) == 0) &&
                (reinterpret_cast<uintptr_t>(a.delta) % (2 * es) == 0) &&
                (!a.z || reinterpret_cast<uintptr_t>(a.z) % (2 * es) == 0) &&
                (reinterpret_cast<uintptr_t>(a.out) % (2 * es) == 0);
    geo.vec_bc = (a.seqlen % CF::V == 0) && (reinterpret_cast<uintptr_t>(a.B) % 16 == 0) &&
                 (reinterpret_cast<uintptr_t>(a.C) % 16 == 0);
    geo.bpg = (a.gch + CF::CW - 1) / CF::CW;
    const int64_t gx = a.ngroups * geo.bpg;
    if (gx > 0x7fffffff) return cudaErrorInvalidValue;
    dim3 grid((unsigned)gx, (unsigned)a.batch);
    kern<<<grid, CF::THREADS, CF::SMEM_BYTES, s>>>(a, geo);
    return cudaGetLastError();
}

// The layouts compiled in, per d_state: X(N, G, S, K).  G states per lane,
// S warps (S > 1: time split), K steps per warp per chunk.
#define SSM_LAYOUTS_16(X)                                     \
    X(16, 4, 1, 16)  /* 0: one warp, 8 channels, direct    */ \
    X(16, 8, 1, 16)  /* 1: one warp, 16 channels, direct   */ \
    X(16, 16, 1, 8)  /* 2: one warp, 32 channels, direct   */ \
    X(16, 4, 4, 8)   /* 3: 4 sub-chunks of 8, 8 channels   */ \
    X(16, 4, 2, 8)   /* 4: 2 sub-chunks of 8, 8 channels   */ \
    X(16, 8, 4, 4)   /* 5: 4 sub-chunks of 4, 16 channels  */ \
    X(16, 4, 8, 8)   /* 6: 8 sub-chunks of 8, 8 channels   */

#define SSM_LAYOUTS_8(X)                                      \
    X(8, 4, 1, 16)   /* 0: one warp, 16 channels, direct   */ \
    X(8, 8, 1, 8)    /* 1: one warp, 32 channels, direct   */ \
    X(8, 4, 4, 8)    /* 2: 4 sub-chunks of 8, 16 channels  */ \
    X(8, 8, 4, 4)    /* 3: 4 sub-chunks of 4, 32 channels  */

#define SSM_LAYOUTS_4(X)                                      \
    X(4, 4, 1, 8)    /* 0: one warp, 32 channels, direct   */ \
    X(4, 4, 4, 8)    /* 1: 4 sub-chunks of 8, 32 channels  */

template <typename T>
cudaError_t launch_layout(const ScanArgs& a, int layout, cudaStream_t s) {
    int i = 0;
#define X(N_, G_, S_, K_) \
    if (a.dstate == N_ && layout == i++) return launch_cfg<T, N_, G_, S_, K_>(a, s);
    if (a.dstate == 16) {
        SSM_LAYOUTS_16(X)
    } else if (a.dstate == 8) {
        SSM_LAYOUTS_8(X)
    } else if (a.dstate == 4) {
        SSM_LAYOUTS_4(X)
    }
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace

int scan_layout_count(int dstate) {
    int n = 0;
#define X(N_, G_, S_, K_) ++n;
    switch (dstate) {
        case 16: SSM_LAYOUTS_16(X) break;
        case 8: SSM_LAYOUTS_8(X) break;
        case 4: SSM_LAYOUTS_4(X) break;
        default: break;
    }
#undef X
    return n;
}

ScanLayoutInfo scan_layout_info(int dstate, int layout) {
    ScanLayoutInfo r{0, 0, 0, 0, 0};
    int i = 0;
#define X(N_, G_, S_, K_) \
    if (layout == i++) r = ScanLayoutInfo{G_, S_, 1, K_, 32 / (N_ / G_)};
    switch (dstate) {
        case 16: SSM_LAYOUTS_16(X) break;
        case 8: SSM_LAYOUTS_8(X) break;
        case 4: SSM_LAYOUTS_4(X) break;
        default: break;
    }
#undef X
    return r;
}

cudaError_t launch_scan_fwd(const ScanArgs& a, DType dt, const ScanPlan& plan, cudaStream_t s) {
    return dt == DType::F32 ? launch_layout<float>(a, plan.layout, s)
                            : launch_layout<__nv_bfloat16>(a, plan.layout, s);
}

}  // namespace ssm
