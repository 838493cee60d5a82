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
//   * lane = (tl, c, g): channel c of the CTA, state group g (G consecutive
//     states; the R = N / G lanes of a channel are adjacent), time lane tl;
//   * a chunk of TC = S * TL * K steps is cut into S * TL sub-chunks of K
//     steps, sub-chunk sc = warp * TL + tl;
//   * S * TL == 1: one lane walks every step of the chunk with its states in
//     registers (the sequential scan of "Efficient Scan");
//   * S * TL > 1: each lane first runs its sub-chunk from a zero state,
//     keeping exp(Delta A) and Delta B u of every step in registers; the
//     sub-chunk summaries (prod exp(Delta A), local end state) are combined
//     in order with the associative operator
//         (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2)
//     ("Efficient Scan", parallel scan), giving each sub-chunk its true
//     incoming state; a second sweep over the stored values then produces
//     h_t and y_t.  No exponential is evaluated twice.
//   * per (t, d) work (softplus, Delta u, D u, silu(z)) is done once per
//     (t, d) per chunk into shared memory; the raw activations and B/C of
//     chunk k+1 are fetched into registers while chunk k is computed;
//   * y_t = sum over the R lanes of a channel: each lane holds K partial sums
//     and a transposed butterfly leaves K / R finished sums per lane;
//   * the inner loop uses packed f32x2 multiplies / FMAs (two states per
//     instruction) and one SFU ex2 per (t, state).
#include <cstdint>
#include <type_traits>

#include "ssm_internal.cuh"

namespace ssm {
namespace {

// ------------------------------------------------------------- f32x2 helpers

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

template <bool kFast>
__device__ __forceinline__ float2 exp2_2(float2 x) {
    return make_float2(decay_exp2<kFast>(x.x), decay_exp2<kFast>(x.y));
}

// ------------------------------------------------------------- configuration

template <typename T, int N_, int G_, int S_, int TL_, int K_>
struct Cfg {
    static constexpr int N = N_, G = G_, S = S_, TL = TL_, K = K_;
    static constexpr int R = N / G;                 // lanes per channel
    static constexpr int CW = 32 / (R * TL);        // channels per CTA
    static constexpr int THREADS = 32 * S;
    static constexpr int NSUB = S * TL;             // sub-chunks per chunk
    static constexpr int TC = NSUB * K;             // steps per chunk
    static constexpr bool kSplit = NSUB > 1;
    static constexpr int V = 16 / (int)sizeof(T);   // elements per 16-byte vector
    static constexpr int PAIRS = TC * CW / 2;       // (t, channel pair) items per chunk
    static constexpr int PAIRS_PT = (PAIRS + THREADS - 1) / THREADS;
    static constexpr int BCV = 2 * N * TC / V;      // 16-byte vectors of B and C per chunk
    static constexpr int BCV_PT = (BCV + THREADS - 1) / THREADS;
    static constexpr int KR = K / R;                // finished sums per lane
    static constexpr int CH_PT = (CW * N + THREADS - 1) / THREADS;  // combine chains per thread
    static_assert(G % 2 == 0, "two states per packed instruction");
    static_assert(N % G == 0 && R * TL <= 16 && 32 % (R * TL) == 0, "lane layout");
    static_assert(K % R == 0, "transposed reduction needs K multiple of R");
    static_assert((N * TC) % V == 0, "B/C chunk rows are whole vectors");
    // shared memory, in floats
    static constexpr int OFF_DD = 0;                           // float2 [TC][CW]  (Delta, Delta u)
    static constexpr int OFF_SG = OFF_DD + 2 * TC * CW;        // float2 [TC][CW]  (D u, silu z)
    static constexpr int OFF_B = OFF_SG + 2 * TC * CW;         // float  [TC][N]
    static constexpr int OFF_C = OFF_B + TC * N;               // float  [TC][N]
    static constexpr int OFF_SUM = OFF_C + TC * N;             // float2 [NSUB][CW][N]
    static constexpr int OFF_CIN = OFF_SUM + (kSplit ? 2 * NSUB * CW * N : 0);  // [NSUB][CW][N]
    static constexpr int OFF_OUT = OFF_CIN + (kSplit ? NSUB * CW * N : 0);      // T [TC][CW]
    static constexpr int SMEM_FLOATS = OFF_OUT + (TC * CW * (int)sizeof(T) + 3) / 4;
    static constexpr size_t SMEM_BYTES = sizeof(float) * SMEM_FLOATS;
};

// Per-launch facts the kernel needs beyond ScanArgs.
struct Geo {
    int vec_x;   // u/delta/z/out rows allow paired (2-element) accesses
    int vec_bc;  // B/C rows allow 16-byte accesses
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

template <typename CF, typename T, bool kFast>
struct ScanKernel {
    using PT = typename Pair<T>::type;
    static constexpr int N = CF::N, G = CF::G, R = CF::R, CW = CF::CW, K = CF::K;
    static constexpr int TC = CF::TC, NSUB = CF::NSUB, V = CF::V;

    // ---- raw fetch of one chunk into registers (zero outside the tensor)
    struct Regs {
        PT u[CF::PAIRS_PT], dl[CF::PAIRS_PT], z[CF::PAIRS_PT];
        uint4 bc[CF::BCV_PT];
    };

    static __device__ __forceinline__ PT load_pair(const T* base, int64_t row, int64_t d, int64_t dim,
                                                   int64_t L, bool vec) {
        if (row < L && d + 1 < dim && vec) return *reinterpret_cast<const PT*>(base + row * dim + d);
        float a = 0.f, b = 0.f;
        if (row < L) {
            if (d < dim) a = to_f32(base[row * dim + d]);
            if (d + 1 < dim) b = to_f32(base[row * dim + d + 1]);
        }
        return Pair<T>::make(a, b);
    }

    static __device__ __forceinline__ void fetch(Regs& r, const ScanArgs& p, const Geo& geo, int64_t b,
                                                 int64_t d0, int64_t t0, int tid) {
        const int64_t L = p.seqlen, dim = p.dim;
        const T* u = static_cast<const T*>(p.u) + b * L * dim;
        const T* dl = static_cast<const T*>(p.delta) + b * L * dim;
        const T* zp = p.z ? static_cast<const T*>(p.z) + b * L * dim : nullptr;
#pragma unroll
        for (int k = 0; k < CF::PAIRS_PT; ++k) {
            const int idx = tid + k * CF::THREADS;
            if (CF::PAIRS % CF::THREADS == 0 || idx < CF::PAIRS) {
                const int t = idx / (CW / 2), cp = idx % (CW / 2);
                const int64_t row = t0 + t, d = d0 + 2 * cp;
                r.u[k] = load_pair(u, row, d, dim, L, geo.vec_x);
                r.dl[k] = load_pair(dl, row, d, dim, L, geo.vec_x);
                r.z[k] = zp ? load_pair(zp, row, d, dim, L, geo.vec_x) : Pair<T>::make(0.f, 0.f);
            }
        }
        const T* Bb = static_cast<const T*>(p.B) + b * N * L;
        const T* Cb = static_cast<const T*>(p.C) + b * N * L;
#pragma unroll
        for (int k = 0; k < CF::BCV_PT; ++k) {
            const int idx = tid + k * CF::THREADS;
            if (CF::BCV % CF::THREADS == 0 || idx < CF::BCV) {
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
    static __device__ __forceinline__ void prologue(const Regs& r, float* sm, const ScanArgs& p, int64_t d0,
                                                    int64_t t0, int tid) {
        float2* s_dd = reinterpret_cast<float2*>(sm + CF::OFF_DD);
        float2* s_sg = reinterpret_cast<float2*>(sm + CF::OFF_SG);
#pragma unroll
        for (int k = 0; k < CF::PAIRS_PT; ++k) {
            const int idx = tid + k * CF::THREADS;
            if (CF::PAIRS % CF::THREADS == 0 || idx < CF::PAIRS) {
                const int t = idx / (CW / 2), cp = idx % (CW / 2);
                const float2 uv = Pair<T>::f(r.u[k]);
                const float2 xv = Pair<T>::f(r.dl[k]);
                const float2 zv = Pair<T>::f(r.z[k]);
                const float ua[2] = {uv.x, uv.y}, xa[2] = {xv.x, xv.y}, za[2] = {zv.x, zv.y};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = 2 * cp + e;
                    const int64_t d = d0 + c;
                    const bool ok = d < p.dim && t0 + t < p.seqlen;
                    float x = xa[e];
                    if (p.delta_bias && ok) x += p.delta_bias[d];
                    float dlt = p.softplus ? softplus_f<kFast>(x) : x;
                    // padded steps / channels: Delta = 0 leaves the state unchanged
                    dlt = ok ? dlt : 0.f;
                    const float skip = (p.D && ok) ? p.D[d] * ua[e] : 0.f;
                    const float gate = p.z ? silu_f<kFast>(za[e]) : 1.f;
                    s_dd[t * CW + c] = make_float2(dlt, dlt * ua[e]);
                    s_sg[t * CW + c] = make_float2(skip, gate);
                }
            }
        }
        float* s_B = sm + CF::OFF_B;
        float* s_C = sm + CF::OFF_C;
#pragma unroll
        for (int k = 0; k < CF::BCV_PT; ++k) {
            const int idx = tid + k * CF::THREADS;
            if (CF::BCV % CF::THREADS == 0 || idx < CF::BCV) {
                const int which = idx / (N * TC / V);
                const int rem = idx % (N * TC / V);
                const int n = rem / (TC / V), tv = rem % (TC / V);
                float* dst = which ? s_C : s_B;
                const T* e = reinterpret_cast<const T*>(&r.bc[k]);
#pragma unroll
                for (int j = 0; j < V; ++j) dst[(tv * V + j) * N + n] = to_f32(e[j]);
            }
        }
    }

    // ---- out tile (shared) -> global, pairs of channels per access
    static __device__ __forceinline__ void store_out(const float* sm, const ScanArgs& p, const Geo& geo,
                                                     int64_t b, int64_t d0, int64_t t0, int tid) {
        const T* s_out = reinterpret_cast<const T*>(sm + CF::OFF_OUT);
        T* out = static_cast<T*>(p.out) + b * p.seqlen * p.dim;
#pragma unroll
        for (int k = 0; k < CF::PAIRS_PT; ++k) {
            const int idx = tid + k * CF::THREADS;
            if (CF::PAIRS % CF::THREADS == 0 || idx < CF::PAIRS) {
                const int t = idx / (CW / 2), cp = idx % (CW / 2);
                const int64_t row = t0 + t, d = d0 + 2 * cp;
                if (row >= p.seqlen) continue;
                const T a = s_out[t * CW + 2 * cp], c = s_out[t * CW + 2 * cp + 1];
                if (geo.vec_x && d + 1 < p.dim) {
                    PT v;
                    reinterpret_cast<T*>(&v)[0] = a;
                    reinterpret_cast<T*>(&v)[1] = c;
                    *reinterpret_cast<PT*>(out + row * p.dim + d) = v;
                } else {
                    if (d < p.dim) out[row * p.dim + d] = a;
                    if (d + 1 < p.dim) out[row * p.dim + d + 1] = c;
                }
            }
        }
    }

    // ---- y: transposed butterfly over the R lanes of a channel.  On return
    // v[0..K/R) of lane g hold the full sums of steps g*K/R .. g*K/R + K/R - 1.
    static __device__ __forceinline__ void reduce_lanes(float (&v)[K], int g) {
#pragma unroll
        for (int m = R / 2, len = K; m >= 1; m >>= 1, len >>= 1) {
            const bool upper = (g & m) != 0;
#pragma unroll
            for (int r = 0; r < len / 2; ++r) {
                const float send = upper ? v[r] : v[r + len / 2];
                const float keep = upper ? v[r + len / 2] : v[r];
                v[r] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
        }
    }

    // ---- finished sums -> gated outputs in the shared out tile
    static __device__ __forceinline__ void write_y(const float (&v)[K], float* sm, int sc, int c, int g) {
        const float2* s_sg = reinterpret_cast<const float2*>(sm + CF::OFF_SG);
        T* s_out = reinterpret_cast<T*>(sm + CF::OFF_OUT);
#pragma unroll
        for (int r = 0; r < CF::KR; ++r) {
            const int t = sc * K + g * CF::KR + r;
            const float2 sg = s_sg[t * CW + c];
            s_out[t * CW + c] = from_f32<T>((v[r] + sg.x) * sg.y);
        }
    }

    static __device__ void run(const ScanArgs& p, const Geo& geo) {
        extern __shared__ float sm[];
        const int tid = threadIdx.x;
        const int warp = tid >> 5, lane = tid & 31;
        const int g = lane % R;
        const int c = (lane / R) % CW;
        const int tl = lane / (R * CW);
        const int sc = warp * CF::TL + tl;           // sub-chunk of this lane
        const int n0 = g * G;
        const int64_t b = blockIdx.y;
        const int64_t d0 = (int64_t)blockIdx.x * CW;
        const int64_t d = d0 + c;
        const bool valid = d < p.dim;
        const int64_t L = p.seqlen;
        const int64_t nchunks = (L + TC - 1) / TC;

        float2 A2[G / 2];
#pragma unroll
        for (int j = 0; j < G / 2; ++j) {
            const float a0 = valid ? p.A[d * N + n0 + 2 * j] : 0.f;
            const float a1 = valid ? p.A[d * N + n0 + 2 * j + 1] : 0.f;
            A2[j] = make_float2(a0 * kLog2e, a1 * kLog2e);
        }
        const float2* s_dd = reinterpret_cast<const float2*>(sm + CF::OFF_DD);
        const float* s_B = sm + CF::OFF_B;
        const float* s_C = sm + CF::OFF_C;

        // state: per lane (non-split) or per (channel, state) combine thread (split)
        float2 h[G / 2];
#pragma unroll
        for (int j = 0; j < G / 2; ++j) h[j] = make_float2(0.f, 0.f);
        // split: running state of the chains tid, tid + THREADS, ... (chain = c * N + n)
        float carry[CF::CH_PT];
#pragma unroll
        for (int k = 0; k < CF::CH_PT; ++k) carry[k] = 0.f;

        Regs rg;
        fetch(rg, p, geo, b, d0, 0, tid);
        prologue(rg, sm, p, d0, 0, tid);
        if (nchunks > 1) fetch(rg, p, geo, b, d0, TC, tid);
        __syncthreads();

        for (int64_t ch = 0; ch < nchunks; ++ch) {
            float v[K];
            if constexpr (!CF::kSplit) {
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    const int t = i;
                    const float2 dd = s_dd[t * CW + c];
                    const float2 x2 = make_float2(dd.x, dd.x), u2 = make_float2(dd.y, dd.y);
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < G / 2; ++j) {
                        const float2 bv = *reinterpret_cast<const float2*>(s_B + t * N + n0 + 2 * j);
                        const float2 cv = *reinterpret_cast<const float2*>(s_C + t * N + n0 + 2 * j);
                        const float2 dA = exp2_2<kFast>(mul2(x2, A2[j]));
                        h[j] = fma2(dA, h[j], mul2(u2, bv));
                        acc = fma2(cv, h[j], acc);
                    }
                    v[i] = acc.x + acc.y;
                }
            } else {
                // pass 1: local scan of this lane's sub-chunk from a zero state
                float2 dA[K][G / 2], dBu[K][G / 2];
                float2 hl[G / 2];
                float sdl = 0.f;
#pragma unroll
                for (int j = 0; j < G / 2; ++j) hl[j] = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    const int t = sc * K + i;
                    const float2 dd = s_dd[t * CW + c];
                    const float2 x2 = make_float2(dd.x, dd.x), u2 = make_float2(dd.y, dd.y);
                    sdl += dd.x;
#pragma unroll
                    for (int j = 0; j < G / 2; ++j) {
                        const float2 bv = *reinterpret_cast<const float2*>(s_B + t * N + n0 + 2 * j);
                        dA[i][j] = exp2_2<kFast>(mul2(x2, A2[j]));
                        dBu[i][j] = mul2(u2, bv);
                        hl[j] = fma2(dA[i][j], hl[j], dBu[i][j]);
                    }
                }
                // sub-chunk summary: (prod_i exp(Delta_i A), local end state)
                float2* s_sum = reinterpret_cast<float2*>(sm + CF::OFF_SUM);
                const float2 s2 = make_float2(sdl, sdl);
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    const float2 P = exp2_2<kFast>(mul2(s2, A2[j]));
                    s_sum[(sc * CW + c) * N + n0 + 2 * j] = make_float2(P.x, hl[j].x);
                    s_sum[(sc * CW + c) * N + n0 + 2 * j + 1] = make_float2(P.y, hl[j].y);
                }
                __syncthreads();
                // ordered combine of the sub-chunk summaries, one thread per chain
                float* s_cin = sm + CF::OFF_CIN;
#pragma unroll
                for (int k = 0; k < CF::CH_PT; ++k) {
                    const int chain = tid + k * CF::THREADS;
                    if (chain < CW * N) {
                        float cr = carry[k];
#pragma unroll
                        for (int s = 0; s < NSUB; ++s) {
                            s_cin[s * CW * N + chain] = cr;
                            const float2 ph = s_sum[s * CW * N + chain];
                            cr = fmaf(ph.x, cr, ph.y);
                        }
                        carry[k] = cr;
                    }
                }
                __syncthreads();
                // pass 2: rerun the sub-chunk from its true incoming state
#pragma unroll
                for (int j = 0; j < G / 2; ++j)
                    h[j] = *reinterpret_cast<const float2*>(s_cin + (sc * CW + c) * N + n0 + 2 * j);
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    const int t = sc * K + i;
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < G / 2; ++j) {
                        const float2 cv = *reinterpret_cast<const float2*>(s_C + t * N + n0 + 2 * j);
                        h[j] = fma2(dA[i][j], h[j], dBu[i][j]);
                        acc = fma2(cv, h[j], acc);
                    }
                    v[i] = acc.x + acc.y;
                }
            }
            reduce_lanes(v, g);
            write_y(v, sm, sc, c, g);
            __syncthreads();
            store_out(sm, p, geo, b, d0, ch * TC, tid);
            if (ch + 1 < nchunks) {
                prologue(rg, sm, p, d0, (ch + 1) * TC, tid);
                if (ch + 2 < nchunks) fetch(rg, p, geo, b, d0, (ch + 2) * TC, tid);
            }
            __syncthreads();
        }

        if (p.last_state) {
            if constexpr (!CF::kSplit) {
                if (valid) {
                    float* ls = p.last_state + (b * p.dim + d) * N + n0;
#pragma unroll
                    for (int j = 0; j < G / 2; ++j) {
                        ls[2 * j] = h[j].x;
                        ls[2 * j + 1] = h[j].y;
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < CF::CH_PT; ++k) {
                    const int chain = tid + k * CF::THREADS;
                    const int64_t dd = d0 + chain / N;
                    if (chain < CW * N && dd < p.dim) p.last_state[(b * p.dim + dd) * N + chain % N] = carry[k];
                }
            }
        }
    }
};

template <typename CF, typename T, bool kFast>
__global__ void __launch_bounds__(CF::THREADS) scan_fwd_kernel(ScanArgs p, Geo geo) {
    ScanKernel<CF, T, kFast>::run(p, geo);
}

template <typename T, int N, int G, int S, int TL, int K>
cudaError_t launch_cfg(const ScanArgs& a, cudaStream_t s) {
    using CF = Cfg<T, N, G, S, TL, K>;
    constexpr bool kFast = !std::is_same<T, float>::value;
    auto kern = scan_fwd_kernel<CF, T, kFast>;
    if (CF::SMEM_BYTES > 48 * 1024) {
        static bool attr_set = false;  // once per instantiation
        if (!attr_set) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)CF::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            attr_set = true;
        }
    }
    const size_t es = sizeof(T);
    Geo geo;
    geo.vec_x = (a.dim % 2 == 0) && (reinterpret_cast<uintptr_t>(a.u) % (2 * es) == 0) &&
                (reinterpret_cast<uintptr_t>(a.delta) % (2 * es) == 0) &&
                (!a.z || reinterpret_cast<uintptr_t>(a.z) % (2 * es) == 0) &&
                (reinterpret_cast<uintptr_t>(a.out) % (2 * es) == 0);
    geo.vec_bc = (a.seqlen % CF::V == 0) && (reinterpret_cast<uintptr_t>(a.B) % 16 == 0) &&
                 (reinterpret_cast<uintptr_t>(a.C) % 16 == 0);
    const int64_t gx = (a.dim + CF::CW - 1) / CF::CW;
    dim3 grid((unsigned)gx, (unsigned)a.batch);
    kern<<<grid, CF::THREADS, CF::SMEM_BYTES, s>>>(a, geo);
    return cudaGetLastError();
}

// The layouts compiled in, by (d_state, dtype).  `plan.layout` indexes this
// table; entry 0 of each list is the default for small problems.
#define SSM_LAYOUTS_16(X)                                   \
    X(16, 4, 1, 1, 16) /* 0: one warp, 8 channels       */ \
    X(16, 8, 1, 1, 16) /* 1: one warp, 16 channels      */ \
    X(16, 16, 1, 1, 16) /* 2: one warp, 32 channels     */ \
    X(16, 4, 4, 1, 8)  /* 3: 4 warps x 8 steps, 8 ch    */ \
    X(16, 4, 4, 2, 8)  /* 4: 8 sub-chunks, 4 channels   */ \
    X(16, 4, 2, 2, 8)  /* 5: 4 sub-chunks, 4 channels   */ \
    X(16, 8, 4, 1, 8)  /* 6: 4 warps, 16 channels       */ \
    X(16, 2, 4, 1, 8)  /* 7: 4 warps, 4 channels, G=2   */

template <typename T, int N>
cudaError_t launch_layout(const ScanArgs& a, int layout, cudaStream_t s);

template <typename T>
cudaError_t launch_16(const ScanArgs& a, int layout, cudaStream_t s) {
    int i = 0;
#define X(N, G, S, TL, K) \
    if (layout == i++) return launch_cfg<T, N, G, S, TL, K>(a, s);
    SSM_LAYOUTS_16(X)
#undef X
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_8(const ScanArgs& a, int layout, cudaStream_t s) {
    switch (layout) {
        case 0: return launch_cfg<T, 8, 4, 1, 1, 16>(a, s);
        case 1: return launch_cfg<T, 8, 8, 1, 1, 16>(a, s);
        case 2: return launch_cfg<T, 8, 2, 4, 1, 8>(a, s);
        case 3: return launch_cfg<T, 8, 4, 4, 1, 8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_4(const ScanArgs& a, int layout, cudaStream_t s) {
    switch (layout) {
        case 0: return launch_cfg<T, 4, 4, 1, 1, 16>(a, s);
        case 1: return launch_cfg<T, 4, 2, 1, 1, 16>(a, s);
        case 2: return launch_cfg<T, 4, 2, 4, 1, 8>(a, s);
        case 3: return launch_cfg<T, 4, 4, 4, 1, 8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int scan_layout_count(int dstate) {
    switch (dstate) {
        case 16: {
            int n = 0;
#define X(N, G, S, TL, K) ++n;
            SSM_LAYOUTS_16(X)
#undef X
            return n;
        }
        case 8: return 4;
        case 4: return 4;
        default: return 0;
    }
}

ScanLayoutInfo scan_layout_info(int dstate, int layout) {
    ScanLayoutInfo r{0, 0, 0, 0, 0};
    auto set = [&](int G, int S, int TL, int K) {
        const int R = dstate / G;
        r = ScanLayoutInfo{G, S, TL, K, 32 / (R * TL)};
    };
    int i = 0;
    switch (dstate) {
        case 16:
#define X(N, G, S, TL, K) \
    if (layout == i++) set(G, S, TL, K);
            SSM_LAYOUTS_16(X)
#undef X
            break;
        case 8: {
            const int t[4][4] = {{4, 1, 1, 16}, {8, 1, 1, 16}, {2, 4, 1, 8}, {4, 4, 1, 8}};
            if (layout >= 0 && layout < 4) set(t[layout][0], t[layout][1], t[layout][2], t[layout][3]);
            break;
        }
        case 4: {
            const int t[4][4] = {{4, 1, 1, 16}, {2, 1, 1, 16}, {2, 4, 1, 8}, {4, 4, 1, 8}};
            if (layout >= 0 && layout < 4) set(t[layout][0], t[layout][1], t[layout][2], t[layout][3]);
            break;
        }
        default: break;
    }
    return r;
}

cudaError_t launch_scan_fwd(const ScanArgs& a, DType dt, const ScanPlan& plan, cudaStream_t s) {
    const bool f32 = dt == DType::F32;
    switch (a.dstate) {
        case 16: return f32 ? launch_16<float>(a, plan.layout, s) : launch_16<__nv_bfloat16>(a, plan.layout, s);
        case 8: return f32 ? launch_8<float>(a, plan.layout, s) : launch_8<__nv_bfloat16>(a, plan.layout, s);
        case 4: return f32 ? launch_4<float>(a, plan.layout, s) : launch_4<__nv_bfloat16>(a, plan.layout, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
