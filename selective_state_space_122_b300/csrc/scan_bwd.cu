// scan_bwd.cu -- the backward of the selective scan: every input's gradient
// given dout = dL/d out (the training half of the pages' "Efficient Scan":
// "Mamba: Selective State Space Models" README).
//
// With x_t = delta_raw_t + bias, Delta_t = softplus(x_t) (or x_t),
// a_t[n] = exp(Delta_t A[n]), h_t = a_t h_{t-1} + Delta_t B_t u_t,
// y_t = C_t . h_t + D u_t, out_t = y_t silu(z_t), the adjoint state
// lambda_t = dL/dh_t runs backwards in time,
//     dy_t = dout_t silu(z_t),   lambda_t = C_t dy_t + mu_{t+1},   mu_t = a_t lambda_t,
// and the gradients are sums of per-step terms (w_t = mu_t h_{t-1}):
//     dC_t[n] = sum_d dy_t h_t[n]          dB_t[n] = sum_d lambda_t[n] Delta_t u_t
//     du_t    = D dy_t + Delta_t sum_n lambda_t[n] B_t[n]
//     dDelta_t = sum_n A[n] w_t[n] + u_t sum_n lambda_t[n] B_t[n]
//     dA[n]   = sum_{b,t} Delta_t w_t[n]
//     dD = sum dy_t u_t,   dz_t = dout_t y_t silu'(z_t),
//     ddelta_raw_t = dDelta_t softplus'(x_t),   dbias = sum ddelta_raw_t.
//
// Work decomposition.  Every (batch row, block of CC channels) chain is cut
// into S segments of whole 8-step chunks, and the two directions of the
// recurrence cross the segment boundaries through per-segment aggregates, so
// every segment runs independently of the others:
//   pass 1 (bwd_local_kernel, one CTA per block and segment): the forward
//       recurrence from a zero state, storing the local state entering every
//       chunk and the sum of Delta up to it; at the segment's end the decay
//       product Q = prod a_t, the local end state, and the adjoint aggregate
//       Lambda = sum_t (prod_{r <= t} a_r) C_t dy_t (all per state).
//   combine (bwd_combine_kernel, one thread per (b, d, n)): the true state
//       entering segment s, H_s = Q_{s-1} H_{s-1} + h_end_{s-1} from the
//       initial state, and the adjoint carried into the segment's last step
//       from the right, rho_{s-1} = Q_s rho_s + Lambda_s from dL/d last_state;
//       rho_{-1} = a_0 lambda_0 is dL/d initial_state.
//   pass 2 (bwd_main_kernel, one CTA per block and segment): the chunks in
//       reverse order; each chunk's entering state is the stored local one
//       plus exp(A * sum Delta) H_s, the chunk's states and decays are
//       recomputed into registers, and the adjoint runs backwards over them
//       from rho_s with every gradient term.
// A lane keeps four states of one channel (N/4 lanes per channel).  The
// chunks' inputs are staged into shared memory with 16-byte asynchronous
// copies three chunks ahead; sums over a channel's states go through shared
// memory (readout) or a transposed two-value shuffle (du, dDelta), and dB, dC
// are halved across warp halves with one shuffle round before their
// per-chunk channel sums in shared memory.  dA, dB, dC, dD and dbias
// accumulate across CTAs with atomics (the launcher zeroes them first).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "device_memo.h"
#include "scan_common.cuh"
#include "ssm_internal.cuh"

namespace ssm {

namespace {

constexpr int kThreads = 128;   // 4 warps
constexpr int kK = 8;           // steps per chunk (the checkpoint interval)
constexpr int kStages = 4;      // staged chunks: the current one and three ahead (3: 1.163 ms, 5: 1.161 ms)
constexpr int kHold = 4;        // recomputed states held in registers at once (a divisor of kK)

// Segments per chain: whole chunks, at least 32 chunks (256 steps) each, at
// most 64 segments.  A function of the sequence length only, so the
// workspace size does not depend on the device.
__host__ __device__ constexpr int64_t bwd_segments(int64_t nch) {
    const int64_t s = (nch + 31) / 32;
    return s < 1 ? 1 : (s > 64 ? 64 : s);
}

template <typename T, int N>
struct BwCfg {
    static constexpr int G = 4;                        // states per lane
    static constexpr int R = N / G;                    // lanes per channel
    static constexpr int CPW = 32 / R;                 // channels per warp
    static constexpr int CC = CPW * (kThreads / 32);   // channels per CTA
    static constexpr int ES = (int)sizeof(T);
    // one staged chunk: u, delta_raw, z, dout tiles [K][CC], then B, C [N][K]
    static constexpr int TILE = kK * CC * ES;
    static constexpr int BCT = N * kK * ES;
    static constexpr int STAGE = 4 * TILE + 2 * BCT;
    // per-(t, d) work: a thread keeps one channel (tid % CC) and takes the
    // steps tid / CC + j * KS, in pairs (k, k + K/2) for packed arithmetic
    static constexpr int KS = kThreads / CC;
    static constexpr int HP = kK / (2 * KS);             // step pairs per thread
    // shared memory (bytes)
    static constexpr int O_TD = kStages * STAGE;           // float4 [K][CC]: Delta, Delta u, dy, u
    static constexpr int O_BC = O_TD + kK * CC * 16;       // float [2][K][N]: B, C
    static constexpr int SMEM1 = O_BC + 2 * kK * N * 4;
    static constexpr int O_YP = SMEM1;                     // float [K][CC][R]: readout partials
    static constexpr int O_SD = O_YP + kK * CC * R * 4;    // float2 [K][CC]: sum lambda B, sum A w
    static constexpr int O_P = O_SD + kK * CC * 8;         // float4 [K][threads]: dB or dC quads
    static constexpr int O_PAR = O_P + kK * kThreads * 16; // float2 [CC]: bias, D of each channel
    static constexpr int O_ACC = O_PAR + CC * 8;           // float2 [threads]: dD, dbias partial sums
    static constexpr int SUMROW = kK + 4;                  // padded row (48 bytes): fewer bank conflicts
    static constexpr int O_SUM = O_ACC + kThreads * 8;     // float [2][N][SUMROW]: the chunk's dB, dC sums
    static constexpr int SMEM3 = O_SUM + 2 * N * SUMROW * 4;
    static_assert(STAGE % 16 == 0 && SMEM3 <= 227 * 1024, "shared memory of one CTA");
    static_assert(HP >= 1 && 2 * HP * KS == kK, "step pairs");
};

// Workspace views (carved by the launcher).
struct BwdWs {
    float* ckpt;    // [batch][nch][dim][N]  local state entering every chunk
    float* cum;     // [batch][nch][dim]     sum of Delta from the segment start to the chunk
    float* aggQ;    // [batch][S][dim][N]    decay product of each segment
    float* aggH;    // [batch][S][dim][N]    local end state -> (combine) true entering state
    float* aggL;    // [batch][S][dim][N]    adjoint aggregate -> (combine) carry from the right
    int64_t nch;    // chunks of the sequence
    int64_t cps;    // chunks per segment
    int64_t nseg;   // segments
    int vec;        // 16-byte asynchronous staging allowed (alignment and sizes)
    int red4;       // dB, dC take 16-byte reductions (alignment, seqlen % 4 == 0)
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
// Four consecutive floats added to global memory in one reduction (16-byte
// aligned address).
__device__ __forceinline__ void red_add_v4(float* p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int n>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

// softplus(x) and its derivative sigmoid(x) for two values.  kFast: one SFU
// exp2 (e = e^-|x|), the polynomial log1p of the forward's fast path and one
// reciprocal; otherwise the library functions.
template <bool kFast>
__device__ __forceinline__ void softplus_and_sigmoid2(float2 x, float2& sp, float2& sg) {
    if constexpr (kFast) {
        const float2 e = make_float2(ex2_approx(-fabsf(x.x) * kLog2e), ex2_approx(-fabsf(x.y) * kLog2e));
        const float2 l = log1p_unit2(e);
        sp = make_float2(fmaxf(x.x, 0.f) + l.x, fmaxf(x.y, 0.f) + l.y);
        const float2 r = make_float2(rcp_approx(1.f + e.x), rcp_approx(1.f + e.y));
        sg = make_float2(x.x >= 0.f ? r.x : e.x * r.x, x.y >= 0.f ? r.y : e.y * r.y);
    } else {
        sp = make_float2(softplus_acc(x.x), softplus_acc(x.y));
        sg = make_float2(1.f / (1.f + expf(-x.x)), 1.f / (1.f + expf(-x.y)));
    }
}

template <bool kFast>
__device__ __forceinline__ float2 sigmoid2(float2 z) {
    if constexpr (kFast) {
        const float2 e = make_float2(ex2_approx(-fabsf(z.x) * kLog2e), ex2_approx(-fabsf(z.y) * kLog2e));
        const float2 r = make_float2(rcp_approx(1.f + e.x), rcp_approx(1.f + e.y));
        return make_float2(z.x >= 0.f ? r.x : e.x * r.x, z.y >= 0.f ? r.y : e.y * r.y);
    } else {
        return make_float2(1.f / (1.f + expf(-z.x)), 1.f / (1.f + expf(-z.y)));
    }
}

// The CTA's place: batch row, B/C group, channel block, segment and chunks.
struct Geo {
    int64_t b, blk;   // batch row; B/C block b * ngroups + group
    int d0, dend;     // channels [d0, dend) (within one group)
    int sgm;
    int64_t c_begin, c_end;
};

template <int CC>
__device__ __forceinline__ Geo make_geo(const BwdArgs& p, const BwdWs& w) {
    Geo q;
    // CTA -> (group, block of CC channels within it): the CTAs of a group
    // cover its channels [grp * gch, dend) only, so every CTA reads and adds
    // to one B/C block (channel indices stay below 2^31: the host rejects
    // larger dims)
    const int gch = (int)p.gch;
    const int bpg = (gch + CC - 1) / CC;
    const int grp = (int)blockIdx.x / bpg;
    q.d0 = grp * gch + ((int)blockIdx.x - grp * bpg) * CC;
    q.dend = q.d0 + min(CC, (grp + 1) * gch - q.d0);
    q.b = blockIdx.z;
    q.blk = q.b * p.ngroups + grp;
    q.sgm = blockIdx.y;
    q.c_begin = (int64_t)q.sgm * w.cps;
    q.c_end = min(w.nch, q.c_begin + w.cps);
    return q;
}

// Stage chunk ch (u, delta_raw, z, dout tiles and the B, C rows) into one
// ring slot; positions past the sequence or the CTA's channels read as zero.
// With 16-byte asynchronous copies (vec: sizes and pointers allow them) each
// thread owns fixed pieces of the slot, whose addresses at chunk 0 are set
// up once (init) and advanced per chunk (one commit group per chunk); plain
// loads otherwise.
template <typename T, int N>
struct Stager {
    using CF = BwCfg<T, N>;
    static constexpr int CC = CF::CC;
    static constexpr int EPP = 16 / CF::ES;         // elements per 16-byte piece
    static constexpr int PR = CC / EPP;             // pieces per tile row
    static constexpr int TP = kK * PR;              // pieces per (t, d) tile
    static constexpr int BR = kK / EPP;             // pieces per B/C row
    static constexpr int TOTAL = 4 * TP + 2 * N * BR;
    static constexpr int MP = (TOTAL + kThreads - 1) / kThreads;
    const char* src0[MP];   // the piece at chunk 0; null: always zero (no channel, no tensor)
    uint32_t dst[MP];       // byte offset within the slot
    int row[MP];            // step offset of the piece within its chunk; +256 for a B/C piece; -1: none
    int64_t tstride;        // bytes of kK rows of a (t, d) tile

    __device__ __forceinline__ void init(const BwdArgs& p, const Geo& q, int tid) {
        const int64_t L = p.seqlen, dim = p.dim;
        tstride = (int64_t)kK * dim * CF::ES;
#pragma unroll
        for (int m = 0; m < MP; ++m) {
            const int i = tid + m * kThreads;
            src0[m] = nullptr;
            dst[m] = 0;
            row[m] = -1;
            if (i < 4 * TP) {
                const int tsr = i / TP, r = i - tsr * TP, k = r / PR, col = r - k * PR;
                const int dd = q.d0 + col * EPP;
                const void* base = tsr == 0 ? p.u : tsr == 1 ? p.delta : tsr == 2 ? p.z : p.dout;
                if (base && dd < q.dend)
                    src0[m] = reinterpret_cast<const char*>(static_cast<const T*>(base) + (q.b * L + k) * dim + dd);
                dst[m] = tsr * CF::TILE + (k * CC + col * EPP) * CF::ES;
                row[m] = k;
            } else if (i < TOTAL) {
                const int j = i - 4 * TP, which = j / (N * BR), r = j - which * N * BR, n = r / BR,
                          pc = r - n * BR;
                const T* bc = static_cast<const T*>(which ? p.C : p.B);
                src0[m] = reinterpret_cast<const char*>(bc + (q.blk * N + n) * L + pc * EPP);
                dst[m] = 4 * CF::TILE + which * CF::BCT + (n * kK + pc * EPP) * CF::ES;
                row[m] = 256 + pc * EPP;
            }
        }
    }

    __device__ __forceinline__ void issue(unsigned char* slot, const BwdArgs& p, int64_t ch) const {
        const uint32_t base = smem_u32(slot);
#pragma unroll
        for (int m = 0; m < MP; ++m) {
            if (row[m] < 0) continue;
            const bool bc = row[m] >= 256;
            const int64_t t = ch * kK + (row[m] & 255);
            const bool ok = src0[m] != nullptr && t < p.seqlen;
            const char* src = ok ? src0[m] + (bc ? ch * (kK * CF::ES) : ch * tstride) : static_cast<const char*>(p.u);
            cp_async16(base + dst[m], src, ok ? 16u : 0u);
        }
        cp_async_commit();
    }
};

template <typename T, int N>
__device__ __forceinline__ void stage_scalar(unsigned char* slot, const BwdArgs& p, const Geo& q, int64_t ch,
                                             int tid) {
    using CF = BwCfg<T, N>;
    constexpr int CC = CF::CC;
    const int64_t t0 = ch * kK, L = p.seqlen, dim = p.dim;
    T* tl = reinterpret_cast<T*>(slot);
    constexpr int TOTAL = 4 * kK * CC + 2 * N * kK;
    for (int i = tid; i < TOTAL; i += kThreads) {
        float v = 0.f;
        if (i < 4 * kK * CC) {
            const int tsr = i / (kK * CC), r = i - tsr * kK * CC, k = r / CC, cc = r - k * CC;
            const int64_t t = t0 + k, dd = q.d0 + cc;
            const T* tp = static_cast<const T*>(tsr == 0 ? p.u : tsr == 1 ? p.delta : tsr == 2 ? p.z : p.dout);
            if (tp && t < L && dd < q.dend) v = to_f32(tp[(q.b * L + t) * dim + dd]);
        } else {
            const int j = i - 4 * kK * CC, which = j / (N * kK), r = j - which * N * kK, n = r / kK,
                      k = r - n * kK;
            const int64_t t = t0 + k;
            const T* bc = static_cast<const T*>(which ? p.C : p.B);
            if (t < L) v = to_f32(bc[(q.blk * N + n) * L + t]);
        }
        tl[i] = from_f32<T>(v);
    }
}

template <typename T, int N>
__device__ __forceinline__ void stage_chunk(const Stager<T, N>& st, unsigned char* slot, const BwdArgs& p,
                                            const Geo& q, int64_t ch, bool vec, int tid) {
    if (vec) st.issue(slot, p, ch);
    else stage_scalar<T, N>(slot, p, q, ch, tid);
}

// The same without held piece addresses (recomputed per chunk): for the
// reverse pass, whose registers go to the chunk's states.
template <typename T, int N>
__device__ __forceinline__ void stage_chunk_direct(unsigned char* slot, const BwdArgs& p, const Geo& q, int64_t ch,
                                                   bool vec, int tid) {
    if (vec) {
        Stager<T, N> st;
        st.init(p, q, tid);
        st.issue(slot, p, ch);
    } else {
        stage_scalar<T, N>(slot, p, q, ch, tid);
    }
}

// A thread's per-(t, d) factors the output pass needs, kept in registers
// across the chunk (item j: step tid / CC + j * KS).
template <int NI>
struct EpiKeep {
    float fz[NI], sg[NI];   // dout silu'(z), softplus'(x)
};

// The per-(t, d) terms of one staged chunk: Delta (zero past the sequence
// and the CTA's channels, so such steps leave the recurrence unchanged),
// Delta u, dy, u into s_td; B and C as float32 into s_BC; with kMain also the
// dz factor dout silu'(z) and softplus'(x) into *keep.  bias: delta_bias of
// this thread's channel.

template <typename T, int N, bool kMain>
__device__ __forceinline__ void chunk_terms(const unsigned char* slot, unsigned char* sm, const BwdArgs& p,
                                            const Geo& q, int64_t ch, float bias, int tid,
                                            EpiKeep<2 * BwCfg<T, N>::HP>* keep = nullptr) {
    using CF = BwCfg<T, N>;
    constexpr int CC = CF::CC;
    constexpr bool kFast = !std::is_same<T, float>::value;
    const T* tu = reinterpret_cast<const T*>(slot);
    const T* tx = reinterpret_cast<const T*>(slot + CF::TILE);
    const T* tz = reinterpret_cast<const T*>(slot + 2 * CF::TILE);
    const T* to = reinterpret_cast<const T*>(slot + 3 * CF::TILE);
    float4* s_td = reinterpret_cast<float4*>(sm + CF::O_TD);
    const int c = tid % CC;
    const bool cok = q.d0 + c < q.dend;
#pragma unroll
    for (int j = 0; j < CF::HP; ++j) {
        const int k0 = tid / CC + j * CF::KS, k1 = k0 + kK / 2;
        const int o0 = k0 * CC + c, o1 = k1 * CC + c;
        const bool ok0 = cok && ch * kK + k0 < p.seqlen, ok1 = cok && ch * kK + k1 < p.seqlen;
        const float2 x = make_float2(to_f32(tx[o0]) + bias, to_f32(tx[o1]) + bias);
        float2 u2 = make_float2(ok0 ? to_f32(tu[o0]) : 0.f, ok1 ? to_f32(tu[o1]) : 0.f);
        const float2 do2 = make_float2(to_f32(to[o0]), to_f32(to[o1]));
        float2 dl, sg = make_float2(1.f, 1.f);
        if (p.softplus) softplus_and_sigmoid2<kFast>(x, dl, sg);
        else dl = x;
        dl = make_float2(ok0 ? dl.x : 0.f, ok1 ? dl.y : 0.f);
        float2 dy = do2, fz = make_float2(0.f, 0.f);
        if (p.z) {
            const float2 zz = make_float2(to_f32(tz[o0]), to_f32(tz[o1]));
            const float2 sz = sigmoid2<kFast>(zz);
            dy = mul2(do2, mul2(zz, sz));
            if constexpr (kMain) {
                // silu'(z) = s (1 + z (1 - s))
                const float2 one = splat2(1.f);
                fz = mul2(do2, mul2(sz, fma2(zz, add2(one, mul2(sz, splat2(-1.f))), one)));
            }
        }
        const float2 du = mul2(dl, u2);
        s_td[o0] = make_float4(dl.x, du.x, dy.x, u2.x);
        s_td[o1] = make_float4(dl.y, du.y, dy.y, u2.y);
        if constexpr (kMain) {
            keep->fz[j] = fz.x, keep->sg[j] = sg.x;
            keep->fz[j + CF::HP] = fz.y, keep->sg[j + CF::HP] = sg.y;
        }
    }
    // B and C rows [N][K] -> float32 [K][N]
    const T* tb = reinterpret_cast<const T*>(slot + 4 * CF::TILE);
    float* s_bc = reinterpret_cast<float*>(sm + CF::O_BC);
    for (int i = tid; i < 2 * N * kK; i += kThreads) {   // i: destination order [which][k][n]
        const int which = i / (N * kK), r = i - which * N * kK, k = r / N, n = r - k * N;
        s_bc[i] = to_f32(tb[which * N * kK + n * kK + k]);
    }
}

// ------------------------------------------------------------ pass 1

template <typename T, int N>
__global__ void __launch_bounds__(kThreads, 5)
bwd_local_kernel(const BwdArgs p, const BwdWs w) {
    using CF = BwCfg<T, N>;
    constexpr int R = CF::R, CPW = CF::CPW, CC = CF::CC;
    constexpr bool kFast = !std::is_same<T, float>::value;
    extern __shared__ __align__(16) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane % R;
    const int cl = warp * CPW + lane / R;
    const Geo q = make_geo<CC>(p, w);
    const int64_t d = q.d0 + cl;
    const bool ch_ok = d < q.dend;
    const int64_t dim = p.dim;
    float2 A0 = make_float2(0.f, 0.f), A1 = A0;
    if (ch_ok) {
        const float* a = p.A + d * N + 4 * g;   // 4-byte alignment only
        A0 = make_float2(a[0] * kLog2e, a[1] * kLog2e);
        A1 = make_float2(a[2] * kLog2e, a[3] * kLog2e);
    }
    const int cb = q.d0 + tid % CC;
    const float bias = (p.delta_bias && cb < q.dend) ? p.delta_bias[cb] : 0.f;
    const float4* s_td = reinterpret_cast<const float4*>(sm + CF::O_TD);
    const float4* s_B4 = reinterpret_cast<const float4*>(sm + CF::O_BC);
    const float4* s_C4 = s_B4 + kK * N / 4;
    const bool vec = w.vec != 0;
    Stager<T, N> st;
    if (vec) st.init(p, q, tid);

    float2 h0 = make_float2(0.f, 0.f), h1 = h0, L0 = h0, L1 = h0;
    float2 Q0 = make_float2(1.f, 1.f), Q1 = Q0;
    float cum = 0.f;
    const int64_t n_ch = q.c_end - q.c_begin;
#pragma unroll 1
    for (int j = 0; j < kStages - 1; ++j)
        if (j < n_ch) stage_chunk<T, N>(st, sm + j * CF::STAGE, p, q, q.c_begin + j, vec, tid);
        else if (vec) cp_async_commit();
#pragma unroll 1
    for (int64_t i = 0; i < n_ch; ++i) {
        const int64_t c = q.c_begin + i;
        if (vec) cp_async_wait<kStages - 2>();
        __syncthreads();
        {
            const int64_t nx = i + kStages - 1;
            if (nx < n_ch) stage_chunk<T, N>(st, sm + (nx % kStages) * CF::STAGE, p, q, q.c_begin + nx, vec, tid);
            else if (vec) cp_async_commit();
        }
        chunk_terms<T, N, false>(sm + (i % kStages) * CF::STAGE, sm, p, q, c, bias, tid);
        if (ch_ok) {
            *reinterpret_cast<float4*>(w.ckpt + ((q.b * w.nch + c) * dim + d) * N + 4 * g) =
                make_float4(h0.x, h0.y, h1.x, h1.y);
            if (g == 0) w.cum[(q.b * w.nch + c) * dim + d] = cum;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            const float4 td = s_td[k * CC + cl];
            const float4 Bq = s_B4[k * R + g], Cq = s_C4[k * R + g];
            const float2 dl2 = splat2(td.x), du2 = splat2(td.y), dy2 = splat2(td.z);
            const float2 e0 = mul2(dl2, A0), e1 = mul2(dl2, A1);
            const float2 a0 = make_float2(decay_exp2<kFast>(e0.x), decay_exp2<kFast>(e0.y));
            const float2 a1 = make_float2(decay_exp2<kFast>(e1.x), decay_exp2<kFast>(e1.y));
            h0 = fma2(a0, h0, mul2(du2, make_float2(Bq.x, Bq.y)));
            h1 = fma2(a1, h1, mul2(du2, make_float2(Bq.z, Bq.w)));
            Q0 = mul2(Q0, a0);
            Q1 = mul2(Q1, a1);
            L0 = fma2(Q0, mul2(make_float2(Cq.x, Cq.y), dy2), L0);
            L1 = fma2(Q1, mul2(make_float2(Cq.z, Cq.w), dy2), L1);
            cum += td.x;
        }
    }
    if (ch_ok) {
        const int64_t o = ((q.b * w.nseg + q.sgm) * dim + d) * N + 4 * g;
        *reinterpret_cast<float4*>(w.aggQ + o) = make_float4(Q0.x, Q0.y, Q1.x, Q1.y);
        *reinterpret_cast<float4*>(w.aggH + o) = make_float4(h0.x, h0.y, h1.x, h1.y);
        *reinterpret_cast<float4*>(w.aggL + o) = make_float4(L0.x, L0.y, L1.x, L1.y);
    }
}

// ------------------------------------------------------------ combine

__global__ void __launch_bounds__(256) bwd_combine_kernel(const BwdArgs p, const BwdWs w) {
    constexpr int kB = 8;   // segments whose aggregates are loaded together
    const int64_t per_b = p.dim * p.dstate;
    const int64_t total = p.batch * per_b;
    const int64_t S = w.nseg;
    const float* __restrict__ aQ = w.aggQ;
    float* __restrict__ aH = w.aggH;
    float* __restrict__ aL = w.aggL;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / per_b, r = i - b * per_b;
        const int64_t o0 = b * S * per_b + r;   // segment s at o0 + s * per_b
        float H = p.h0 ? p.h0[i] : 0.f;
        for (int64_t s0 = 0; s0 < S; s0 += kB) {
            float q[kB], he[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j)
                if (s0 + j < S) q[j] = aQ[o0 + (s0 + j) * per_b], he[j] = aH[o0 + (s0 + j) * per_b];
#pragma unroll
            for (int j = 0; j < kB; ++j)
                if (s0 + j < S) {
                    aH[o0 + (s0 + j) * per_b] = H;
                    H = fmaf(q[j], H, he[j]);
                }
        }
        float rho = p.dlast ? p.dlast[i] : 0.f;
        for (int64_t s1 = S; s1 > 0; s1 -= kB) {
            float q[kB], lm[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j)
                if (s1 - 1 - j >= 0) q[j] = aQ[o0 + (s1 - 1 - j) * per_b], lm[j] = aL[o0 + (s1 - 1 - j) * per_b];
#pragma unroll
            for (int j = 0; j < kB; ++j)
                if (s1 - 1 - j >= 0) {
                    aL[o0 + (s1 - 1 - j) * per_b] = rho;
                    rho = fmaf(q[j], rho, lm[j]);
                }
        }
        if (p.dh0) p.dh0[i] = rho;
    }
}

// ------------------------------------------------------------ pass 2

template <typename T, int N>
__global__ void __launch_bounds__(kThreads, 4)
bwd_main_kernel(const BwdArgs p, const BwdWs w) {
    using CF = BwCfg<T, N>;
    constexpr int R = CF::R, CPW = CF::CPW, CC = CF::CC;
    constexpr bool kFast = !std::is_same<T, float>::value;
    extern __shared__ __align__(16) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane % R;
    const int cl = warp * CPW + lane / R;
    const Geo q = make_geo<CC>(p, w);
    const int64_t d = q.d0 + cl;
    const bool ch_ok = d < q.dend;
    const int64_t dim = p.dim, L = p.seqlen;
    // the segment's entering state H_s stays in global memory (read per
    // chunk, an L1 hit) to keep registers for the chunk's states
    const int64_t seg_o = ((q.b * w.nseg + q.sgm) * dim + d) * N + 4 * g;
    float2 A0 = make_float2(0.f, 0.f), A1 = A0, mu0 = A0, mu1 = A0;
    if (ch_ok) {
        const float* a = p.A + d * N + 4 * g;   // 4-byte alignment only
        A0 = make_float2(a[0] * kLog2e, a[1] * kLog2e);
        A1 = make_float2(a[2] * kLog2e, a[3] * kLog2e);
        const float4 rh = *reinterpret_cast<const float4*>(w.aggL + seg_o);
        mu0 = make_float2(rh.x, rh.y);
        mu1 = make_float2(rh.z, rh.w);
    }
    // this thread's channel for the per-(t, d) work; its bias and D, and its
    // dD and dbias partial sums, live in shared memory
    const int ct = tid % CC;
    const int dt = q.d0 + ct;
    const bool tok_c = dt < q.dend;
    float2* s_par = reinterpret_cast<float2*>(sm + CF::O_PAR);
    float2* s_acc = reinterpret_cast<float2*>(sm + CF::O_ACC);
    if (tid < CC)
        s_par[tid] = make_float2((p.delta_bias && tok_c) ? p.delta_bias[dt] : 0.f, (p.D && tok_c) ? p.D[dt] : 0.f);
    s_acc[tid] = make_float2(0.f, 0.f);

    const float4* s_td = reinterpret_cast<const float4*>(sm + CF::O_TD);
    const float4* s_B4 = reinterpret_cast<const float4*>(sm + CF::O_BC);
    const float4* s_C4 = s_B4 + kK * N / 4;
    float* s_yp = reinterpret_cast<float*>(sm + CF::O_YP);
    float* s_sd = reinterpret_cast<float*>(sm + CF::O_SD);
    float4* s_P = reinterpret_cast<float4*>(sm + CF::O_P);
    const bool vec = w.vec != 0;
    float2 dA0 = make_float2(0.f, 0.f), dA1 = dA0;

    const int64_t n_ch = q.c_end - q.c_begin;
    // staging order: the segment's chunks from the last one back
#pragma unroll 1
    for (int j = 0; j < kStages - 1; ++j)
        if (j < n_ch) stage_chunk_direct<T, N>(sm + j * CF::STAGE, p, q, q.c_end - 1 - j, vec, tid);
        else if (vec) cp_async_commit();
#pragma unroll 1
    for (int64_t i = 0; i < n_ch; ++i) {
        const int64_t c = q.c_end - 1 - i;
        const int64_t t0 = c * kK;
        if (vec) cp_async_wait<kStages - 2>();
        __syncthreads();
        {
            const int64_t nx = i + kStages - 1;
            if (nx < n_ch) stage_chunk_direct<T, N>(sm + (nx % kStages) * CF::STAGE, p, q, q.c_end - 1 - nx, vec, tid);
            else if (vec) cp_async_commit();
        }
        // the stored local state entering the chunk, the sum of Delta before
        // it within the segment, and H_s (loads issued before the chunk's terms)
        float4 ckc = make_float4(0.f, 0.f, 0.f, 0.f), hs = ckc;
        float cmc = 0.f;
        if (ch_ok) {
            ckc = *reinterpret_cast<const float4*>(w.ckpt + ((q.b * w.nch + c) * dim + d) * N + 4 * g);
            cmc = w.cum[(q.b * w.nch + c) * dim + d];
            hs = *reinterpret_cast<const float4*>(w.aggH + seg_o);
        }
        EpiKeep<2 * CF::HP> keep;
        chunk_terms<T, N, true>(sm + (i % kStages) * CF::STAGE, sm, p, q, c, s_par[ct].x, tid, &keep);
        __syncthreads();
        // the true state entering the chunk: local state + exp(A sum Delta) H_s
        const float2 cm2 = splat2(cmc);
        const float2 q0 = mul2(cm2, A0), q1 = mul2(cm2, A1);
        const float2 hin0 = fma2(make_float2(decay_exp2<kFast>(q0.x), decay_exp2<kFast>(q0.y)),
                                 make_float2(hs.x, hs.y), make_float2(ckc.x, ckc.y));
        const float2 hin1 = fma2(make_float2(decay_exp2<kFast>(q1.x), decay_exp2<kFast>(q1.y)),
                                 make_float2(hs.z, hs.w), make_float2(ckc.z, ckc.w));
        // The chunk in parts of kHold steps, the last part first: the state
        // entering the part (recomputed through the earlier steps), the
        // part's states (readout partials stored once), then the adjoint back
        // over the part.  The decays are recomputed in the adjoint rather
        // than held, keeping registers for the states.
        const bool hi = (lane & 16) != 0;
#pragma unroll
        for (int part = kK / kHold - 1; part >= 0; --part) {
            const int kb = part * kHold;
            float2 hp0 = hin0, hp1 = hin1;
#pragma unroll
            for (int k = 0; k < kb; ++k) {
                const float4 td = s_td[k * CC + cl];
                const float4 Bq = s_B4[k * R + g];
                const float2 dl2 = splat2(td.x), du2 = splat2(td.y);
                const float2 e0 = mul2(dl2, A0), e1 = mul2(dl2, A1);
                hp0 = fma2(make_float2(decay_exp2<kFast>(e0.x), decay_exp2<kFast>(e0.y)), hp0,
                           mul2(du2, make_float2(Bq.x, Bq.y)));
                hp1 = fma2(make_float2(decay_exp2<kFast>(e1.x), decay_exp2<kFast>(e1.y)), hp1,
                           mul2(du2, make_float2(Bq.z, Bq.w)));
            }
            float2 hk0[kHold], hk1[kHold];
#pragma unroll
            for (int j = 0; j < kHold; ++j) {
                const int k = kb + j;
                const float4 td = s_td[k * CC + cl];
                const float4 Bq = s_B4[k * R + g], Cq = s_C4[k * R + g];
                const float2 dl2 = splat2(td.x), du2 = splat2(td.y);
                const float2 e0 = mul2(dl2, A0), e1 = mul2(dl2, A1);
                const float2 a0 = make_float2(decay_exp2<kFast>(e0.x), decay_exp2<kFast>(e0.y));
                const float2 a1 = make_float2(decay_exp2<kFast>(e1.x), decay_exp2<kFast>(e1.y));
                hk0[j] = fma2(a0, j ? hk0[j - 1] : hp0, mul2(du2, make_float2(Bq.x, Bq.y)));
                hk1[j] = fma2(a1, j ? hk1[j - 1] : hp1, mul2(du2, make_float2(Bq.z, Bq.w)));
                const float2 yv = fma2(make_float2(Cq.z, Cq.w), hk1[j], mul2(make_float2(Cq.x, Cq.y), hk0[j]));
                s_yp[(k * CC + cl) * R + g] = yv.x + yv.y;
            }
#pragma unroll
            for (int j = kHold - 1; j >= 0; --j) {
                const int k = kb + j;
                const float4 td = s_td[k * CC + cl];
                const float4 Bq = s_B4[k * R + g], Cq = s_C4[k * R + g];
                const float2 dl2 = splat2(td.x), du2 = splat2(td.y), dy2 = splat2(td.z);
                const float2 B0 = make_float2(Bq.x, Bq.y), B1 = make_float2(Bq.z, Bq.w);
                const float2 e0 = mul2(dl2, A0), e1 = mul2(dl2, A1);
                const float2 a0 = make_float2(decay_exp2<kFast>(e0.x), decay_exp2<kFast>(e0.y));
                const float2 a1 = make_float2(decay_exp2<kFast>(e1.x), decay_exp2<kFast>(e1.y));
                const float2 l0 = fma2(make_float2(Cq.x, Cq.y), dy2, mu0);
                const float2 l1 = fma2(make_float2(Cq.z, Cq.w), dy2, mu1);
                mu0 = mul2(a0, l0);
                mu1 = mul2(a1, l1);
                const float2 w0 = mul2(mu0, j ? hk0[j - 1] : hp0);
                const float2 w1 = mul2(mu1, j ? hk1[j - 1] : hp1);
                dA0 = fma2(dl2, w0, dA0);
                dA1 = fma2(dl2, w1, dA1);
                const float2 aw = fma2(A1, w1, mul2(A0, w0));
                const float2 lb = fma2(B1, l1, mul2(B0, l0));
                float v0 = lb.x + lb.y, v1 = aw.x + aw.y;
                // sums over the channel's R lanes: transposed, lane g ends with
                // sum lambda B (g even) or sum A w (g odd)
                const int o = k * CC + cl;
                if constexpr (R == 1) {
                    reinterpret_cast<float2*>(s_sd)[o] = make_float2(v0, v1);
                } else {
                    const bool odd = (g & 1) != 0;
                    float keep = odd ? v1 : v0;
                    keep += __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                    if constexpr (R == 4) keep += __shfl_xor_sync(0xffffffffu, keep, 2);
                    if (g < 2) s_sd[2 * o + g] = keep;
                }
                // dB (lambda Delta u) and dC (h dy) quads; the lane pairs 16 apart
                // (same states, other channels) add them up, the lower lane keeps dB
                const float2 db0 = mul2(l0, du2), db1 = mul2(l1, du2);
                const float2 dc0 = mul2(hk0[j], dy2), dc1 = mul2(hk1[j], dy2);
                float4 keep = hi ? make_float4(dc0.x, dc0.y, dc1.x, dc1.y) : make_float4(db0.x, db0.y, db1.x, db1.y);
                const float4 send = hi ? make_float4(db0.x, db0.y, db1.x, db1.y) : make_float4(dc0.x, dc0.y, dc1.x, dc1.y);
                keep.x += __shfl_xor_sync(0xffffffffu, send.x, 16);
                keep.y += __shfl_xor_sync(0xffffffffu, send.y, 16);
                keep.z += __shfl_xor_sync(0xffffffffu, send.z, 16);
                keep.w += __shfl_xor_sync(0xffffffffu, send.w, 16);
                s_P[k * kThreads + tid] = keep;
            }
        }
        __syncthreads();
        // per-(t, d) outputs of the chunk
        {
            const float2* s_sd2 = reinterpret_cast<const float2*>(sm + CF::O_SD);
            const float Dd = s_par[ct].y;
            float accD = 0.f, accb = 0.f;
#pragma unroll
            for (int j = 0; j < 2 * CF::HP; ++j) {
                const int k = tid / CC + j * CF::KS;
                const int64_t t = t0 + k;
                const int o = k * CC + ct;
                const float4 ta = s_td[o];
                const float2 sd = s_sd2[o];
                const float dlj = ta.x, dyj = ta.z, uj = ta.w;
                float y = 0.f;
                if constexpr (R == 4) {
                    const float4 v = reinterpret_cast<const float4*>(s_yp)[o];
                    y = (v.x + v.y) + (v.z + v.w);
                } else if constexpr (R == 2) {
                    const float2 v = reinterpret_cast<const float2*>(s_yp)[o];
                    y = v.x + v.y;
                } else {
                    y = s_yp[o];
                }
                y = fmaf(Dd, uj, y);
                const float du = fmaf(Dd, dyj, dlj * sd.x);
                float dd = fmaf(uj, sd.x, kLn2 * sd.y);
                if (p.softplus) dd *= keep.sg[j];
                const bool ok = tok_c && t < L;
                accD = fmaf(dyj, uj, accD);
                accb += ok ? dd : 0.f;
                if (ok) {
                    const int64_t gi = (q.b * L + t) * dim + dt;
                    static_cast<T*>(p.du)[gi] = from_f32<T>(du);
                    static_cast<T*>(p.ddelta)[gi] = from_f32<T>(dd);
                    if (p.z && p.dz) static_cast<T*>(p.dz)[gi] = from_f32<T>(keep.fz[j] * y);
                }
            }
            const float2 a = s_acc[tid];
            s_acc[tid] = make_float2(a.x + accD, a.y + accb);
        }
        // dB, dC of the chunk: each (step, which, state quad) summed over the
        // CTA's channels by TPS threads, then added to global memory
        {
            constexpr int TPS = 8 / R;                 // threads per sum
            constexpr int LPW = 16 / R;                // lanes per warp holding one sum's quads
            const int si = tid / TPS, part = tid % TPS;
            const int k = si / (2 * R), rem = si % (2 * R), which = rem / R, gq = rem % R;
            float2 a01 = make_float2(0.f, 0.f), a23 = a01;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int j = part + TPS * m;
                const int wv = j / LPW, cw = which * LPW + j % LPW;
                const float4 v = s_P[k * kThreads + wv * 32 + gq + R * cw];
                a01 = add2(a01, make_float2(v.x, v.y));
                a23 = add2(a23, make_float2(v.z, v.w));
            }
            float4 acc = make_float4(a01.x, a01.y, a23.x, a23.y);
#pragma unroll
            for (int o = 1; o < TPS; o <<= 1) {
                acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
                acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
                acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
                acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
            }
            if (w.red4) {
                // the sums as [which][n][k], then one 16-byte reduction per
                // (which, state, four steps)
                float* s_sum = reinterpret_cast<float*>(sm + CF::O_SUM);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    if (jj % TPS == part) s_sum[(which * N + 4 * gq + jj) * CF::SUMROW + k] = comp(acc, jj);
                __syncthreads();
                constexpr int NQ = 2 * N * kK / 4;
                for (int i2 = tid; i2 < NQ; i2 += kThreads) {
                    const int wh = i2 / (2 * N), n = (i2 % (2 * N)) / 2, kq = i2 % 2;
                    const int64_t t = t0 + 4 * kq;
                    if (t < L)
                        red_add_v4((wh ? p.dC : p.dB) + (q.blk * N + n) * L + t,
                                   reinterpret_cast<const float4*>(s_sum + (wh * N + n) * CF::SUMROW)[kq]);
                }
            } else {
                const int64_t t = t0 + k;
                if (t < L) {
                    float* dst = (which ? p.dC : p.dB) + (q.blk * N + 4 * gq) * L + t;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (jj % TPS == part) atomicAdd(dst + jj * L, comp(acc, jj));
                }
            }
        }
    }
    if (ch_ok) {
        float* da = p.dA + d * N + 4 * g;
        atomicAdd(da, dA0.x);
        atomicAdd(da + 1, dA0.y);
        atomicAdd(da + 2, dA1.x);
        atomicAdd(da + 3, dA1.y);
    }
    // dD, dbias: the KS threads on one channel, then one atomic each
    if (p.dD || p.dbias) {
        __syncthreads();
        if (tid < CC && tok_c) {
            float2 s2 = s_acc[tid];
            for (int j = 1; j < CF::KS; ++j) {
                const float2 v = s_acc[tid + j * CC];
                s2.x += v.x;
                s2.y += v.y;
            }
            if (p.dD) atomicAdd(p.dD + dt, s2.x);
            if (p.dbias) atomicAdd(p.dbias + dt, s2.y);
        }
    }
}

template <typename T, int N>
cudaError_t launch_bwd_t(const BwdArgs& a, const BwdWs& w, cudaStream_t s) {
    using CF = BwCfg<T, N>;
    // shared-memory sizes of both passes, set once per device
    static DeviceMemo memo;
    int dev = 0, set = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    cudaError_t err = cudaSuccess;
    if (!memo.get(dev, [&](int& r) {
            err = cudaFuncSetAttribute(bwd_local_kernel<T, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       CF::SMEM1);
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(bwd_main_kernel<T, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           CF::SMEM3);
            r = 1;
            return err == cudaSuccess;
        }, &set))
        return err;
    const int64_t gx = a.ngroups * ((a.gch + CF::CC - 1) / CF::CC);
    if (gx > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)gx, (unsigned)w.nseg, (unsigned)a.batch);
    bwd_local_kernel<T, N><<<grid, kThreads, CF::SMEM1, s>>>(a, w);
    if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
    const int64_t total = a.batch * a.dim * N;
    const int64_t nb = std::min<int64_t>((total + 255) / 256, 65535 * 16);
    bwd_combine_kernel<<<(unsigned)nb, 256, 0, s>>>(a, w);
    if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
    bwd_main_kernel<T, N><<<grid, kThreads, CF::SMEM3, s>>>(a, w);
    return cudaGetLastError();
}

constexpr int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

struct WsSizes {
    int64_t nch, nseg, ckpt, cum, agg;
};

WsSizes ws_sizes(int64_t batch, int64_t dim, int64_t seqlen, int dstate) {
    WsSizes z;
    z.nch = (seqlen + kK - 1) / kK;
    z.nseg = bwd_segments(z.nch);
    z.ckpt = align256(batch * z.nch * dim * dstate * 4);
    z.cum = align256(batch * z.nch * dim * 4);
    z.agg = align256(batch * z.nseg * dim * dstate * 4);
    return z;
}

bool al16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int64_t bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate) {
    const WsSizes z = ws_sizes(batch, dim, seqlen, dstate);
    return z.ckpt + z.cum + 3 * z.agg;
}

cudaError_t launch_scan_bwd(const BwdArgs& a, DType dt, void* workspace, int sms, cudaStream_t s) {
    (void)sms;
    // the accumulated gradients start from zero
    const int64_t N = a.dstate;
    cudaError_t e = cudaMemsetAsync(a.dA, 0, a.dim * N * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dB, 0, a.batch * a.ngroups * N * a.seqlen * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dC, 0, a.batch * a.ngroups * N * a.seqlen * 4, s);
    if (e == cudaSuccess && a.dD) e = cudaMemsetAsync(a.dD, 0, a.dim * 4, s);
    if (e == cudaSuccess && a.dbias) e = cudaMemsetAsync(a.dbias, 0, a.dim * 4, s);
    if (e != cudaSuccess) return e;
    const WsSizes z = ws_sizes(a.batch, a.dim, a.seqlen, a.dstate);
    char* base = static_cast<char*>(workspace);
    BwdWs w;
    w.ckpt = reinterpret_cast<float*>(base);
    w.cum = reinterpret_cast<float*>(base + z.ckpt);
    w.aggQ = reinterpret_cast<float*>(base + z.ckpt + z.cum);
    w.aggH = reinterpret_cast<float*>(base + z.ckpt + z.cum + z.agg);
    w.aggL = reinterpret_cast<float*>(base + z.ckpt + z.cum + 2 * z.agg);
    w.nch = z.nch;
    w.cps = (z.nch + z.nseg - 1) / z.nseg;
    w.nseg = (z.nch + w.cps - 1) / w.cps;
    const int64_t es = dt == DType::BF16 ? 2 : 4;
    // 16-byte staging: every staged row piece starts on a 16-byte boundary
    w.vec = al16(a.u) && al16(a.delta) && al16(a.z) && al16(a.dout) && al16(a.B) && al16(a.C) &&
            (a.dim * es) % 16 == 0 && (a.gch * es) % 16 == 0 && (a.seqlen * es) % 16 == 0;
    w.red4 = al16(a.dB) && al16(a.dC) && a.seqlen % 4 == 0;
    const bool bf = dt == DType::BF16;
    switch (a.dstate) {
        case 4: return bf ? launch_bwd_t<__nv_bfloat16, 4>(a, w, s) : launch_bwd_t<float, 4>(a, w, s);
        case 8: return bf ? launch_bwd_t<__nv_bfloat16, 8>(a, w, s) : launch_bwd_t<float, 8>(a, w, s);
        case 16: return bf ? launch_bwd_t<__nv_bfloat16, 16>(a, w, s) : launch_bwd_t<float, 16>(a, w, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
