// scan_seg.cu -- the segmented selective scan (float32 activations, or
// d_state 4 / 8), the B/C staging kernel it shares with the tensor-memory
// kernels' hosts, and the TMA capability checks of the fast paths.
//
// Computes, per (batch b, channel d), the recurrence of the Mamba selective
// SSM ("Mamba: Selective State Space Models" README, "State Space Model",
// "Selective Mechanism", "Efficient Scan"):
//     Delta_t = softplus(delta_raw_t + delta_bias)
//     h_t     = exp(Delta_t A) * h_{t-1} + Delta_t B_t u_t
//     out_t   = (C_t . h_t + D u_t) * silu(z_t)
//
// A lane keeps 4 of a channel's N states in registers (R = N / 4 lanes per
// channel).  Pairs of warps on one scheduler scan CW = 32 / R channels of one
// batch row straight through K-step chunks: a helper warp issues the TMA
// loads of the u, delta_raw and z tiles and computes the per-(t, d) terms into
// a double buffer, the main warp runs the recurrence with B and C from the
// staged rows in shared memory, the readout over the R lanes of each channel
// and the output store.  Every (batch, channel group) chain is cut into S
// segments taken by different warps in turn; the state passes between
// segments through the workspace under a bounded release/acquire flag wait.
//
// Waits are bounded: a wait that exceeds ~1 s sets a bit in the device error
// word (ssm_device_error) and the warp stops early; nothing in the kernel can
// spin forever.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "device_memo.h"
#include "scan_common.cuh"
#include "ssm_internal.cuh"

namespace ssm {

namespace {


// ===================================================================
// Segmented direct scan: one warp scans CW channels straight through
// K-step chunks; every (batch, unit) chain is cut into S segments that
// different warps take in turn, so the work divides evenly over all warps.
// ===================================================================


// Four consecutive staged values as float32: one 8-byte shared load and a
// bit-shift unpack for bf16, one 16-byte load for float32.
template <typename T>
__device__ __forceinline__ float4 ld_quad(const T* p);
template <>
__device__ __forceinline__ float4 ld_quad<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 ld_quad<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

template <typename T, int N_>
struct SegCfg {
    static constexpr int N = N_;
    static constexpr int G = 4;                 // states per lane
    static constexpr int R = N / G;             // lanes per channel
    static constexpr int CW = 32 / R;           // channels per chain (one warp-width)
    // Steps per chunk: 64 for 16 states in bf16 (per-chunk costs spread over
    // more steps), 16 for 4 states (32-channel tiles), 32 otherwise.
    static constexpr int K = (N == 16 && sizeof(T) == 2) ? 64 : (N == 4 ? 16 : 32);
    static constexpr int P = (N == 8 && sizeof(T) == 4) ? 2 : 4;   // ring slots per pair (a power of two)
    static constexpr int PAIRS = 4;             // (main, helper) warp pairs per CTA: one per scheduler
    static constexpr int THREADS = 64 * PAIRS;
    static constexpr int KR = K / R;            // items / finished steps per lane
    static constexpr int ES = (int)sizeof(T);
    static constexpr int TILE = K * CW * ES;
    static constexpr int BC = K * 2 * N * ES;   // staged B|C rows, in the activation type
    static constexpr int align128(int x) { return (x + 127) / 128 * 128; }
    static constexpr int SLOT_U = 0;
    static constexpr int SLOT_D = align128(TILE);
    static constexpr int SLOT_Z = SLOT_D + align128(TILE);
    static constexpr int SLOT_BC = SLOT_Z + align128(TILE);
    static constexpr int SLOT = align128(SLOT_BC + BC);
    static constexpr int RS2 = 34;              // float2 stride of a step-pair row of the reduction buffer
    static constexpr int HALF = K * CW * 8;     // one float2 per (step, channel)
    // per-pair layout
    static constexpr int P_RING = 0;                              // [P] slots
    static constexpr int P_DP = P_RING + P * SLOT;                 // [2][K][CW] float2 (Delta, Delta u)
    static constexpr int P_SG = P_DP + 2 * HALF;                   // [2][K][CW] float2 (u, silu z)
    static constexpr int P_RED = P_SG + 2 * HALF;                  // [K/2][RS2] float2
    static constexpr int P_OUT = P_RED + (R > 1 ? align128((K / 2) * RS2 * 8) : 0);   // [3] out tiles
    static constexpr int OUT = align128(TILE);
    static constexpr int P_BAR = P_OUT + 3 * OUT;                  // full[P], dpf[2], done[2]
    static constexpr int PAIR_BYTES = align128(P_BAR + (P + 4) * 8);
    static constexpr int SMEM = PAIRS * PAIR_BYTES;
    static_assert(SMEM <= 227 * 1024, "a CTA's shared memory must fit an SM");
    static_assert(K % 8 == 0 && 64 % K == 0, "chunks tile the 64-step padded sequence");
    static_assert((P & (P - 1)) == 0 && P >= 2, "ring depth is a power of two, at least two");
};

struct SegParams {
    const float* A;
    const float* D;
    const float* delta_bias;
    const void* bc;         // staged B|C, [batch * ngroups][lpad][2N] in the activation type
    float* last_state;
    float* seg_state;       // [M][CW][N] f32: state handed between segments
    int* seg_flag;          // [M]: number of finished segments of each chain
    int dim, seqlen;
    int64_t lpad;
    int units;              // channel groups per batch row
    int M;                  // chains = batch * units
    int S;                  // segments per chain
    int cps;                // chunks per segment
    int workers;            // (main, helper) pairs in the grid
    const float* h0;        // initial state (batch, dim, N) or null
    int ngroups, gch;       // B/C groups, channels per group (a multiple of CW)
};

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *flag >= want; false after ~1 s.
__device__ __forceinline__ bool flag_wait(const int* flag, int want) {
    if (ld_acquire(flag) >= want) return true;
    const unsigned long long t0 = globaltimer();
    while (ld_acquire(flag) < want)
        if (globaltimer() - t0 > wait_limit_ns()) return false;
    return true;
}

// One worker is a (main, helper) pair of warps on the same scheduler; it
// walks its tasks (segment s of chain m, task = s * M + m) in slot order.
//   helper: issues the TMA loads of its chunks (P in flight), then for each
//           chunk computes the per-(t, d) terms -- Delta = softplus(delta_raw
//           + bias), Delta u, u, silu(z) -- into a double buffer and signals
//           "prologue done";
//   main:   waits for it, runs the recurrence over the chunk (exp(Delta A),
//           Delta B u, the state update, the per-lane readout C . h), sums the
//           R lanes of each channel, applies D u and the gate, stores the
//           output tile by TMA and signals "chunk done", which frees the
//           double buffer and the ring slot for the helper.
// The scheduler interleaves the helper's SFU-heavy prologue with the main
// warp's dependency stalls.
template <typename T, int N, bool kFast, bool kSoftplus, bool kGate>
__global__ void __launch_bounds__(SegCfg<T, N>::THREADS, 1)
scan_seg_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_d,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_out,
                const SegParams p) {
    using CF = SegCfg<T, N>;
    constexpr int K = CF::K, P = CF::P, R = CF::R, CW = CF::CW, KR = CF::KR, RS2 = CF::RS2;
    constexpr int NP = KR / 2;
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = warp % CF::PAIRS;
    const bool helper = warp >= CF::PAIRS;
    const int ch = lane / R, g = lane % R;
    unsigned char* pb = smem + pair * CF::PAIR_BYTES;
    const uint32_t ring_s = smem_u32(pb + CF::P_RING);
    const uint32_t bar_full = smem_u32(pb + CF::P_BAR);
    const uint32_t bar_dpf = bar_full + 8u * P;
    const uint32_t bar_done = bar_dpf + 16u;
    float2* dpb = reinterpret_cast<float2*>(pb + CF::P_DP);
    float2* sgb = reinterpret_cast<float2*>(pb + CF::P_SG);
    float2* red = reinterpret_cast<float2*>(pb + CF::P_RED);

    const int L = p.seqlen;
    const int nch = (L + K - 1) / K;
    const int T_total = p.M * p.S;
    const int wid = blockIdx.x * CF::PAIRS + pair;

    if (helper && lane == 0) {
        for (int i = 0; i < P; ++i) mbar_init(bar_full + 8u * i, 1);
        for (int i = 0; i < 4; ++i) mbar_init(bar_dpf + 8u * i, 1);   // dpf[2], done[2]
        fence_mbar_init();
    }
    __syncthreads();

    // this lane's items of a chunk, as NP step pairs in an order rotated by g
    // (conflict-free shared-memory rows); the same mapping on both warps
    int tas[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) tas[j] = g * KR + 2 * ((j + g) % NP);

    bool ok = true;
    if (helper) {
        // ------------------------------------------------------------ helper
        constexpr uint32_t tx_bytes = (uint32_t)((kGate ? 3 : 2) * CF::TILE + CF::BC);
        int pf_task = wid, pf_c = 0, pf_end = 0, issued = 0;
        int pf_b = 0, pf_d0 = 0;
        const T* pf_bc = nullptr;
        auto pf_enter = [&](int task) {
            const int sgm = task / p.M, m = task - sgm * p.M;
            pf_b = m / p.units;
            pf_d0 = (m - pf_b * p.units) * CW;
            pf_c = sgm * p.cps;
            pf_end = min(pf_c + p.cps, nch);
            const size_t blk = (size_t)pf_b * p.ngroups + (size_t)(pf_d0 / p.gch);
            pf_bc = static_cast<const T*>(p.bc) + (blk * p.lpad + (size_t)pf_c * K) * (2 * N);
        };
        if (pf_task < T_total) pf_enter(pf_task);
        auto issue_next = [&]() {   // lane 0 only
            while (pf_task < T_total && pf_c >= pf_end) {
                pf_task += p.workers;
                if (pf_task < T_total) pf_enter(pf_task);
            }
            if (pf_task >= T_total) return;
            const int slot = issued & (P - 1);
            const uint32_t base = ring_s + (uint32_t)(slot * CF::SLOT);
            const uint32_t bar = bar_full + 8u * (uint32_t)slot;
            const int t0 = pf_c * K;
            mbar_expect_tx(bar, tx_bytes);
            tma_load_3d(base + CF::SLOT_U, &tm_u, pf_d0, t0, pf_b, bar);
            tma_load_3d(base + CF::SLOT_D, &tm_d, pf_d0, t0, pf_b, bar);
            if constexpr (kGate) tma_load_3d(base + CF::SLOT_Z, &tm_z, pf_d0, t0, pf_b, bar);
            bulk_load(base + CF::SLOT_BC, pf_bc, CF::BC, bar);
            pf_bc += K * 2 * N;
            ++pf_c;
            ++issued;
        };
        if (lane == 0)
            for (int i = 0; i < P; ++i) issue_next();

        int j = 0;        // chunk sequence number of this worker
        int landed = 0;   // chunks whose loads this warp has waited for
        for (int task = wid; task < T_total && ok; task += p.workers) {
            const int sgm = task / p.M, m = task - sgm * p.M;
            const int b = m / p.units;
            const int d = (m - b * p.units) * CW + ch;
            const bool ch_ok = d < p.dim;
            const float2 bias2 = splat2((p.delta_bias && ch_ok) ? p.delta_bias[d] : 0.f);
            const int cb = sgm * p.cps, ce = min(cb + p.cps, nch);
            for (int c = cb; c < ce; ++c, ++j) {
                const int buf = j & 1;
                if (j >= 2) {
                    // the main warp finished chunk j-2: its buffers and ring slot are free
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_done + 8u * buf, (uint32_t)(((j - 2) >> 1) & 1)))) {
                        ok = false;
                        if (lane == 0) raise_error(2u);
                        break;
                    }
                    if (lane == 0) issue_next();
                }
                const int slot = j & (P - 1);
                if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8u * slot, (uint32_t)((j / P) & 1)))) {
                    ok = false;
                    if (lane == 0) raise_error(1u);
                    break;
                }
                ++landed;
                const unsigned char* sb = pb + CF::P_RING + slot * CF::SLOT;
                const T* su = reinterpret_cast<const T*>(sb + CF::SLOT_U);
                const T* sd = reinterpret_cast<const T*>(sb + CF::SLOT_D);
                const T* sz = reinterpret_cast<const T*>(sb + CF::SLOT_Z);
                const int t0 = c * K;
                const bool tail = t0 + K > L;
                float2 uk[NP], xr[NP], zr[NP];
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const int ta = tas[q], tb = ta + 1;
                    uk[q] = make_float2(ld_elem(su + ta * CW + ch), ld_elem(su + tb * CW + ch));
                    xr[q] = make_float2(ld_elem(sd + ta * CW + ch), ld_elem(sd + tb * CW + ch));
                    if constexpr (kGate) zr[q] = make_float2(ld_elem(sz + ta * CW + ch), ld_elem(sz + tb * CW + ch));
                }
                float2 dpv[2 * NP], sgv[2 * NP];
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    float2 dl = add2(xr[q], bias2);
                    if constexpr (kSoftplus) dl = softplus2_path<kFast>(dl);
                    if (tail) dl = mul2(dl, make_float2(t0 + tas[q] < L ? 1.f : 0.f, t0 + tas[q] + 1 < L ? 1.f : 0.f));
                    const float2 du = mul2(dl, uk[q]);
                    float2 gt = splat2(1.f);
                    if constexpr (kGate) gt = seg_silu2<kFast>(zr[q]);
                    dpv[2 * q] = make_float2(dl.x, du.x);
                    dpv[2 * q + 1] = make_float2(dl.y, du.y);
                    sgv[2 * q] = make_float2(uk[q].x, gt.x);
                    sgv[2 * q + 1] = make_float2(uk[q].y, gt.y);
                }
                float2* dp = dpb + buf * (K * CW);
                float2* sg = sgb + buf * (K * CW);
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    dp[tas[q] * CW + ch] = dpv[2 * q];
                    dp[(tas[q] + 1) * CW + ch] = dpv[2 * q + 1];
                    sg[tas[q] * CW + ch] = sgv[2 * q];
                    sg[(tas[q] + 1) * CW + ch] = sgv[2 * q + 1];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_dpf + 8u * buf);
            }
        }
        // Drain: every issued load must land before shared memory is released.
        if (!ok) {
            const int iss = __shfl_sync(0xffffffffu, issued, 0);
            for (int k = landed; k < iss; ++k)
                if (!mbar_wait(bar_full + 8u * (uint32_t)(k & (P - 1)), (uint32_t)((k / P) & 1))) break;
        }
        return;
    }

    // ---------------------------------------------------------------- main
    int j = 0;
    int oslot = 0;
    for (int task = wid; task < T_total && ok; task += p.workers) {
        const int sgm = task / p.M, m = task - sgm * p.M;
        const int b = m / p.units;
        const int d0 = (m - b * p.units) * CW;
        const int d = d0 + ch;
        const bool ch_ok = d < p.dim;
        const int cb = sgm * p.cps, ce = min(cb + p.cps, nch);

        float2 A2[2];
        {
            const float4 a = ch_ok ? *reinterpret_cast<const float4*>(p.A + (size_t)d * N + 4 * g)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            A2[0] = make_float2(a.x * kLog2e, a.y * kLog2e);
            A2[1] = make_float2(a.z * kLog2e, a.w * kLog2e);
        }
        const float2 dskip2 = splat2((p.D && ch_ok) ? p.D[d] : 0.f);

        // state entering the segment
        float2 h0 = make_float2(0.f, 0.f), h1 = make_float2(0.f, 0.f);
        float* hst = p.seg_state + ((size_t)m * CW + ch) * N + 4 * g;
        if (sgm > 0) {
            if (!__all_sync(0xffffffffu, flag_wait(p.seg_flag + m, sgm))) {
                ok = false;
                if (lane == 0) raise_error(4u);
                break;
            }
            const float4 v = __ldcg(reinterpret_cast<const float4*>(hst));
            h0 = make_float2(v.x, v.y);
            h1 = make_float2(v.z, v.w);
        } else if (p.h0 && ch_ok) {
            const float4 v = *reinterpret_cast<const float4*>(p.h0 + ((size_t)b * p.dim + d) * N + 4 * g);
            h0 = make_float2(v.x, v.y);
            h1 = make_float2(v.z, v.w);
        }

        for (int c = cb; c < ce; ++c, ++j) {
            const int buf = j & 1;
            const int slot = j & (P - 1);
            if (!__all_sync(0xffffffffu, mbar_wait(bar_dpf + 8u * buf, (uint32_t)((j >> 1) & 1)) &&
                                             mbar_wait(bar_full + 8u * slot, (uint32_t)((j / P) & 1)))) {
                ok = false;
                if (lane == 0) raise_error(2u);
                break;
            }
            const int t0 = c * K;
            const float2* dp = dpb + buf * (K * CW);
            const float2* sg = sgb + buf * (K * CW);
            const T* sbc = reinterpret_cast<const T*>(pb + CF::P_RING + slot * CF::SLOT + CF::SLOT_BC);

            // ---- the recurrence as a software pipeline over the chunk's K steps:
            // step t loads the Delta/B/C rows of step t+LA, evaluates
            // exp(Delta A) and Delta B u of step t+EA, advances the state by
            // step t (one packed FMA per two states: the only serial work) and
            // reads out C_t . h_t.
            constexpr int LA = 4, EA = 2;
            float2 qv[K];
            float4 bv[K], cv[K];
            float2 dA[K][2], dB[K][2];
            float2 s2v[K / 2];
            auto load_step = [&](int t) {
                qv[t] = dp[t * CW + ch];
                bv[t] = ld_quad<T>(sbc + t * (2 * N) + 4 * g);
                cv[t] = ld_quad<T>(sbc + t * (2 * N) + N + 4 * g);
            };
            auto exp_step = [&](int t) {
                const float2 dl2 = splat2(qv[t].x), du2 = splat2(qv[t].y);
                const float2 e0 = mul2(dl2, A2[0]);
                const float2 e1 = mul2(dl2, A2[1]);
                dA[t][0] = make_float2(decay_exp2<kFast>(e0.x), decay_exp2<kFast>(e0.y));
                dA[t][1] = make_float2(decay_exp2<kFast>(e1.x), decay_exp2<kFast>(e1.y));
                dB[t][0] = mul2(du2, make_float2(bv[t].x, bv[t].y));
                dB[t][1] = mul2(du2, make_float2(bv[t].z, bv[t].w));
            };
#pragma unroll
            for (int t = 0; t < LA; ++t) load_step(t);
#pragma unroll
            for (int t = 0; t < EA; ++t) exp_step(t);
            float2 acc_prev = make_float2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < K; ++t) {
                if (t + LA < K) load_step(t + LA);
                if (t + EA < K) exp_step(t + EA);
                h0 = fma2(dA[t][0], h0, dB[t][0]);
                h1 = fma2(dA[t][1], h1, dB[t][1]);
                const float2 acc = fma2(make_float2(cv[t].z, cv[t].w), h1, mul2(make_float2(cv[t].x, cv[t].y), h0));
                if (t & 1) s2v[t / 2] = make_float2(acc_prev.x + acc_prev.y, acc.x + acc.y);
                acc_prev = acc;
            }

            // ---- sum the R lanes of each channel for this lane's pairs (same rotation)
            float2 yv[NP];
            if constexpr (R == 1) {
#pragma unroll
                for (int q = 0; q < NP; ++q) yv[q] = s2v[tas[q] / 2];
            } else {
#pragma unroll
                for (int t = 0; t < K / 2; ++t) red[t * RS2 + lane] = s2v[t];
                __syncwarp();
                float2 pr[NP][R];
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2* row = red + (tas[q] / 2) * RS2 + ch * R;
#pragma unroll
                    for (int gg = 0; gg < R; ++gg) pr[q][gg] = row[gg];
                }
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    float2 sum = pr[q][0];
#pragma unroll
                    for (int gg = 1; gg < R; ++gg) sum = add2(sum, pr[q][gg]);
                    yv[q] = sum;
                }
            }

            // ---- D u, gate, output tile (triple-buffered; lane 0 owns the TMA
            // store groups: before a tile is rewritten, the store that read it
            // three chunks ago must have finished reading)
            float2 sgl[2 * NP];
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                sgl[2 * q] = sg[tas[q] * CW + ch];
                sgl[2 * q + 1] = sg[(tas[q] + 1) * CW + ch];
            }
            T* so = reinterpret_cast<T*>(pb + CF::P_OUT + oslot * CF::OUT);
            if (lane == 0) bulk_wait_read<2>();
            __syncwarp();
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 uq = make_float2(sgl[2 * q].x, sgl[2 * q + 1].x);
                const float2 gq = make_float2(sgl[2 * q].y, sgl[2 * q + 1].y);
                const float2 y = mul2(fma2(dskip2, uq, yv[q]), gq);
                st_pair<T>(so + tas[q] * CW + ch, so + (tas[q] + 1) * CW + ch, y);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&tm_out, d0, t0, b, smem_u32(so));
                bulk_commit();
                mbar_arrive(bar_done + 8u * buf);   // buffers and ring slot of chunk j are free
            }
            oslot = oslot == 2 ? 0 : oslot + 1;
        }
        if (!ok) break;

        // state leaving the segment
        if (sgm + 1 < p.S) {
            __stcg(reinterpret_cast<float4*>(hst), make_float4(h0.x, h0.y, h1.x, h1.y));
            __threadfence();
            __syncwarp();
            if (lane == 0 && !withhold_handoff(m, sgm)) st_release(p.seg_flag + m, sgm + 1);
        } else if (p.last_state && ch_ok) {
            *reinterpret_cast<float4*>(p.last_state + ((size_t)b * p.dim + d) * N + 4 * g) =
                make_float4(h0.x, h0.y, h1.x, h1.y);
        }
    }
    if (lane == 0) bulk_wait_all();
}

// B and C (rows, N, L) -> staged rows [rows][lpad][B_0..B_{N-1}, C_0..C_{N-1}] of
// type O (the activation type, so that the segmented kernel's per-step reads
// move half the bytes of float32), zero beyond L; rows =
// batch, or batch * ngroups for B and C per channel group.  One CTA per
// (64-step tile, row), transposed through shared memory.
template <typename T, int N, typename O>
__global__ void __launch_bounds__(256) bc_stage_kernel(const T* __restrict__ B, const T* __restrict__ C,
                                                       O* __restrict__ bc, int64_t L, int64_t lpad,
                                                       int* __restrict__ flags, int nflags) {
    constexpr int TT = 64;
    if (flags && blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < nflags; i += blockDim.x) flags[i] = 0;
    __shared__ float tile[TT][2 * N + 1];
    const int64_t b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * TT;
    for (int i = threadIdx.x; i < 2 * N * TT; i += blockDim.x) {
        const int row = i / TT, t = i % TT;     // row: 0..N-1 = B_n, N..2N-1 = C_n
        const int64_t tt = t0 + t;
        const T* src = row < N ? B + (b * N + row) * L : C + (b * N + row - N) * L;
        tile[t][row] = tt < L ? to_f32(src[tt]) : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * N * TT; i += blockDim.x) {
        const int t = i / (2 * N), col = i % (2 * N);
        const int64_t tt = t0 + t;
        if (tt < lpad) bc[(b * lpad + tt) * (2 * N) + col] = from_f32<O>(tile[t][col]);
    }
}

// ------------------------------------------------------------- host side

// The driver's tensor-map encoder (one process-wide entry point), looked up
// once; the initialisation of a function-local static is thread-safe.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// (dim, seqlen, batch) activation tensor, box (CW channels, K steps, 1 row).
template <typename T>
bool make_map(CUtensorMap* m, const void* base, int64_t dim, int64_t L, int64_t batch, int cw, int k) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t gstride[2] = {(cuuint64_t)(dim * sizeof(T)), (cuuint64_t)(dim * L * sizeof(T))};
    const cuuint32_t box[3] = {(cuuint32_t)cw, (cuuint32_t)k, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        std::is_same<T, float>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return fn(m, dt, 3, const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Work split of the segmented scan for one call.
struct SegPlan {
    int units, M, S, cps, workers, grid;
};

template <int N, int K>
SegPlan seg_plan(int64_t batch, int64_t dim, int64_t seqlen, int sms, int ctas_per_sm) {
    constexpr int CW = 32 / (N / 4), WARPS = 4;   // workers (warp pairs) per CTA
    SegPlan pl{};
    pl.units = (int)((dim + CW - 1) / CW);
    pl.M = (int)(batch * pl.units);
    const int nch = (int)((seqlen + K - 1) / K);
    const int per_wave = sms * WARPS;
    if (pl.M < per_wave) {
        // fewer chains than schedulers: one task per chain
        pl.grid = (pl.M + WARPS - 1) / WARPS;
        pl.workers = pl.grid * WARPS;
        pl.S = 1;
        pl.cps = nch;
        return pl;
    }
    int k = pl.M / per_wave;                       // warps per scheduler, at most what fits
    if (k > ctas_per_sm) k = ctas_per_sm;
    if (k < 1) k = 1;
    pl.grid = sms * k;
    pl.workers = pl.grid * WARPS;
    // Segments per chain: the most even split of M * S tasks over the workers,
    // with segments of at least four chunks and at most 64 segments.
    int bestS = 1;
    double best = 1e30;
    const int smax = std::max(1, std::min(64, nch / 4));
    for (int S = 1; S <= smax; ++S) {
        const int cps = (nch + S - 1) / S;
        const int s_eff = (nch + cps - 1) / cps;
        const double tasks = double(pl.M) * s_eff / pl.workers;        // tasks per worker (mean)
        const double slots = std::ceil(tasks);                           // the busiest worker
        const double cost = slots * cps;                                 // chunks on the critical worker
        if (cost < best * 0.999) {
            best = cost;
            bestS = S;
        }
    }
    pl.cps = (nch + bestS - 1) / bestS;
    pl.S = (nch + pl.cps - 1) / pl.cps;
    return pl;
}

template <typename T, int N>
cudaError_t launch_seg_t(const ScanArgs& a, void* ws, int sms, cudaStream_t s) {
    using CF = SegCfg<T, N>;
    constexpr bool kFast = !std::is_same<T, float>::value;
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, SegParams);
    static const Kern kerns[4] = {scan_seg_kernel<T, N, kFast, false, false>,
                                  scan_seg_kernel<T, N, kFast, false, true>,
                                  scan_seg_kernel<T, N, kFast, true, false>,
                                  scan_seg_kernel<T, N, kFast, true, true>};
    const int which = (a.softplus ? 2 : 0) + (a.z ? 1 : 0);
    // shared-memory size set and resident CTAs per SM measured, once per device
    static DeviceMemo memo[4];
    int dev = 0, occ = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    cudaError_t err = cudaSuccess;
    if (!memo[which].get(dev, [&](int& r) {
            err = cudaFuncSetAttribute(kerns[which], cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
            if (err == cudaSuccess)
                err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, kerns[which], CF::THREADS, CF::SMEM);
            if (err == cudaSuccess && r < 1) err = cudaErrorInvalidConfiguration;
            return err == cudaSuccess;
        }, &occ))
        return err;
    const SegPlan pl = seg_plan<N, CF::K>(a.batch, a.dim, a.seqlen, sms, occ);
    const int64_t lpad = staged_lpad(a.seqlen);
    unsigned char* w = static_cast<unsigned char*>(ws);
    T* bc = reinterpret_cast<T*>(w);
    const int64_t bc_bytes = (a.batch * a.ngroups * lpad * 2 * N * (int64_t)sizeof(T) + 255) / 256 * 256;
    float* st = reinterpret_cast<float*>(w + bc_bytes);
    const int64_t st_bytes = ((int64_t)pl.M * CF::CW * N * 4 + 255) / 256 * 256;
    int* flags = reinterpret_cast<int*>(w + bc_bytes + st_bytes);
    {
        dim3 grid((unsigned)((lpad + 63) / 64), (unsigned)(a.batch * a.ngroups));
        bc_stage_kernel<T, N, T><<<grid, 256, 0, s>>>(static_cast<const T*>(a.B), static_cast<const T*>(a.C), bc,
                                                      a.seqlen, lpad, flags, pl.M);
    }
    CUtensorMap mu, md, mz, mo;
    if (!make_map<T>(&mu, a.u, a.dim, a.seqlen, a.batch, CF::CW, CF::K) ||
        !make_map<T>(&md, a.delta, a.dim, a.seqlen, a.batch, CF::CW, CF::K) ||
        !make_map<T>(&mz, a.z ? a.z : a.u, a.dim, a.seqlen, a.batch, CF::CW, CF::K) ||
        !make_map<T>(&mo, a.out, a.dim, a.seqlen, a.batch, CF::CW, CF::K))
        return cudaErrorInvalidValue;
    SegParams sp{a.A, a.D, a.delta_bias, bc, a.last_state, st, flags, (int)a.dim, (int)a.seqlen, lpad,
                 pl.units, pl.M, pl.S, pl.cps, pl.workers, a.h0, (int)a.ngroups, (int)a.gch};
    void* args[] = {&mu, &md, &mz, &mo, &sp};
    // Segments wait on segments of other warps: every CTA must be resident,
    // which the cooperative launch guarantees (the grid never exceeds the
    // occupancy the plan was sized with).
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kerns[which]), dim3(pl.grid),
                                       dim3(CF::THREADS), args, CF::SMEM, s);
}

}  // namespace

int64_t seg_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate, int elem_bytes,
                            int64_t ngroups) {
    const int cw = 32 / (dstate / 4);
    const int64_t units = (dim + cw - 1) / cw;
    const int64_t M = batch * units;
    const int64_t bc_bytes = (batch * ngroups * staged_lpad(seqlen) * 2 * dstate * elem_bytes + 255) / 256 * 256;
    const int64_t st_bytes = (M * cw * dstate * 4 + 255) / 256 * 256;
    return bc_bytes + st_bytes + (M * 4 + 255) / 256 * 256;
}

cudaError_t launch_scan_seg(const ScanArgs& a, DType dt, void* ws, int sms, cudaStream_t s) {
    if (dt == DType::F32) {
        switch (a.dstate) {
            case 4: return launch_seg_t<float, 4>(a, ws, sms, s);
            case 8: return launch_seg_t<float, 8>(a, ws, sms, s);
            case 16: return launch_seg_t<float, 16>(a, ws, sms, s);
        }
    } else {
        switch (a.dstate) {
            case 4: return launch_seg_t<__nv_bfloat16, 4>(a, ws, sms, s);
            case 8: return launch_seg_t<__nv_bfloat16, 8>(a, ws, sms, s);
            case 16: return launch_seg_t<__nv_bfloat16, 16>(a, ws, sms, s);
        }
    }
    return cudaErrorInvalidValue;
}

int64_t staged_lpad(int64_t seqlen) { return (seqlen + 63) / 64 * 64; }

bool tma_rows_supported(const ScanArgs& a, DType dt) {
    const int64_t es = dt == DType::BF16 ? 2 : 4;
    auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (!al16(a.u) || !al16(a.delta) || !al16(a.out) || (a.z && !al16(a.z)) || !al16(a.A) ||
        (a.last_state && !al16(a.last_state)) || (a.h0 && !al16(a.h0)))
        return false;
    if ((a.dim * es) % 16 != 0) return false;
    if (a.dim > (int64_t(1) << 31) - 64 || a.seqlen > (int64_t(1) << 31) - 64 || a.batch > 65535) return false;
    // B/C groups: the staging grid has one row per (batch row, group), and
    // every CTA or warp's block of 32 / (N / 4) channels lies in one group
    if (a.ngroups != 1 && (a.batch * a.ngroups > 65535 || a.gch % (32 / (a.dstate / 4)) != 0)) return false;
    if (a.dim * a.seqlen * es >= (int64_t(1) << 40)) return false;
    return encode_fn() != nullptr;
}

int set_wait_test_seg(int withhold, unsigned long long limit_ns) {
    if (cudaMemcpyToSymbol(g_withhold_flag, &withhold, sizeof(withhold)) != cudaSuccess) return -1;
    if (cudaMemcpyToSymbol(g_wait_limit_ns, &limit_ns, sizeof(limit_ns)) != cudaSuccess) return -1;
    return 0;
}

int read_device_error(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return -1;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return -1;
    }
    return (int)v;
}

}  // namespace ssm
