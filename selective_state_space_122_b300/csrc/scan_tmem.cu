// scan_tmem.cu -- the selective scan with B and C delivered through tensor
// memory (sm_100-family tcgen05), for bfloat16 activations.
//
// Computes, per (batch b, channel d), the recurrence of the Mamba selective
// SSM ("Mamba: Selective State Space Models" README, "State Space Model",
// "Selective Mechanism", "Efficient Scan"):
//     Delta_t = softplus(delta_raw_t + delta_bias)
//     h_t     = exp(Delta_t A) * h_{t-1} + Delta_t B_t u_t
//     out_t   = (C_t . h_t + D u_t) * silu(z_t)
//
// Why tensor memory
// -----------------
// A lane keeps 4 of a channel's N states (lane = channel * R + g, R = N / 4,
// states 4g .. 4g+3), so at every step it needs 4 values of B_t and 4 of
// C_t -- the same 8 values for all channels.  Read from shared memory, that
// is 32 bytes per lane per step through the load/store unit, which bounds the
// scan well before the SFU does.  Here a one-hot matrix product writes them
// into tensor memory instead, already in per-lane order: with
//     S[r, k] = 1 if k == g(r) else 0          (128 x 8, one row per lane)
//     X[k, 8t + j] = B_t[4k + j] (j < 4),  C_t[4k + j - 4] (j >= 4)
// the product D = S X (tcgen05.mma, kind::tf32, f32 accumulate) has in row r
// exactly the quads lane r needs, and the lane fetches a step's 8 values with
// a quarter of one tcgen05.ld.  The product is exact: B and C are bfloat16
// values (8-bit significands, exactly representable in tf32), multiplied by
// 1 or 0 and summed with zeros.
//
// Work decomposition
// ------------------
// A CTA owns CC = 4 * CW consecutive channels of one batch row (CW = 32 / R
// per consumer warp) and walks a segment of the sequence in chunks of K
// steps.  Every (batch, channel group) chain is cut into S segments; task
// i = s * M + m (segment s of chain m) goes to CTA i mod W in slot i div W,
// so a segment's predecessor always sits in an earlier slot (W <= M) and the
// state passes between segments through the workspace with a bounded
// release/acquire flag wait; the launch is cooperative, so every CTA a
// segment may wait on is resident.
//   producer warp: TMA loads of the u, delta_raw and z tiles (64- or 128-byte
//     rows, hardware-swizzled so the consumers' column reads are free of bank
//     conflicts) and of the chunk's staged X operand; then the one-hot MMA
//     into one of two TMEM buffers;
//   consumer warps (the four TMEM lane quarters): the per-(t, d) terms
//     (softplus, Delta u, silu(z)), the recurrence with B and C from TMEM, the
//     readout summed over the R lanes of each channel, D u and the gate, and a
//     TMA store of the output tile.
//
// Every wait is bounded (~1 s, %globaltimer); on giving up a warp sets a bit
// in the device error word, drains its own copies and the CTA still frees its
// tensor memory before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "scan_common.cuh"
#include "ssm_internal.cuh"

namespace ssm {

namespace {

// ------------------------------------------------------------- tcgen05 wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] = A[smem] * B[smem] (no accumulation), one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(0u)
        : "memory");
}

// Arrive on an mbarrier once every MMA this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive TMEM columns of this thread's lane -> 32 registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

// Wait for this thread's outstanding tcgen05.ld; the registers are tied to the
// wait so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait(uint32_t (&v)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                   "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                   "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor, no swizzle: start address, leading-dimension
// byte offset (between core matrices adjacent in K), stride-dimension byte
// offset (between core matrices adjacent in M or N), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::tf32: f32 accumulator, tf32 A and B, both
// K-major, N columns, M rows.
__host__ __device__ constexpr uint32_t idesc_tf32(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// ------------------------------------------------------------- configuration

template <int N_>
struct TmCfg {
    static constexpr int N = N_;
    static constexpr int G = 4;                 // states per lane
    static constexpr int R = N / G;             // lanes per channel
    static constexpr int CW = 32 / R;           // channels per consumer warp
    static constexpr int WARPS = 4;             // consumer warps = TMEM lane quarters
    static constexpr int CC = WARPS * CW;       // channels per CTA
    static constexpr int K = 32;                // steps per chunk
    static constexpr int KR = K / R;            // steps per lane in the per-(t, d) phase
    static constexpr int NP = KR / 2;           // step pairs per lane
    static constexpr int P = 4;                 // ring slots
    static constexpr int THREADS = 32 * (WARPS + 1);
    static constexpr int ROWB = CC * 2;         // bytes of a bf16 tile row
    static_assert(ROWB == 64 || ROWB == 128, "tile rows are 64 or 128 bytes (swizzled)");
    static constexpr int TILE = K * ROWB;
    static constexpr int OPB = K * 8 * 16;      // X operand of a chunk: 8 columns of 4 tf32 per step
    static constexpr int TCOLS = 8 * K;         // TMEM columns of a chunk
    static constexpr int TMEM_COLS = 2 * TCOLS; // two buffers
    static_assert(TCOLS <= 256 && TMEM_COLS <= 512, "one MMA per chunk, two chunks of TMEM");
    static constexpr int al(int x, int a) { return (x + a - 1) / a * a; }
    static constexpr int SLOT_U = 0;
    static constexpr int SLOT_D = al(TILE, 1024);
    static constexpr int SLOT_Z = 2 * al(TILE, 1024);
    static constexpr int SLOT_X = 3 * al(TILE, 1024);
    static constexpr int SLOT = al(SLOT_X + OPB, 1024);
    static constexpr int A_OP = P * SLOT;                    // 128 x 8 tf32 selector, 4 KB
    static constexpr int W_BASE = A_OP + 4096;
    static constexpr int DPS = CW + 2;                       // float2 stride of a dp row (conflict-free stores)
    static constexpr int RS2 = 33;                           // float2 stride of a reduction row
    static constexpr int W_RED = al(K * DPS * 8, 128);
    static constexpr int W_OUT = W_RED + (R > 1 ? al((K / 2) * RS2 * 8, 128) : 0);
    static constexpr int OUTT = al(K * CW * 2, 128);
    static constexpr int W_BYTES = W_OUT + 3 * OUTT;
    static constexpr int BAR = W_BASE + WARPS * W_BYTES;     // full[P] empty[P] tfull[2] tempty[2] taddr
    static constexpr int USED = BAR + (2 * P + 4) * 8 + 16;
    // Over half of an SM's shared memory (plus 1 KB to align the base), so a
    // CTA never shares its SM: the 512 TMEM columns it allocates are free.
    static constexpr int SMEM = (USED + 1024 > 120 * 1024) ? USED + 1024 : 120 * 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

struct TmParams {
    const float* A;
    const float* D;
    const float* delta_bias;
    const float* xop;       // staged X operands, [batch][lpad / K][K][8][4] f32
    float* last_state;
    float* seg_state;       // [M * WARPS][CW][N] f32: state handed between segments
    int* seg_flag;          // [M * WARPS]: finished segments of each warp's channel group
    int dim, seqlen;
    int64_t lpad;
    int units;              // channel groups (CTA-wide) per batch row
    int M;                  // chains = batch * units
    int S;                  // segments per chain
    int cps;                // chunks per segment
    int workers;            // CTAs in the grid
};

__device__ __forceinline__ int tm_ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void tm_st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ bool tm_flag_wait(const int* flag, int want) {
    if (tm_ld_acquire(flag) >= want) return true;
    const unsigned long long t0 = globaltimer();
    while (tm_ld_acquire(flag) < want)
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    return true;
}

// Byte offset of element (row x, column c) of a bf16 tile whose rows are
// ROWB bytes, written by TMA with the matching swizzle (16-byte chunk index
// XOR address bits 7 and up).
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int x, int c) {
    const uint32_t o = (uint32_t)(x * ROWB + c * 2);
    return o ^ (((o >> 7) & (uint32_t)(ROWB / 16 - 1)) << 4);
}

template <int N, bool kSoftplus, bool kGate>
__global__ void __launch_bounds__(TmCfg<N>::THREADS, 1)
scan_tmem_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_d,
                 const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_out,
                 const TmParams p) {
    using CF = TmCfg<N>;
    using T = __nv_bfloat16;
    constexpr int K = CF::K, P = CF::P, R = CF::R, CW = CF::CW, CC = CF::CC, KR = CF::KR, NP = CF::NP;
    constexpr int DPS = CF::DPS, RS2 = CF::RS2;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base: the swizzle pattern follows absolute address bits
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring_s = smem_u32(smem);
    const uint32_t bar_full = smem_u32(smem + CF::BAR);
    const uint32_t bar_empty = bar_full + 8u * P;
    const uint32_t bar_tfull = bar_empty + 8u * P;
    const uint32_t bar_tempty = bar_tfull + 16u;
    uint32_t* taddr_slot = reinterpret_cast<uint32_t*>(smem + CF::BAR + (2 * P + 4) * 8);

    const int L = p.seqlen;
    const int nch = (L + K - 1) / K;
    const int T_total = p.M * p.S;

    // one-hot selector S[r][k] = (k == g(r)), K-major without swizzle: the
    // 8-row x 16-byte core matrix of rows 8 rg.. and k-half kh at rg*256 + kh*128
    {
        float* sa = reinterpret_cast<float*>(smem + CF::A_OP);
        for (int e = threadIdx.x; e < 128 * 8; e += CF::THREADS) {
            const int r = e >> 3, k = e & 7;
            sa[(r >> 3) * 64 + (k >> 2) * 32 + (r & 7) * 4 + (k & 3)] = (k == ((r & 31) % R)) ? 1.f : 0.f;
        }
    }
    fence_async_smem();
    if (threadIdx.x == 0) {
        for (int i = 0; i < P; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, CF::WARPS);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_tfull + 8u * i, 1);
            mbar_init(bar_tempty + 8u * i, CF::WARPS);
        }
        fence_mbar_init();
    }
    if (warp == CF::WARPS) {
        tmem_alloc(smem_u32(taddr_slot), CF::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;

    if (warp == CF::WARPS) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int total = 0;
            for (int task = blockIdx.x; task < T_total; task += p.workers) {
                const int sgm = task / p.M;
                total += min((sgm + 1) * p.cps, nch) - sgm * p.cps;
            }
            constexpr uint32_t tx_bytes = (uint32_t)((kGate ? 3 : 2) * CF::TILE + CF::OPB);
            int ld_task = blockIdx.x, ld_c = 0, ld_end = 0, ld_b = 0, ld_d0 = 0;
            const float* ld_x = nullptr;
            auto enter = [&](int task) {
                const int sgm = task / p.M, m = task - sgm * p.M;
                ld_b = m / p.units;
                ld_d0 = (m - ld_b * p.units) * CC;
                ld_c = sgm * p.cps;
                ld_end = min(ld_c + p.cps, nch);
                ld_x = p.xop + ((size_t)ld_b * p.lpad + (size_t)ld_c * K) * 32;
            };
            if (ld_task < T_total) enter(ld_task);
            int issued = 0;
            auto issue = [&]() {
                while (ld_task < T_total && ld_c >= ld_end) {
                    ld_task += p.workers;
                    if (ld_task < T_total) enter(ld_task);
                }
                if (ld_task >= T_total) return;
                const int slot = issued & (P - 1);
                const uint32_t base = ring_s + (uint32_t)(slot * CF::SLOT);
                const uint32_t bar = bar_full + 8u * (uint32_t)slot;
                const int t0 = ld_c * K;
                mbar_expect_tx(bar, tx_bytes);
                tma_load_3d(base + CF::SLOT_U, &tm_u, ld_d0, t0, ld_b, bar);
                tma_load_3d(base + CF::SLOT_D, &tm_d, ld_d0, t0, ld_b, bar);
                if constexpr (kGate) tma_load_3d(base + CF::SLOT_Z, &tm_z, ld_d0, t0, ld_b, bar);
                bulk_load(base + CF::SLOT_X, ld_x, CF::OPB, bar);
                ld_x += K * 32;
                ++ld_c;
                ++issued;
            };
            for (int i = 0; i < P && i < total; ++i) issue();

            const uint64_t adesc = smem_desc(smem_u32(smem + CF::A_OP), 128, 256);
            constexpr uint32_t idesc = idesc_tf32(128, CF::TCOLS);
            bool ok = true;
            int landed = 0, mmas = 0;
            for (int j = 0; j < total; ++j) {
                const int slot = j & (P - 1), tb = j & 1;
                if (!mbar_wait(bar_full + 8u * slot, (uint32_t)((j / P) & 1))) {
                    ok = false;
                    raise_error(1u);
                    break;
                }
                ++landed;
                if (j >= 2 && !mbar_wait(bar_tempty + 8u * tb, (uint32_t)(((j - 2) >> 1) & 1))) {
                    ok = false;
                    raise_error(2u);
                    break;
                }
                tc_fence_after();
                // X of this slot: 8-row core matrices of 16-byte rows, one per
                // step (SBO 128); the second k-half aliases the first (LBO 0),
                // which the selector multiplies by zero.
                const uint64_t bdesc = smem_desc(ring_s + (uint32_t)(slot * CF::SLOT + CF::SLOT_X), 0, 128);
                mma_tf32(tmem + (uint32_t)(tb * CF::TCOLS), adesc, bdesc, idesc);
                mma_commit(bar_tfull + 8u * tb);
                ++mmas;
                if (j + P < total) {
                    // the slot is free once every consumer has read its tiles
                    // and seen this chunk's MMA complete
                    if (!mbar_wait(bar_empty + 8u * slot, (uint32_t)((j / P) & 1))) {
                        ok = false;
                        raise_error(2u);
                        break;
                    }
                    issue();
                }
            }
            if (!ok) {
                // let issued copies land and the last MMA finish before the
                // shared and tensor memory are released
                for (int k = landed; k < issued; ++k)
                    if (!mbar_wait(bar_full + 8u * (uint32_t)(k & (P - 1)), (uint32_t)((k / P) & 1))) break;
                if (mmas > 0) mbar_wait(bar_tfull + 8u * (uint32_t)((mmas - 1) & 1), (uint32_t)(((mmas - 1) >> 1) & 1));
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int w = warp;
        const int ch = lane / R, g = lane % R;
        float2* dp = reinterpret_cast<float2*>(smem + CF::W_BASE + w * CF::W_BYTES);
        float2* red = reinterpret_cast<float2*>(smem + CF::W_BASE + w * CF::W_BYTES + CF::W_RED);
        unsigned char* outb = smem + CF::W_BASE + w * CF::W_BYTES + CF::W_OUT;
        const uint32_t tlane = tmem + ((uint32_t)(32 * w) << 16);

        int tas[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) tas[q] = g * KR + 2 * ((q + g * (CW / 8)) % NP);

        bool ok = true;
        int j = 0, oslot = 0;
        for (int task = blockIdx.x; task < T_total && ok; task += p.workers) {
            const int sgm = task / p.M, m = task - sgm * p.M;
            const int b = m / p.units;
            const int dcta = (m - b * p.units) * CC;
            const int dw = dcta + w * CW;
            const int d = dw + ch;
            const bool ch_ok = d < p.dim;
            const int cb = sgm * p.cps, ce = min(cb + p.cps, nch);
            const int chain = m * CF::WARPS + w;

            float2 A2[2];
            {
                const float4 a = ch_ok ? *reinterpret_cast<const float4*>(p.A + (size_t)d * N + 4 * g)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                A2[0] = make_float2(a.x * kLog2e, a.y * kLog2e);
                A2[1] = make_float2(a.z * kLog2e, a.w * kLog2e);
            }
            const float2 dskip2 = splat2((p.D && ch_ok) ? p.D[d] : 0.f);
            const float2 bias2 = splat2((p.delta_bias && ch_ok) ? p.delta_bias[d] : 0.f);

            float2 h0 = make_float2(0.f, 0.f), h1 = make_float2(0.f, 0.f);
            float* hst = p.seg_state + ((size_t)chain * CW + ch) * N + 4 * g;
            if (sgm > 0) {
                if (!__all_sync(0xffffffffu, tm_flag_wait(p.seg_flag + chain, sgm))) {
                    ok = false;
                    if (lane == 0) raise_error(4u);
                    break;
                }
                const float4 v = __ldcg(reinterpret_cast<const float4*>(hst));
                h0 = make_float2(v.x, v.y);
                h1 = make_float2(v.z, v.w);
            }

            for (int c = cb; c < ce; ++c, ++j) {
                const int slot = j & (P - 1), tb = j & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8u * slot, (uint32_t)((j / P) & 1)))) {
                    ok = false;
                    if (lane == 0) raise_error(1u);
                    break;
                }
                const int t0 = c * K;
                const unsigned char* sb = smem + slot * CF::SLOT;

                // ---- per-(t, d) terms for this lane's step pairs
                float2 uk[NP], gate[NP];
                {
                    float2 dpv[2 * NP];
#pragma unroll
                    for (int q = 0; q < NP; ++q) {
                        const int ta = tas[q];
                        const uint32_t oa = swz<CF::ROWB>(ta, w * CW + ch);
                        const uint32_t ob = swz<CF::ROWB>(ta + 1, w * CW + ch);
                        const float2 uv = make_float2(ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_U + oa)),
                                                      ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_U + ob)));
                        const float2 xr = make_float2(ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_D + oa)),
                                                      ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_D + ob)));
                        float2 dl = add2(xr, bias2);
                        if constexpr (kSoftplus) dl = relay_softplus2<true>(dl);
                        if (t0 + K > L)
                            dl = mul2(dl, make_float2(t0 + ta < L ? 1.f : 0.f, t0 + ta + 1 < L ? 1.f : 0.f));
                        const float2 du = mul2(dl, uv);
                        dpv[2 * q] = make_float2(dl.x, du.x);
                        dpv[2 * q + 1] = make_float2(dl.y, du.y);
                        uk[q] = uv;
                        if constexpr (kGate) {
                            const float2 zv = make_float2(ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_Z + oa)),
                                                          ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_Z + ob)));
                            gate[q] = seg_silu2<true>(zv);
                        } else {
                            gate[q] = splat2(1.f);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < NP; ++q) {
                        dp[tas[q] * DPS + ch] = dpv[2 * q];
                        dp[(tas[q] + 1) * DPS + ch] = dpv[2 * q + 1];
                    }
                }
                __syncwarp();

                // ---- this chunk's B and C are in TMEM buffer tb once its MMA completed
                if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8u * tb, (uint32_t)((j >> 1) & 1)))) {
                    ok = false;
                    if (lane == 0) raise_error(2u);
                    break;
                }
                tc_fence_after();
                if (lane == 0) mbar_arrive(bar_empty + 8u * slot);

                // ---- the recurrence, software-pipelined over the chunk's K steps:
                // step t loads Delta and Delta u of step t+LA, evaluates exp(Delta A)
                // and Delta B u of step t+EA, advances the state by step t and reads
                // out C_t . h_t.  B and C come from TMEM in groups of 4 steps (32
                // columns), each group requested one group ahead of its use.
                constexpr int LA = 4, EA = 2, NG = K / 4;
                const uint32_t tcol = tlane + (uint32_t)(tb * CF::TCOLS);
                uint32_t gv[NG][32];
                tmem_ld32(tcol, gv[0]);
                tmem_wait(gv[0]);
                if (NG > 1) tmem_ld32(tcol + 32, gv[1]);
                float2 qv[K];
                float2 dA[K][2], dB[K][2];
                float2 s2v[K / 2];
                auto bq = [&](int t, int i) { return __uint_as_float(gv[t >> 2][(t & 3) * 8 + i]); };
                auto load_step = [&](int t) { qv[t] = dp[t * DPS + ch]; };
                auto exp_step = [&](int t) {
                    const float2 dl2 = splat2(qv[t].x), du2 = splat2(qv[t].y);
                    const float2 e0 = mul2(dl2, A2[0]);
                    const float2 e1 = mul2(dl2, A2[1]);
                    dA[t][0] = make_float2(decay_exp2<true>(e0.x), decay_exp2<true>(e0.y));
                    dA[t][1] = make_float2(decay_exp2<true>(e1.x), decay_exp2<true>(e1.y));
                    dB[t][0] = mul2(du2, make_float2(bq(t, 0), bq(t, 1)));
                    dB[t][1] = mul2(du2, make_float2(bq(t, 2), bq(t, 3)));
                };
#pragma unroll
                for (int t = 0; t < LA; ++t) load_step(t);
#pragma unroll
                for (int t = 0; t < EA; ++t) exp_step(t);
                float2 acc_prev = make_float2(0.f, 0.f);
#pragma unroll
                for (int t = 0; t < K; ++t) {
                    if (t + EA < K && ((t + EA) & 3) == 0) {
                        const int gr = (t + EA) >> 2;
                        tmem_wait(gv[gr]);
                        if (gr + 1 < NG) tmem_ld32(tcol + 32u * (uint32_t)(gr + 1), gv[gr + 1]);
                    }
                    if (t + LA < K) load_step(t + LA);
                    if (t + EA < K) exp_step(t + EA);
                    h0 = fma2(dA[t][0], h0, dB[t][0]);
                    h1 = fma2(dA[t][1], h1, dB[t][1]);
                    const float2 acc = fma2(make_float2(bq(t, 6), bq(t, 7)), h1,
                                            mul2(make_float2(bq(t, 4), bq(t, 5)), h0));
                    if (t & 1) s2v[t / 2] = make_float2(acc_prev.x + acc_prev.y, acc.x + acc.y);
                    acc_prev = acc;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tempty + 8u * tb);

                // ---- sum the R lanes of each channel for this lane's pairs
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

                // ---- D u, gate, output tile (triple-buffered; before a tile is
                // rewritten, the store that read it three chunks ago has finished)
                T* so = reinterpret_cast<T*>(outb + oslot * CF::OUTT);
                if (lane == 0) bulk_wait_read<2>();
                __syncwarp();
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    const float2 y = mul2(fma2(dskip2, uk[q], yv[q]), gate[q]);
                    st_pair<T>(so + tas[q] * CW + ch, so + (tas[q] + 1) * CW + ch, y);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0 && dw < p.dim) {   // a group wholly past dim has nothing to store
                    tma_store_3d(&tm_out, dw, t0, b, smem_u32(so));
                    bulk_commit();
                }
                oslot = oslot == 2 ? 0 : oslot + 1;
            }
            if (!ok) break;

            // state leaving the segment
            if (sgm + 1 < p.S) {
                __stcg(reinterpret_cast<float4*>(hst), make_float4(h0.x, h0.y, h1.x, h1.y));
                __threadfence();
                __syncwarp();
                if (lane == 0) tm_st_release(p.seg_flag + chain, sgm + 1);
            } else if (p.last_state && ch_ok) {
                *reinterpret_cast<float4*>(p.last_state + ((size_t)b * p.dim + d) * N + 4 * g) =
                    make_float4(h0.x, h0.y, h1.x, h1.y);
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    // every warp ends here: the tensor memory is released exactly once
    tc_fence_before();
    __syncthreads();
    if (warp == CF::WARPS) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, CF::TMEM_COLS);
    }
}

// X operands of every chunk: [batch][t][j][k] f32 with X[k, 8t + j] =
// B_t[4k + j] (j < 4), C_t[4k + j - 4] (j >= 4), zero for k >= N / 4 and for
// t >= L; also zeroes the segment flags.
template <int N>
__global__ void __launch_bounds__(256) tm_stage_kernel(const __nv_bfloat16* __restrict__ B,
                                                       const __nv_bfloat16* __restrict__ C, float* __restrict__ xop,
                                                       int L, int64_t lpad, int* flags, int nflags) {
    __shared__ float sb[2][N][65];
    const int b = blockIdx.y;
    const int t0 = blockIdx.x * 64;
    if (flags) {
        const size_t nthr = (size_t)gridDim.x * gridDim.y * blockDim.x;
        for (size_t i = ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x; i < (size_t)nflags;
             i += nthr)
            flags[i] = 0;
    }
    for (int e = threadIdx.x; e < 2 * N * 64; e += 256) {
        const int which = e / (N * 64), n = (e / 64) % N, t = e % 64;
        const __nv_bfloat16* src = which ? C : B;
        sb[which][n][t] = (t0 + t < L) ? __bfloat162float(src[((size_t)b * N + n) * L + t0 + t]) : 0.f;
    }
    __syncthreads();
    float* dst = xop + ((size_t)b * lpad + t0) * 32;
    for (int e = threadIdx.x; e < 64 * 32; e += 256) {
        const int t = e / 32, jj = (e / 4) % 8, k = e % 4;
        const int n = 4 * k + (jj & 3);
        dst[e] = (n < N) ? sb[jj >> 2][n][t] : 0.f;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tm_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// (dim, seqlen, batch) bf16 tensor, box (cw channels, k steps, 1 row).
bool tm_make_map(CUtensorMap* m, const void* base, int64_t dim, int64_t L, int64_t batch, int cw, int k,
                 CUtensorMapSwizzle sw) {
    auto fn = tm_encode_fn();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t gstride[2] = {(cuuint64_t)(dim * 2), (cuuint64_t)(dim * L * 2)};
    const cuuint32_t box[3] = {(cuuint32_t)cw, (cuuint32_t)k, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TmPlan {
    int units, M, S, cps, grid;
};

template <int N>
TmPlan tm_plan(int64_t batch, int64_t dim, int64_t seqlen, int sms) {
    using CF = TmCfg<N>;
    TmPlan pl{};
    pl.units = (int)((dim + CF::CC - 1) / CF::CC);
    pl.M = (int)(batch * pl.units);
    const int nch = (int)((seqlen + CF::K - 1) / CF::K);
    if (pl.M <= sms) {
        pl.grid = pl.M;
        pl.S = 1;
        pl.cps = nch;
        return pl;
    }
    pl.grid = sms;
    // segments per chain: the most even split of M * S tasks over the CTAs,
    // with segments of at least four chunks and at most 64 segments
    int bestS = 1;
    double best = 1e30;
    const int smax = std::max(1, std::min(64, nch / 4));
    for (int S = 1; S <= smax; ++S) {
        const int cps = (nch + S - 1) / S;
        const int s_eff = (nch + cps - 1) / cps;
        const double cost = std::ceil(double(pl.M) * s_eff / pl.grid) * cps;
        if (cost < best * 0.999) {
            best = cost;
            bestS = S;
        }
    }
    pl.cps = (nch + bestS - 1) / bestS;
    pl.S = (nch + pl.cps - 1) / pl.cps;
    return pl;
}

template <int N>
int64_t tm_ws_bytes(int64_t batch, int64_t dim, int64_t seqlen) {
    using CF = TmCfg<N>;
    const int64_t units = (dim + CF::CC - 1) / CF::CC;
    const int64_t chains = batch * units * CF::WARPS;
    const int64_t x_bytes = (batch * relay_lpad(seqlen) * 32 * 4 + 255) / 256 * 256;
    const int64_t st_bytes = (chains * CF::CW * N * 4 + 255) / 256 * 256;
    return x_bytes + st_bytes + (chains * 4 + 255) / 256 * 256;
}

template <int N>
cudaError_t launch_tmem_t(const ScanArgs& a, void* ws, int sms, cudaStream_t s) {
    using CF = TmCfg<N>;
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TmParams);
    static const Kern kerns[4] = {scan_tmem_kernel<N, false, false>, scan_tmem_kernel<N, false, true>,
                                  scan_tmem_kernel<N, true, false>, scan_tmem_kernel<N, true, true>};
    const int which = (a.softplus ? 2 : 0) + (a.z ? 1 : 0);
    static int occ[4] = {0, 0, 0, 0};
    if (occ[which] == 0) {
        cudaError_t e = cudaFuncSetAttribute(kerns[which], cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
        if (e != cudaSuccess) return e;
        int o = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kerns[which], CF::THREADS, CF::SMEM);
        if (e != cudaSuccess) return e;
        if (o != 1) return cudaErrorInvalidConfiguration;   // one CTA per SM: TMEM is never contended
        occ[which] = o;
    }
    const TmPlan pl = tm_plan<N>(a.batch, a.dim, a.seqlen, sms);
    const int64_t lpad = relay_lpad(a.seqlen);
    unsigned char* w = static_cast<unsigned char*>(ws);
    float* xop = reinterpret_cast<float*>(w);
    const int64_t x_bytes = (a.batch * lpad * 32 * 4 + 255) / 256 * 256;
    const int64_t chains = (int64_t)pl.M * CF::WARPS;
    float* st = reinterpret_cast<float*>(w + x_bytes);
    const int64_t st_bytes = (chains * CF::CW * N * 4 + 255) / 256 * 256;
    int* flags = reinterpret_cast<int*>(w + x_bytes + st_bytes);
    {
        dim3 grid((unsigned)(lpad / 64), (unsigned)a.batch);
        tm_stage_kernel<N><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(a.B),
                                                static_cast<const __nv_bfloat16*>(a.C), xop, (int)a.seqlen, lpad,
                                                flags, (int)chains);
    }
    const CUtensorMapSwizzle sw = CF::ROWB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap mu, md, mz, mo;
    if (!tm_make_map(&mu, a.u, a.dim, a.seqlen, a.batch, CF::CC, CF::K, sw) ||
        !tm_make_map(&md, a.delta, a.dim, a.seqlen, a.batch, CF::CC, CF::K, sw) ||
        !tm_make_map(&mz, a.z ? a.z : a.u, a.dim, a.seqlen, a.batch, CF::CC, CF::K, sw) ||
        !tm_make_map(&mo, a.out, a.dim, a.seqlen, a.batch, CF::CW, CF::K, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TmParams tp{a.A, a.D, a.delta_bias, xop, a.last_state, st, flags, (int)a.dim, (int)a.seqlen, lpad,
                pl.units, pl.M, pl.S, pl.cps, pl.grid};
    void* args[] = {&mu, &md, &mz, &mo, &tp};
    // Segments wait on segments of other CTAs: every CTA must be resident,
    // which the cooperative launch guarantees (one CTA per SM, grid <= SMs).
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kerns[which]), dim3(pl.grid),
                                       dim3(CF::THREADS), args, CF::SMEM, s);
}

}  // namespace

bool tmem_supported(const ScanArgs& a, DType dt) {
    if (dt != DType::BF16 || a.dstate != 16) return false;
    if (!relay_supported(a, dt)) return false;
    // the total task count (chains * 64 segments) stays a 32-bit int
    return a.batch * ((a.dim + 31) / 32) * 64 < (int64_t(1) << 31);
}

int64_t tmem_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate) {
    return dstate == 16 ? tm_ws_bytes<16>(batch, dim, seqlen) : 0;
}

cudaError_t launch_scan_tmem(const ScanArgs& a, DType dt, void* workspace, int sms, cudaStream_t s) {
    if (dt != DType::BF16 || a.dstate != 16) return cudaErrorInvalidValue;
    return launch_tmem_t<16>(a, workspace, sms, s);
}

int read_tmem_device_error(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return -1;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return -1;
    }
    return (int)v;
}

}  // namespace ssm
