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
// A lane keeps G of a channel's 16 states (G = 2 in scan_tmem2_kernel, 4 in
// scan_ws_kernel; lane group g holds states G g .. G g + G - 1), so at every
// step it needs G values of B_t and G of C_t -- the same values for all
// channels.  Read from shared memory, that is 8 G bytes per lane per step
// through the load/store unit, which bounds the scan well before the SFU
// does.  Here a one-hot matrix product writes them into tensor memory
// instead, already in per-lane order: with a selector
//     S[r, k] = 1 if k == g(r) else 0          (128 x 8, one row per lane)
// and X[k, :] the B and C values of lane group k step after step, the
// product D = S X (tcgen05.mma, kind::tf32, f32 accumulate) has in row r
// exactly the values lane r needs, and the lane fetches several steps of them
// with one tcgen05.ld.  The product is exact: B and C are bfloat16 values
// (8-bit significands, exactly representable in tf32), multiplied by 1 or 0
// and summed with zeros.
//
// Work decomposition
// ------------------
// A CTA (one per SM) owns 32 consecutive channels of one batch row and walks
// a segment of the sequence in chunks.  Every (batch, channel group) chain is
// cut into S segments; task i = s * M + m (segment s of chain m) goes to CTA
// i mod W in slot i div W, so a segment's predecessor always sits in an
// earlier slot (W <= M) and the state passes between segments through the
// workspace with a bounded release/acquire flag wait; the launch is
// cooperative, so every CTA a segment may wait on is resident.  A loader
// warp issues the TMA loads of the u, delta_raw and z tiles (64-byte rows,
// hardware-swizzled: with the consumers' row order, column reads are free of
// bank conflicts) and of
// the chunk's staged X operand, an MMA warp the one-hot product into one of
// two TMEM buffers, a store warp the TMA stores of the output tiles; the
// compute warps of the two kernels are described with each.
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

#include "device_memo.h"
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

struct TmParams {
    const float* A;
    const float* D;
    const float* delta_bias;
    const float* xop;       // staged X operands, [batch * ngroups][lpad / K][K][8][4] f32
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
    const float* h0;        // initial state (batch, dim, N) or null
    int ngroups, gch;       // B/C groups, channels per group (a multiple of 32)
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
        if (globaltimer() - t0 > wait_limit_ns()) return false;
    return true;
}

// Byte offset of element (row x, column c) of a bf16 tile whose rows are
// ROWB bytes, laid out by TMA with the matching swizzle (16-byte chunk index
// XOR address bits 7 and up).
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int x, int c) {
    const uint32_t o = (uint32_t)(x * ROWB + c * 2);
    return o ^ (((o >> 7) & (uint32_t)(ROWB / 16 - 1)) << 4);
}

// The chunks a CTA walks: its tasks (segment s of chain m, task = s * M + m,
// every workers-th task from blockIdx.x), each a run of chunks.
struct ChunkCursor {
    int task, c, end, b, d0, xb;   // xb: the B/C block (X operands) of the channels
    __device__ void enter(const TmParams& p, int nch, int cc) {
        const int sgm = task / p.M, m = task - sgm * p.M;
        b = m / p.units;
        d0 = (m - b * p.units) * cc;
        xb = b * p.ngroups + d0 / p.gch;
        c = sgm * p.cps;
        end = min(c + p.cps, nch);
    }
    __device__ void start(const TmParams& p, int nch, int cc) {
        task = blockIdx.x;
        if (task < p.M * p.S) enter(p, nch, cc);
    }
    // move to the next chunk; false when the CTA has none left
    __device__ bool valid(const TmParams& p, int nch, int cc) {
        while (task < p.M * p.S && c >= end) {
            task += p.workers;
            if (task < p.M * p.S) enter(p, nch, cc);
        }
        return task < p.M * p.S;
    }
};

// ===================================================================
// Two states per lane: 8 consumer warps, two per TMEM lane quarter (both read
// the same rows: B and C do not depend on the channel), so every scheduler
// runs two independent recurrences.  A lane keeps states 2g, 2g+1 of its
// channel (lane = channel * 8 + g); a warp covers 4 channels, a CTA 32.
// ===================================================================

constexpr int tm_al(int x, int a) { return (x + a - 1) / a * a; }

struct Tm2Cfg {
    static constexpr int N = 16;
    static constexpr int G = 2;                 // states per lane
    static constexpr int R = N / G;             // lanes per channel (8)
    static constexpr int CW = 32 / R;           // channels per consumer warp (4)
    static constexpr int WARPS = 8;             // consumer warps, two per lane quarter
    static constexpr int CC = WARPS * CW;       // channels per CTA (32)
    static constexpr int K = 64;                // steps per chunk
    static constexpr int NI = (K / 2) * CW / 32;   // (step pair, channel) items per lane (4)
    static constexpr int SG = 8;                // steps per TMEM load group (32 columns)
    static constexpr int P = 4;                 // input ring slots
    static constexpr int OB = 4;                // output tiles (3: +0.5% on the long sequence)
    static constexpr int W_LOAD = WARPS, W_MMA = WARPS + 1, W_STORE = WARPS + 2;
    static constexpr int THREADS = 32 * (WARPS + 3);
    static constexpr int ROWB = CC * 2;         // 64-byte tile rows
    static constexpr int TILE = K * ROWB;
    static constexpr int OPB = K * 4 * 8 * 4;   // X: 4 columns x 8 tf32 per step
    static constexpr int TCOLS = 4 * K;         // TMEM columns of a chunk (256)
    static constexpr int TMEM_COLS = 2 * TCOLS;
    static_assert(TCOLS <= 256 && TMEM_COLS <= 512, "one MMA per chunk, two chunks of TMEM");
    static constexpr int SLOT_U = 0;
    static constexpr int SLOT_D = tm_al(TILE, 1024);
    static constexpr int SLOT_Z = 2 * tm_al(TILE, 1024);
    static constexpr int SLOT_X = 3 * tm_al(TILE, 1024);
    static constexpr int SLOT = tm_al(SLOT_X + OPB, 1024);
    static constexpr int A_OP = P * SLOT;
    static constexpr int OUT = A_OP + 4096;
    static constexpr int OUTT = tm_al(TILE, 1024);
    static constexpr int W_BASE = OUT + OB * OUTT;
    static constexpr int DPS = K + 4;           // float2 stride of a channel's dp row (conflict-free 16-byte stores)
    static constexpr int RS2 = 49;              // float2 stride of a reduction row (= 1 mod 16)
    static constexpr int W_RED = tm_al(CW * DPS * 8, 128);
    static constexpr int W_BYTES = W_RED + tm_al((K / 2) * RS2 * 8, 128);
    static constexpr int BAR = W_BASE + WARPS * W_BYTES;
    static constexpr int NBAR = 2 * P + 4 + 2 * OB;
    static constexpr int USED = BAR + NBAR * 8 + 16;
    static constexpr int SMEM = (USED + 1024 > 120 * 1024) ? USED + 1024 : 120 * 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

template <bool kSoftplus, bool kGate>
__global__ void __launch_bounds__(Tm2Cfg::THREADS, 1)
scan_tmem2_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_d,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_out,
                  const TmParams p) {
    using CF = Tm2Cfg;
    using T = __nv_bfloat16;
    constexpr int N = CF::N, K = CF::K, P = CF::P, OB = CF::OB, R = CF::R, CW = CF::CW, CC = CF::CC,
                  NI = CF::NI, SG = CF::SG;
    constexpr int DPS = CF::DPS, RS2 = CF::RS2;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring_s = smem_u32(smem);
    const uint32_t bar_full = smem_u32(smem + CF::BAR);
    const uint32_t bar_empty = bar_full + 8u * P;
    const uint32_t bar_tfull = bar_empty + 8u * P;
    const uint32_t bar_tempty = bar_tfull + 16u;
    const uint32_t bar_ofull = bar_tempty + 16u;
    const uint32_t bar_oempty = bar_ofull + 8u * OB;
    uint32_t* taddr_slot = reinterpret_cast<uint32_t*>(smem + CF::BAR + CF::NBAR * 8);

    const int L = p.seqlen;
    const int nch = (L + K - 1) / K;

    // selector S[r][k] = (k == g(r)), g = lane % 8 (all 8 k used)
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
        for (int i = 0; i < OB; ++i) {
            mbar_init(bar_ofull + 8u * i, CF::WARPS);
            mbar_init(bar_oempty + 8u * i, 1);
        }
        fence_mbar_init();
    }
    if (warp == CF::W_LOAD) {
        tmem_alloc(smem_u32(taddr_slot), CF::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;

    int total = 0;
    for (int task = blockIdx.x; task < p.M * p.S; task += p.workers) {
        const int sgm = task / p.M;
        total += min((sgm + 1) * p.cps, nch) - sgm * p.cps;
    }

    if (warp == CF::W_LOAD) {
        if (lane == 0) {
            constexpr uint32_t tx_bytes = (uint32_t)((kGate ? 3 : 2) * CF::TILE + CF::OPB);
            ChunkCursor cur;
            cur.start(p, nch, CC);
            int issued = 0;
            auto issue = [&]() {
                if (!cur.valid(p, nch, CC)) return;
                const int slot = issued & (P - 1);
                const uint32_t base = ring_s + (uint32_t)(slot * CF::SLOT);
                const uint32_t bar = bar_full + 8u * (uint32_t)slot;
                const int t0 = cur.c * K;
                mbar_expect_tx(bar, tx_bytes);
                tma_load_3d(base + CF::SLOT_U, &tm_u, cur.d0, t0, cur.b, bar);
                tma_load_3d(base + CF::SLOT_D, &tm_d, cur.d0, t0, cur.b, bar);
                if constexpr (kGate) tma_load_3d(base + CF::SLOT_Z, &tm_z, cur.d0, t0, cur.b, bar);
                bulk_load(base + CF::SLOT_X, p.xop + ((size_t)cur.xb * p.lpad + (size_t)t0) * 32, CF::OPB, bar);
                ++cur.c;
                ++issued;
            };
            for (int i = 0; i < P && i < total; ++i) issue();
            for (int j = 0; j + P < total; ++j) {
                if (!mbar_wait(bar_empty + 8u * (uint32_t)(j & (P - 1)), (uint32_t)((j / P) & 1))) {
                    raise_error(2u);
                    break;
                }
                issue();
            }
            for (int k = max(0, issued - P); k < issued; ++k)
                if (!mbar_wait(bar_full + 8u * (uint32_t)(k & (P - 1)), (uint32_t)((k / P) & 1))) break;
        }
    } else if (warp == CF::W_MMA) {
        if (lane == 0) {
            const uint64_t adesc = smem_desc(smem_u32(smem + CF::A_OP), 128, 256);
            constexpr uint32_t idesc = idesc_tf32(128, CF::TCOLS);
            int mmas = 0;
            for (int j = 0; j < total; ++j) {
                const int slot = j & (P - 1), tb = j & 1;
                if (!mbar_wait(bar_full + 8u * slot, (uint32_t)((j / P) & 1))) {
                    raise_error(1u);
                    break;
                }
                if (j >= 2 && !mbar_wait(bar_tempty + 8u * tb, (uint32_t)(((j - 2) >> 1) & 1))) {
                    raise_error(2u);
                    break;
                }
                tc_fence_after();
                // X of this slot: per step pair, the k-half 0 core matrix (8
                // rows of 16 bytes) then the k-half 1 one (LBO 128); step
                // pairs 256 bytes apart (SBO)
                const uint64_t bdesc = smem_desc(ring_s + (uint32_t)(slot * CF::SLOT + CF::SLOT_X), 128, 256);
                mma_tf32(tmem + (uint32_t)(tb * CF::TCOLS), adesc, bdesc, idesc);
                mma_commit(bar_tfull + 8u * tb);
                ++mmas;
            }
            for (int k = max(0, mmas - 2); k < mmas; ++k)
                if (!mbar_wait(bar_tfull + 8u * (uint32_t)(k & 1), (uint32_t)((k >> 1) & 1))) break;
        }
    } else if (warp == CF::W_STORE) {
        if (lane == 0) {
            ChunkCursor cur;
            cur.start(p, nch, CC);
            for (int j = 0; j < total && cur.valid(p, nch, CC); ++j, ++cur.c) {
                const int o = j % OB;
                if (!mbar_wait(bar_ofull + 8u * o, (uint32_t)((j / OB) & 1))) {
                    raise_error(2u);
                    break;
                }
                tma_store_3d(&tm_out, cur.d0, cur.c * K, cur.b, smem_u32(smem + CF::OUT + o * CF::OUTT));
                bulk_commit();
                bulk_wait_read<1>();
                if (j >= 1) mbar_arrive(bar_oempty + 8u * (uint32_t)((j - 1) % OB));
            }
            bulk_wait_all();
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int w = warp;
        const int ch = lane / R, g = lane % R;      // recurrence: channel, state pair
        const int ich = lane & (CW - 1);           // per-(t, d) items: channel
        float2* dp = reinterpret_cast<float2*>(smem + CF::W_BASE + w * CF::W_BYTES);
        float2* red = reinterpret_cast<float2*>(smem + CF::W_BASE + w * CF::W_BYTES + CF::W_RED);
        const uint32_t tlane = tmem + ((uint32_t)(32 * (w & 3)) << 16);
        // a lane's slot in a reduction row: lanes 16-31 four slots further on,
        // so that the channel sums read back (channels c and c + 2 of a half
        // warp) fall in different banks
        const int rpos = lane + ((lane >> 4) << 2);
        // per-(t, d) items: lanes 16-31 take their odd step first, so that the
        // eight rows of every tile access differ mod 8 (distinct banks)
        const bool sw = lane >= 16;
        int ipv[NI];   // step pair of each item
#pragma unroll
        for (int i = 0; i < NI; ++i) ipv[i] = (lane + 32 * i) / CW;

        bool ok = true;
        int j = 0;
        for (int task = blockIdx.x; task < p.M * p.S && ok; task += p.workers) {
            const int sgm = task / p.M, m = task - sgm * p.M;
            const int b = m / p.units;
            const int dcta = (m - b * p.units) * CC;
            const int d = dcta + w * CW + ch;
            const int di = dcta + w * CW + ich;
            const bool ch_ok = d < p.dim, it_ok = di < p.dim;
            const int cb = sgm * p.cps, ce = min(cb + p.cps, nch);
            const int chain = m * CF::WARPS + w;

            float2 A2 = make_float2(0.f, 0.f);
            if (ch_ok) {
                const float2 a = *reinterpret_cast<const float2*>(p.A + (size_t)d * N + 2 * g);
                A2 = make_float2(a.x * kLog2e, a.y * kLog2e);
            }
            const float2 dskip2 = splat2((p.D && it_ok) ? p.D[di] : 0.f);
            const float2 bias2 = splat2((p.delta_bias && it_ok) ? p.delta_bias[di] : 0.f);

            float2 h = make_float2(0.f, 0.f);
            float* hst = p.seg_state + ((size_t)chain * CW + ch) * N + 2 * g;
            if (sgm > 0) {
                if (!__all_sync(0xffffffffu, tm_flag_wait(p.seg_flag + chain, sgm))) {
                    ok = false;
                    if (lane == 0) raise_error(4u);
                    break;
                }
                h = __ldcg(reinterpret_cast<const float2*>(hst));
            } else if (p.h0 && ch_ok) {
                h = *reinterpret_cast<const float2*>(p.h0 + ((size_t)b * p.dim + d) * N + 2 * g);
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

                // ---- per-(t, d) terms of this lane's items (step pair, channel)
                float2 uk[NI], gate[NI];
                {
                    float2 dpv[2 * NI];
#pragma unroll
                    for (int i = 0; i < NI; ++i) {
                        const int ta = 2 * ipv[i];
                        const int tf = ta + (sw ? 1 : 0), ts = ta + (sw ? 0 : 1);
                        const uint32_t oa = swz<CF::ROWB>(tf, w * CW + ich);
                        const uint32_t ob = swz<CF::ROWB>(ts, w * CW + ich);
                        const float2 uv = make_float2(ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_U + oa)),
                                                      ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_U + ob)));
                        const float2 xr = make_float2(ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_D + oa)),
                                                      ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_D + ob)));
                        float2 dl = add2(xr, bias2);
                        if constexpr (kSoftplus) dl = softplus2_path<true>(dl);
                        if (t0 + K > L)
                            dl = mul2(dl, make_float2(t0 + tf < L ? 1.f : 0.f, t0 + ts < L ? 1.f : 0.f));
                        const float2 du = mul2(dl, uv);
                        dpv[2 * i] = sw ? make_float2(dl.y, du.y) : make_float2(dl.x, du.x);
                        dpv[2 * i + 1] = sw ? make_float2(dl.x, du.x) : make_float2(dl.y, du.y);
                        uk[i] = uv;
                        if constexpr (kGate) {
                            const float2 zv = make_float2(ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_Z + oa)),
                                                          ld_elem(reinterpret_cast<const T*>(sb + CF::SLOT_Z + ob)));
                            gate[i] = seg_silu2<true>(zv);
                        } else {
                            gate[i] = splat2(1.f);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < NI; ++i)
                        *reinterpret_cast<float4*>(dp + ich * DPS + 2 * ipv[i]) =
                            make_float4(dpv[2 * i].x, dpv[2 * i].y, dpv[2 * i + 1].x, dpv[2 * i + 1].y);
                }
                __syncwarp();

                if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8u * tb, (uint32_t)((j >> 1) & 1)))) {
                    ok = false;
                    if (lane == 0) raise_error(2u);
                    break;
                }
                tc_fence_after();
                if (lane == 0) mbar_arrive(bar_empty + 8u * slot);

                // the output tile j % OB is free once the store of chunk j - OB read it
                const int o = j % OB;
                if (j >= OB &&
                    !__all_sync(0xffffffffu, mbar_wait(bar_oempty + 8u * o, (uint32_t)(((j / OB) - 1) & 1)))) {
                    ok = false;
                    if (lane == 0) raise_error(2u);
                    break;
                }
                unsigned char* so = smem + CF::OUT + o * CF::OUTT;

                // ---- the recurrence over the chunk's K steps (software-pipelined
                // as in the four-state kernel); B and C of 8 steps per TMEM load.
                // Each step pair's partial sums go to the reduction buffer as they
                // are made; after every 16 steps the lane sums the 8 partials of
                // one of its items (the items of step pairs 8q .. 8q+7) and writes
                // that item's output, overlapping the following steps.
                constexpr int LA = 4, EA = 2, NG = K / SG;
                const uint32_t tcol = tlane + (uint32_t)(tb * CF::TCOLS);
                uint32_t gv[NG][32];
                tmem_ld32(tcol, gv[0]);
                tmem_wait(gv[0]);
                tmem_ld32(tcol + 32, gv[1]);
                float2 qv[K], dA[K], dB[K];
                auto bc = [&](int t, int i) { return __uint_as_float(gv[t / SG][(t % SG) * 4 + i]); };
                // Delta and Delta u of steps t, t+1 (t even) in one 16-byte load
                auto load_step = [&](int t) {
                    if ((t & 1) == 0) {
                        const float4 v = *reinterpret_cast<const float4*>(dp + ch * DPS + t);
                        qv[t] = make_float2(v.x, v.y);
                        qv[t + 1] = make_float2(v.z, v.w);
                    }
                };
                auto finish_item = [&](int q) {
                    const float2* row = red + ipv[q] * RS2 + ich * R + (ich >= 2 ? 4 : 0);
                    float2 pr[R];
#pragma unroll
                    for (int gg = 0; gg < R; ++gg) pr[gg] = row[gg];
                    const float2 a0 = add2(pr[0], pr[1]), a1 = add2(pr[2], pr[3]);
                    const float2 a2 = add2(pr[4], pr[5]), a3 = add2(pr[6], pr[7]);
                    const float2 ys = add2(add2(a0, a1), add2(a2, a3));
                    const float2 yv = sw ? make_float2(ys.y, ys.x) : ys;
                    const float2 y = mul2(fma2(dskip2, uk[q], yv), gate[q]);
                    const int ta = 2 * ipv[q];
                    st_pair<T>(reinterpret_cast<T*>(so + swz<CF::ROWB>(ta + (sw ? 1 : 0), w * CW + ich)),
                               reinterpret_cast<T*>(so + swz<CF::ROWB>(ta + (sw ? 0 : 1), w * CW + ich)), y);
                };
                auto exp_step = [&](int t) {
                    const float2 e = mul2(splat2(qv[t].x), A2);
                    dA[t] = make_float2(decay_exp2<true>(e.x), decay_exp2<true>(e.y));
                    dB[t] = mul2(splat2(qv[t].y), make_float2(bc(t, 0), bc(t, 1)));
                };
#pragma unroll
                for (int t = 0; t < LA + 2; ++t) load_step(t);
#pragma unroll
                for (int t = 0; t < EA; ++t) exp_step(t);
                float s_prev = 0.f;
#pragma unroll
                for (int t = 0; t < K; ++t) {
                    if (t + EA < K && ((t + EA) % SG) == 0) {
                        const int gr = (t + EA) / SG;
                        tmem_wait(gv[gr]);
                        if (gr + 1 < NG) tmem_ld32(tcol + 32u * (uint32_t)(gr + 1), gv[gr + 1]);
                    }
                    if (t + LA + 1 < K) load_step(t + LA + 1);
                    if (t + EA < K) exp_step(t + EA);
                    h = fma2(dA[t], h, dB[t]);
                    const float2 cy = mul2(make_float2(bc(t, 2), bc(t, 3)), h);
                    const float sy = cy.x + cy.y;
                    if (t & 1) red[(t / 2) * RS2 + rpos] = make_float2(s_prev, sy);
                    s_prev = sy;
                    if ((t % 16) == 15 && t / 16 < NI) {
                        __syncwarp();
                        finish_item(t / 16);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tempty + 8u * tb);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_ofull + 8u * o);
            }
            if (!ok) break;

            if (sgm + 1 < p.S) {
                __stcg(reinterpret_cast<float2*>(hst), h);
                __threadfence();
                __syncwarp();
                if (lane == 0 && !withhold_handoff(chain, sgm)) tm_st_release(p.seg_flag + chain, sgm + 1);
            } else if (p.last_state && ch_ok) {
                *reinterpret_cast<float2*>(p.last_state + ((size_t)b * p.dim + d) * N + 2 * g) = h;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == CF::W_LOAD) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, CF::TMEM_COLS);
    }
}

// X operands for two states per lane: per step pair a 256-byte block, the
// k-half-0 core matrix then the k-half-1 one, row 4 (t & 1) + j holding
// X[k, 4t + j] for k in the half: B_t[2k + j] (j < 2), C_t[2k + j - 2].
__global__ void __launch_bounds__(256) tm2_stage_kernel(const __nv_bfloat16* __restrict__ B,
                                                        const __nv_bfloat16* __restrict__ C, float* __restrict__ xop,
                                                        int L, int64_t lpad, int* flags, int nflags) {
    constexpr int N = 16;
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
        const int pair = e / 64, wi = e % 64;
        const int kh = wi / 32, row = (wi % 32) / 4, kk = wi % 4;
        const int t = 2 * pair + row / 4, jj = row % 4, k = 4 * kh + kk;
        dst[e] = sb[jj >> 1][2 * k + (jj & 1)][t];
    }
}

// ===================================================================
// Warp-specialised scan: four states per lane, the per-(t, d) work on
// separate warps.
//
// The recurrence warps (one per TMEM lane quarter) do only the per-element
// work: a lane keeps states 4g .. 4g+3 of one channel (lane = c + 8 g, eight
// channels per warp), reads Delta and Delta u of its channel with one 16-byte
// shared load per step (stored duplicated, {Delta, Delta, Delta u, Delta u},
// so the packed multiplies take them as they are), B and C from tensor memory
// (the one-hot product of the four-state layout), and sums C . h over its
// four states.  The four partial sums of a channel are combined over the
// channel's four lanes where the output is made: every lane stores its
// partial sum of each step into a shared buffer (one 4-byte store per step,
// 128 contiguous bytes per warp), which costs the recurrence far less than
// any exchange between its lanes.
//
// The aux warps (one per scheduler as well) do the per-(t, d) work on both
// sides of the recurrence: per chunk, lane (channel octet, step) reads eight
// channels of u, delta_raw and z with one 16-byte load each, computes Delta
// (softplus with a polynomial log1p, accurate for every Delta), Delta u,
// D u and silu(z), and writes the recurrence's input rows; one chunk later
// it reads the four partial sums of each of its items back (one 16-byte
// load), adds them and D u, applies the gate and writes eight bf16 outputs
// with one 16-byte store into the output tile.
//
// Work split, TMA ring, one-hot MMA, segments and bounded waits are those of
// the kernels above.
// ===================================================================

struct WsCfg {
    static constexpr int N = 16;
    static constexpr int G = 4;                 // states per lane
    static constexpr int CW = 8;                // channels per recurrence warp
    static constexpr int RW = 4;                // recurrence warps = TMEM lane quarters
    static constexpr int AW = 4;                // aux warps
    static constexpr int CC = RW * CW;          // channels per CTA (32)
    static constexpr int K = 32;                // steps per chunk
    static constexpr int P = 6;                 // input ring slots
    static constexpr int OB = 3;                // output tiles
    static constexpr int W_AUX = RW;
    static constexpr int W_LOAD = RW + AW, W_MMA = W_LOAD + 1, W_STORE = W_LOAD + 2;
    static constexpr int THREADS = 32 * (W_STORE + 1);
    static constexpr int ROWB = CC * 2;         // 64-byte tile rows
    static constexpr int TILE = K * ROWB;
    static constexpr int OPB = K * 8 * 16;      // X: 8 columns x 4 tf32 per step
    static constexpr int TCOLS = 8 * K;         // TMEM columns of a chunk (256)
    static constexpr int TMEM_COLS = 2 * TCOLS;
    static_assert(TCOLS <= 256 && TMEM_COLS <= 512, "one MMA per chunk, two chunks of TMEM");
    static constexpr int SLOT_U = 0;
    static constexpr int SLOT_D = tm_al(TILE, 1024);
    static constexpr int SLOT_Z = 2 * tm_al(TILE, 1024);
    static constexpr int SLOT_X = 3 * tm_al(TILE, 1024);
    static constexpr int SLOT = tm_al(SLOT_X + OPB, 1024);
    static constexpr int A_OP = P * SLOT;                 // 128 x 8 tf32 selector
    static constexpr int REC = A_OP + 4096;               // [2][K][CC] float4 {Delta, Delta, Delta u, Delta u}
    static constexpr int REC_BYTES = K * CC * 16;
    static constexpr int YB = REC + 2 * REC_BYTES;        // [2][K][CC][4] f32 partial readouts
    static constexpr int YB_BYTES = K * CC * 16;
    static constexpr int OUT = tm_al(YB + 2 * YB_BYTES, 1024);
    static constexpr int OUTT = tm_al(TILE, 1024);
    static constexpr int BAR = OUT + OB * OUTT;
    // full[P] empty[P] ready[2] done[2] ofull[OB] oempty[OB]
    static constexpr int NBAR = 2 * P + 4 + 2 * OB;
    static constexpr int USED = BAR + NBAR * 8 + 16;
    // over half of an SM's shared memory: one CTA per SM, so its 512 TMEM
    // columns are always free
    static constexpr int SMEM = (USED + 1024 > 120 * 1024) ? USED + 1024 : 120 * 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

// Byte offset of the 16-byte group o of row r of a 64-byte-row tile laid out
// by TMA with the 64-byte swizzle (group index XOR address bits 7-8).
__device__ __forceinline__ uint32_t swz64_group(int r, int o) {
    return (uint32_t)(r * 64 + ((o ^ ((r >> 1) & 3)) << 4));
}

// bf16 pair (one 32-bit word) -> two floats
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t f2_to_bf2(float2 v) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// 16-byte slot (t, channel) of a chunk's recurrence input rows and of its
// partial readouts, XOR-swizzled within each channel octet so that the aux
// warps' accesses (one channel octet, 8 steps per quarter-warp) and the
// recurrence warps' (8 channels of one step) are free of bank conflicts.
__device__ __forceinline__ int ws_rec_slot(int t, int col) { return t * 32 + (col ^ (t & 7)); }

template <bool kSoftplus, bool kGate>
__global__ void __launch_bounds__(WsCfg::THREADS, 1)
scan_ws_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_d,
               const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_out,
               const TmParams p) {
    using CF = WsCfg;
    constexpr int N = CF::N, K = CF::K, P = CF::P, OB = CF::OB, CC = CF::CC;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring_s = smem_u32(smem);
    const uint32_t bar_full = smem_u32(smem + CF::BAR);
    const uint32_t bar_empty = bar_full + 8u * P;
    // ready[b]: chunk j (b = j & 1) may be scanned -- its MMA has filled TMEM
    // buffer b and the aux warps have written its recurrence rows (after
    // finishing the output of chunk j - 2, so the partial-sum buffer is free);
    // done[b]: the recurrence warps have finished chunk j -- TMEM buffer,
    // recurrence rows and partial sums of b may be read or reused
    const uint32_t bar_ready = bar_empty + 8u * P;
    const uint32_t bar_done = bar_ready + 16u;
    const uint32_t bar_ofull = bar_done + 16u;
    const uint32_t bar_oempty = bar_ofull + 8u * OB;
    uint32_t* taddr_slot = reinterpret_cast<uint32_t*>(smem + CF::BAR + CF::NBAR * 8);

    const int L = p.seqlen;
    const int nch = (L + K - 1) / K;

    // selector S[r][k] = (k == g(r)), g = (lane of the quarter) / 8; k < 4 used
    {
        float* sa = reinterpret_cast<float*>(smem + CF::A_OP);
        for (int e = threadIdx.x; e < 128 * 8; e += CF::THREADS) {
            const int r = e >> 3, k = e & 7;
            sa[(r >> 3) * 64 + (k >> 2) * 32 + (r & 7) * 4 + (k & 3)] = (k == ((r & 31) >> 3)) ? 1.f : 0.f;
        }
    }
    fence_async_smem();
    if (threadIdx.x == 0) {
        for (int i = 0; i < P; ++i) {
            mbar_init(bar_full + 8u * i, 1);
            mbar_init(bar_empty + 8u * i, CF::AW + 1);   // the aux warps and the MMA's completion
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_ready + 8u * i, CF::AW + 1);   // the aux warps and the MMA's completion
            mbar_init(bar_done + 8u * i, CF::RW);
        }
        for (int i = 0; i < OB; ++i) {
            mbar_init(bar_ofull + 8u * i, CF::AW);
            mbar_init(bar_oempty + 8u * i, 1);
        }
        fence_mbar_init();
    }
    if (warp == CF::W_LOAD) {
        tmem_alloc(smem_u32(taddr_slot), CF::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;

    // chunks this CTA walks (the same sequence for every role)
    int total = 0;
    for (int task = blockIdx.x; task < p.M * p.S; task += p.workers) {
        const int sgm = task / p.M;
        total += min((sgm + 1) * p.cps, nch) - sgm * p.cps;
    }

    if (warp == CF::W_LOAD) {
        // ------------------------------------------------------------ TMA loads
        if (lane == 0) {
            constexpr uint32_t tx_bytes = (uint32_t)((kGate ? 3 : 2) * CF::TILE + CF::OPB);
            ChunkCursor cur;
            cur.start(p, nch, CC);
            int issued = 0;
            auto issue = [&]() {
                if (!cur.valid(p, nch, CC)) return;
                const int slot = issued % P;
                const uint32_t base = ring_s + (uint32_t)(slot * CF::SLOT);
                const uint32_t bar = bar_full + 8u * (uint32_t)slot;
                const int t0 = cur.c * K;
                mbar_expect_tx(bar, tx_bytes);
                tma_load_3d(base + CF::SLOT_U, &tm_u, cur.d0, t0, cur.b, bar);
                tma_load_3d(base + CF::SLOT_D, &tm_d, cur.d0, t0, cur.b, bar);
                if constexpr (kGate) tma_load_3d(base + CF::SLOT_Z, &tm_z, cur.d0, t0, cur.b, bar);
                bulk_load(base + CF::SLOT_X, p.xop + ((size_t)cur.xb * p.lpad + (size_t)t0) * 32, CF::OPB, bar);
                ++cur.c;
                ++issued;
            };
            for (int i = 0; i < P && i < total; ++i) issue();
            for (int j = 0; j + P < total; ++j) {
                // slot j % P is free once the aux warps have read chunk j's
                // tiles and its MMA (the reader of X) has completed
                if (!mbar_wait(bar_empty + 8u * (uint32_t)(j % P), (uint32_t)((j / P) & 1))) {
                    raise_error(2u);
                    break;
                }
                issue();
            }
            // the CTA's shared memory outlives every copy into it
            for (int k = max(0, issued - P); k < issued; ++k)
                if (!mbar_wait(bar_full + 8u * (uint32_t)(k % P), (uint32_t)((k / P) & 1))) break;
        }
    } else if (warp == CF::W_MMA) {
        // ------------------------------------------------------------ one-hot MMA
        if (lane == 0) {
            const uint64_t adesc = smem_desc(smem_u32(smem + CF::A_OP), 128, 256);
            constexpr uint32_t idesc = idesc_tf32(128, CF::TCOLS);
            int mmas = 0;
            for (int j = 0; j < total; ++j) {
                const int slot = j % P, tb = j & 1;
                if (!mbar_wait(bar_full + 8u * slot, (uint32_t)((j / P) & 1))) {
                    raise_error(1u);
                    break;
                }
                if (j >= 2 && !mbar_wait(bar_done + 8u * tb, (uint32_t)(((j - 2) >> 1) & 1))) {
                    raise_error(2u);
                    break;
                }
                tc_fence_after();
                // X: one 8-row x 16-byte core matrix per step (SBO 128); the
                // second k-half aliases the first (LBO 0) and meets zeros
                const uint64_t bdesc = smem_desc(ring_s + (uint32_t)(slot * CF::SLOT + CF::SLOT_X), 0, 128);
                mma_tf32(tmem + (uint32_t)(tb * CF::TCOLS), adesc, bdesc, idesc);
                mma_commit(bar_ready + 8u * tb);
                mma_commit(bar_empty + 8u * slot);
                ++mmas;
            }
            // tensor memory is released only after the last MMAs completed
            for (int k = max(0, mmas - 2); k < mmas; ++k)
                if (!mbar_wait(bar_ready + 8u * (uint32_t)(k & 1), (uint32_t)((k >> 1) & 1))) break;
        }
    } else if (warp == CF::W_STORE) {
        // ------------------------------------------------------------ output stores
        if (lane == 0) {
            ChunkCursor cur;
            cur.start(p, nch, CC);
            for (int j = 0; j < total && cur.valid(p, nch, CC); ++j, ++cur.c) {
                const int o = j % OB;
                if (!mbar_wait(bar_ofull + 8u * o, (uint32_t)((j / OB) & 1))) {
                    raise_error(2u);
                    break;
                }
                tma_store_3d(&tm_out, cur.d0, cur.c * K, cur.b, smem_u32(smem + CF::OUT + o * CF::OUTT));
                bulk_commit();
                // the store before this one has read its tile: hand it back
                bulk_wait_read<1>();
                if (j >= 1) mbar_arrive(bar_oempty + 8u * (uint32_t)((j - 1) % OB));
            }
            bulk_wait_all();
        }
    } else if (warp >= CF::W_AUX) {
        // ------------------------------------------------------------ aux: per-(t, d) work
        const int a = warp - CF::W_AUX;
        const int oct = lane >> 3, ts = lane & 7;
        const int trow = 8 * a + ts;               // step of the chunk this lane serves
        float4* rec = reinterpret_cast<float4*>(smem + CF::REC);
        const float4* pb = reinterpret_cast<const float4*>(smem + CF::YB);
        ChunkCursor cur;
        cur.start(p, nch, CC);
        int ptask = -1;
        float2 bias2[4], dsk2[4];
        bool ok = true;

        // Delta, Delta u into the recurrence rows of chunk j; keeps D u and
        // silu(z) of this lane's eight items for the chunk's output
        auto prologue = [&](int j, float2 (&du)[4], float2 (&sg)[4]) -> bool {
            if (!cur.valid(p, nch, CC)) return false;
            if (cur.task != ptask) {
                ptask = cur.task;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float v[2], dd[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int d = cur.d0 + 8 * oct + 2 * k + h;
                        v[h] = (p.delta_bias && d < p.dim) ? p.delta_bias[d] : 0.f;
                        dd[h] = (p.D && d < p.dim) ? p.D[d] : 0.f;
                    }
                    bias2[k] = make_float2(v[0], v[1]);
                    dsk2[k] = make_float2(dd[0], dd[1]);
                }
            }
            const bool valid = cur.c * K + trow < L;
            ++cur.c;
            const int slot = j % P;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8u * slot, (uint32_t)((j / P) & 1)))) {
                if (lane == 0) raise_error(1u);
                return false;
            }
            if (j >= 2 &&
                !__all_sync(0xffffffffu, mbar_wait(bar_done + 8u * (j & 1), (uint32_t)(((j - 2) >> 1) & 1)))) {
                if (lane == 0) raise_error(2u);
                return false;
            }
            const unsigned char* sb = smem + slot * CF::SLOT;
            const uint32_t off = swz64_group(trow, oct);
            const uint4 uw = *reinterpret_cast<const uint4*>(sb + CF::SLOT_U + off);
            const uint4 xw = *reinterpret_cast<const uint4*>(sb + CF::SLOT_D + off);
            uint4 zw = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (kGate) zw = *reinterpret_cast<const uint4*>(sb + CF::SLOT_Z + off);
            const uint32_t uv[4] = {uw.x, uw.y, uw.z, uw.w}, xv[4] = {xw.x, xw.y, xw.z, xw.w},
                           zv[4] = {zw.x, zw.y, zw.z, zw.w};
            float4* rrow = rec + (j & 1) * K * CC;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 u2 = bf2_to_f2(uv[k]);
                float2 dl = add2(bf2_to_f2(xv[k]), bias2[k]);
                if constexpr (kSoftplus) dl = softplus_poly2(dl);
                if (!valid) dl = splat2(0.f);
                const float2 dlu = mul2(dl, u2);
                rrow[ws_rec_slot(trow, 8 * oct + 2 * k)] = make_float4(dl.x, dl.x, dlu.x, dlu.x);
                rrow[ws_rec_slot(trow, 8 * oct + 2 * k + 1)] = make_float4(dl.y, dl.y, dlu.y, dlu.y);
                du[k] = mul2(dsk2[k], u2);
                if constexpr (kGate) sg[k] = seg_silu2<true>(bf2_to_f2(zv[k]));
                else sg[k] = splat2(1.f);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_ready + 8u * (j & 1));
                mbar_arrive(bar_empty + 8u * slot);
            }
            return true;
        };

        // (readout + D u) * silu(z) of chunk j into its output tile
        auto epilogue = [&](int j, const float2 (&du)[4], const float2 (&sg)[4]) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_done + 8u * (j & 1), (uint32_t)((j >> 1) & 1)))) {
                if (lane == 0) raise_error(2u);
                return false;
            }
            const int o = j % OB;
            if (j >= OB &&
                !__all_sync(0xffffffffu, mbar_wait(bar_oempty + 8u * o, (uint32_t)(((j / OB) - 1) & 1)))) {
                if (lane == 0) raise_error(2u);
                return false;
            }
            const float4* pr = pb + (j & 1) * K * CC;
            uint32_t ov[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // the four lanes' partial sums of channels 2k, 2k+1 of the octet
                const float4 a = pr[ws_rec_slot(trow, 8 * oct + 2 * k)];
                const float4 b = pr[ws_rec_slot(trow, 8 * oct + 2 * k + 1)];
                const float2 s = add2(add2(make_float2(a.x, b.x), make_float2(a.y, b.y)),
                                      add2(make_float2(a.z, b.z), make_float2(a.w, b.w)));
                ov[k] = f2_to_bf2(mul2(add2(s, du[k]), sg[k]));
            }
            *reinterpret_cast<uint4*>(smem + CF::OUT + o * CF::OUTT + swz64_group(trow, oct)) =
                make_uint4(ov[0], ov[1], ov[2], ov[3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ofull + 8u * o);
            return true;
        };

        float2 du_a[4], sg_a[4], du_b[4], sg_b[4];
        int j = 0;
        while (ok && j < total) {
            ok = prologue(j, du_a, sg_a);
            if (ok && j >= 1) ok = epilogue(j - 1, du_b, sg_b);
            ++j;
            if (!ok || j >= total) break;
            ok = prologue(j, du_b, sg_b);
            if (ok) ok = epilogue(j - 1, du_a, sg_a);
            ++j;
        }
        if (ok && total > 0) {
            if ((total - 1) & 1) epilogue(total - 1, du_b, sg_b);
            else epilogue(total - 1, du_a, sg_a);
        }
    } else {
        // ------------------------------------------------------------ recurrence
        const int w = warp;
        const int c = lane & 7, g = lane >> 3;       // channel of the warp, state group
        const int col = CF::CW * w + c;              // channel of the CTA
        const uint32_t tlane = tmem + ((uint32_t)(32 * w) << 16);
        const float4* rec = reinterpret_cast<const float4*>(smem + CF::REC);
        float* pb = reinterpret_cast<float*>(smem + CF::YB);

        bool ok = true;
        int j = 0;
        for (int task = blockIdx.x; task < p.M * p.S && ok; task += p.workers) {
            const int sgm = task / p.M, m = task - sgm * p.M;
            const int b = m / p.units;
            const int d = (m - b * p.units) * CC + col;
            const bool ch_ok = d < p.dim;
            const int cb = sgm * p.cps, ce = min(cb + p.cps, nch);
            const int chain = m * CF::RW + w;

            float2 A01 = make_float2(0.f, 0.f), A23 = make_float2(0.f, 0.f);
            if (ch_ok) {
                const float4 av = *reinterpret_cast<const float4*>(p.A + (size_t)d * N + 4 * g);
                A01 = make_float2(av.x * kLog2e, av.y * kLog2e);
                A23 = make_float2(av.z * kLog2e, av.w * kLog2e);
            }
            float2 h01 = make_float2(0.f, 0.f), h23 = make_float2(0.f, 0.f);
            float* hst = p.seg_state + ((size_t)chain * CF::CW + c) * N + 4 * g;
            if (sgm > 0) {
                if (!__all_sync(0xffffffffu, tm_flag_wait(p.seg_flag + chain, sgm))) {
                    ok = false;
                    if (lane == 0) raise_error(4u);
                    break;
                }
                const float4 v = __ldcg(reinterpret_cast<const float4*>(hst));
                h01 = make_float2(v.x, v.y);
                h23 = make_float2(v.z, v.w);
            } else if (p.h0 && ch_ok) {
                const float4 v = *reinterpret_cast<const float4*>(p.h0 + ((size_t)b * p.dim + d) * N + 4 * g);
                h01 = make_float2(v.x, v.y);
                h23 = make_float2(v.z, v.w);
            }

            for (int cc = cb; cc < ce; ++cc, ++j) {
                const int tb = j & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_ready + 8u * tb, (uint32_t)((j >> 1) & 1)))) {
                    ok = false;
                    if (lane == 0) raise_error(2u);
                    break;
                }
                tc_fence_after();
                const float4* rr = rec + tb * K * CC;
                float* pr = pb + tb * K * CC * 4;

                // Steps of the chunk, software-pipelined: step t loads the
                // inputs of step t + LA, evaluates exp(Delta A) and Delta B u of
                // step t + EA and advances the state by step t.  B and C come
                // from TMEM four steps (32 columns) per load, one load ahead.
                constexpr int LA = 6, EA = 3, NG = K / 4;
                const uint32_t tcol = tlane + (uint32_t)(tb * CF::TCOLS);
                uint32_t gv[NG][32];
                tmem_ld32(tcol, gv[0]);
                tmem_wait(gv[0]);
                tmem_ld32(tcol + 32, gv[1]);
                float4 qv[K];
                float2 dA[K][2], dB[K][2];
                auto bc = [&](int t, int i) { return __uint_as_float(gv[t >> 2][(t & 3) * 8 + i]); };
                auto load_step = [&](int t) { qv[t] = rr[ws_rec_slot(t, col)]; };
                auto exp_step = [&](int t) {
                    const float2 dl = make_float2(qv[t].x, qv[t].y), dlu = make_float2(qv[t].z, qv[t].w);
                    const float2 e0 = mul2(dl, A01), e1 = mul2(dl, A23);
                    dA[t][0] = make_float2(ex2_approx(e0.x), ex2_approx(e0.y));
                    dA[t][1] = make_float2(ex2_approx(e1.x), ex2_approx(e1.y));
                    dB[t][0] = mul2(dlu, make_float2(bc(t, 0), bc(t, 1)));
                    dB[t][1] = mul2(dlu, make_float2(bc(t, 2), bc(t, 3)));
                };
#pragma unroll
                for (int t = 0; t < LA; ++t) load_step(t);
#pragma unroll
                for (int t = 0; t < EA; ++t) exp_step(t);
#pragma unroll
                for (int t = 0; t < K; ++t) {
                    if (t + EA < K && ((t + EA) & 3) == 0) {
                        const int gr = (t + EA) >> 2;
                        tmem_wait(gv[gr]);
                        if (gr + 1 < NG) tmem_ld32(tcol + 32u * (uint32_t)(gr + 1), gv[gr + 1]);
                    }
                    if (t + LA < K) load_step(t + LA);
                    if (t + EA < K) exp_step(t + EA);
                    h01 = fma2(dA[t][0], h01, dB[t][0]);
                    h23 = fma2(dA[t][1], h23, dB[t][1]);
                    const float2 r = fma2(make_float2(bc(t, 6), bc(t, 7)), h23,
                                          mul2(make_float2(bc(t, 4), bc(t, 5)), h01));
                    // this lane's share of C_t . h_t, summed with the channel's
                    // other three lanes by the aux warps
                    pr[ws_rec_slot(t, col) * 4 + g] = r.x + r.y;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_done + 8u * tb);
            }
            if (!ok) break;

            // state leaving the segment
            const float4 hv = make_float4(h01.x, h01.y, h23.x, h23.y);
            if (sgm + 1 < p.S) {
                __stcg(reinterpret_cast<float4*>(hst), hv);
                __threadfence();
                __syncwarp();
                if (lane == 0 && !withhold_handoff(chain, sgm)) tm_st_release(p.seg_flag + chain, sgm + 1);
            } else if (p.last_state && ch_ok) {
                *reinterpret_cast<float4*>(p.last_state + ((size_t)b * p.dim + d) * N + 4 * g) = hv;
            }
        }
    }

    // every warp ends here: the tensor memory is released exactly once
    tc_fence_before();
    __syncthreads();
    if (warp == CF::W_LOAD) {
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

// The driver's tensor-map encoder (one process-wide entry point), looked up
// once; the initialisation of a function-local static is thread-safe.
PFN_cuTensorMapEncodeTiled_v12000 tm_encode_fn() {
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

// Work split of one call: M chains (batch rows x channel groups of cc),
// each cut into S segments of cps chunks of k steps; task i = s * M + m runs
// on CTA i % grid.  With more chains than SMs, S is the most even split of
// M * S tasks over the CTAs (segments of at least four chunks, at most 64).
TmPlan tm_plan(int64_t batch, int64_t dim, int64_t seqlen, int sms, int cc, int k) {
    TmPlan pl{};
    pl.units = (int)((dim + cc - 1) / cc);
    pl.M = (int)(batch * pl.units);
    const int nch = (int)((seqlen + k - 1) / k);
    if (pl.M <= sms) {
        pl.grid = pl.M;
        pl.S = 1;
        pl.cps = nch;
        return pl;
    }
    pl.grid = sms;
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


cudaError_t launch_tmem2(const ScanArgs& a, void* ws, int sms, cudaStream_t s) {
    using CF = Tm2Cfg;
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TmParams);
    static const Kern kerns[4] = {scan_tmem2_kernel<false, false>, scan_tmem2_kernel<false, true>,
                                  scan_tmem2_kernel<true, false>, scan_tmem2_kernel<true, true>};
    const int which = (a.softplus ? 2 : 0) + (a.z ? 1 : 0);
    // shared-memory size set and one CTA per SM confirmed, once per device
    static DeviceMemo memo[4];
    int dev = 0, occ = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    cudaError_t err = cudaSuccess;
    if (!memo[which].get(dev, [&](int& r) {
            err = cudaFuncSetAttribute(kerns[which], cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
            if (err == cudaSuccess)
                err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, kerns[which], CF::THREADS, CF::SMEM);
            if (err == cudaSuccess && r != 1) err = cudaErrorInvalidConfiguration;   // TMEM never contended
            return err == cudaSuccess;
        }, &occ))
        return err;
    // the work split depends only on the CTA's channel count and chunk length
    const TmPlan pl = tm_plan(a.batch, a.dim, a.seqlen, sms, CF::CC, CF::K);
    const int64_t lpad = staged_lpad(a.seqlen);
    unsigned char* w = static_cast<unsigned char*>(ws);
    float* xop = reinterpret_cast<float*>(w);
    const int64_t x_bytes = (a.batch * a.ngroups * lpad * 32 * 4 + 255) / 256 * 256;
    const int64_t chains = (int64_t)pl.M * CF::WARPS;
    float* st = reinterpret_cast<float*>(w + x_bytes);
    const int64_t st_bytes = (chains * CF::CW * CF::N * 4 + 255) / 256 * 256;
    int* flags = reinterpret_cast<int*>(w + x_bytes + st_bytes);
    {
        dim3 grid((unsigned)(lpad / 64), (unsigned)(a.batch * a.ngroups));
        tm2_stage_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(a.B),
                                              static_cast<const __nv_bfloat16*>(a.C), xop, (int)a.seqlen, lpad, flags,
                                              (int)chains);
    }
    CUtensorMap mu, md, mz, mo;
    if (!tm_make_map(&mu, a.u, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !tm_make_map(&md, a.delta, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !tm_make_map(&mz, a.z ? a.z : a.u, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !tm_make_map(&mo, a.out, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    TmParams tp{a.A, a.D, a.delta_bias, xop, a.last_state, st, flags, (int)a.dim, (int)a.seqlen, lpad,
                pl.units, pl.M, pl.S, pl.cps, pl.grid, a.h0, (int)a.ngroups, (int)a.gch};
    void* args[] = {&mu, &md, &mz, &mo, &tp};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kerns[which]), dim3(pl.grid),
                                       dim3(CF::THREADS), args, CF::SMEM, s);
}

cudaError_t launch_ws(const ScanArgs& a, void* ws, int sms, cudaStream_t s) {
    using CF = WsCfg;
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TmParams);
    static const Kern kerns[4] = {scan_ws_kernel<false, false>, scan_ws_kernel<false, true>,
                                  scan_ws_kernel<true, false>, scan_ws_kernel<true, true>};
    const int which = (a.softplus ? 2 : 0) + (a.z ? 1 : 0);
    // shared-memory size set and one CTA per SM confirmed, once per device
    static DeviceMemo memo[4];
    int dev = 0, occ = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    cudaError_t err = cudaSuccess;
    if (!memo[which].get(dev, [&](int& r) {
            err = cudaFuncSetAttribute(kerns[which], cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
            if (err == cudaSuccess)
                err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, kerns[which], CF::THREADS, CF::SMEM);
            if (err == cudaSuccess && r != 1) err = cudaErrorInvalidConfiguration;   // TMEM never contended
            return err == cudaSuccess;
        }, &occ))
        return err;
    const TmPlan pl = tm_plan(a.batch, a.dim, a.seqlen, sms, CF::CC, CF::K);
    const int64_t lpad = staged_lpad(a.seqlen);
    unsigned char* w = static_cast<unsigned char*>(ws);
    float* xop = reinterpret_cast<float*>(w);
    const int64_t x_bytes = (a.batch * a.ngroups * lpad * 32 * 4 + 255) / 256 * 256;
    const int64_t chains = (int64_t)pl.M * CF::RW;
    float* st = reinterpret_cast<float*>(w + x_bytes);
    const int64_t st_bytes = (chains * CF::CW * CF::N * 4 + 255) / 256 * 256;
    int* flags = reinterpret_cast<int*>(w + x_bytes + st_bytes);
    {
        dim3 grid((unsigned)(lpad / 64), (unsigned)(a.batch * a.ngroups));
        tm_stage_kernel<16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(a.B),
                                                 static_cast<const __nv_bfloat16*>(a.C), xop, (int)a.seqlen, lpad,
                                                 flags, (int)chains);
    }
    CUtensorMap mu, md, mz, mo;
    if (!tm_make_map(&mu, a.u, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !tm_make_map(&md, a.delta, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !tm_make_map(&mz, a.z ? a.z : a.u, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !tm_make_map(&mo, a.out, a.dim, a.seqlen, a.batch, CF::CC, CF::K, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    TmParams tp{a.A, a.D, a.delta_bias, xop, a.last_state, st, flags, (int)a.dim, (int)a.seqlen, lpad,
                pl.units, pl.M, pl.S, pl.cps, pl.grid, a.h0, (int)a.ngroups, (int)a.gch};
    void* args[] = {&mu, &md, &mz, &mo, &tp};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kerns[which]), dim3(pl.grid),
                                       dim3(CF::THREADS), args, CF::SMEM, s);
}

}  // namespace

bool tmem_supported(const ScanArgs& a, DType dt) {
    if (dt != DType::BF16 || a.dstate != 16) return false;
    if (!tma_rows_supported(a, dt)) return false;
    // B/C groups: every CTA's 32 channels lie in one group
    if (a.ngroups != 1 && a.gch % 32 != 0) return false;
    // the total task count (chains * 64 segments) stays a 32-bit int
    return a.batch * ((a.dim + 31) / 32) * 64 < (int64_t(1) << 31);
}

int64_t tmem_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate, int64_t ngroups) {
    if (dstate != 16) return 0;
    // both variants: staged operands (per B/C block), one f32 state per
    // (channel, state) of every 32-channel group, and one flag per consumer
    // warp of each group
    const int64_t groups = batch * ((dim + 31) / 32);
    const int64_t x_bytes = (batch * ngroups * staged_lpad(seqlen) * 32 * 4 + 255) / 256 * 256;
    const int64_t st_bytes = (groups * 32 * 16 * 4 + 255) / 256 * 256;
    return x_bytes + st_bytes + (groups * 8 * 4 + 255) / 256 * 256;
}

cudaError_t launch_scan_tmem(const ScanArgs& a, DType dt, void* workspace, int sms, cudaStream_t s, int variant) {
    if (dt != DType::BF16 || a.dstate != 16) return cudaErrorInvalidValue;
    if (variant == 3) return launch_ws(a, workspace, sms, s);
    return launch_tmem2(a, workspace, sms, s);
}

int set_wait_test_tmem(int withhold, unsigned long long limit_ns) {
    if (cudaMemcpyToSymbol(g_withhold_flag, &withhold, sizeof(withhold)) != cudaSuccess) return -1;
    if (cudaMemcpyToSymbol(g_wait_limit_ns, &limit_ns, sizeof(limit_ns)) != cudaSuccess) return -1;
    return 0;
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
