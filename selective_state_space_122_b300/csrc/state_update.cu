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
// channel).  Two kernels: the bulk-copy pipeline below (state tiles moved by
// cp.async.bulk through a shared-memory ring; taken when the copies are
// legal and there are at least two (row, tile) pairs per SM), and the
// register kernel described here for every other call.  The state is read and written as 16-byte quads by L = N / 4
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
#include <algorithm>

#include "device_memo.h"
#include "scan_common.cuh"
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

// ------------------------------------------------------------ bulk-copy pipeline
// Measured on a B300 (256 x 5120 x 16, CUDA events, 2.05 us timer steps):
// 30.7 us with a clean L2 (5.8 TB/s for 178.6 MB, 89% of the measured HBM
// copy rate), 36.9 us when L2 first holds dirty lines, against 34.8 / 38.9 us
// for the register kernel.  Three or four stages time the same; six (fewer
// resident CTAs) 34.8 us; 256-channel tiles 43.0 us.
// The same step with the state moved by the copy engine: a persistent CTA
// owns one tile of kBulkCT channels and every rsplit-th batch row.  Its
// producer warp streams, per row, the tile's state (kBulkCT x N float32,
// contiguous), the row's x, dt, z slices and B, C rows into a ring of
// kBulkStages shared-memory stages with cp.async.bulk (one mbarrier per
// stage); four consumer warps update the state in place in shared memory
// (L = N / 4 lanes per channel, a 16-byte quad each, as above) and write
// the outputs; the producer then writes the tile back with one bulk store and
// reuses the stage once the store has read it.  The bytes in flight per SM
// are the ring's, not the registers': up to kBulkStages tiles per CTA.

constexpr int kBulkCT = 128;                      // channels per tile
constexpr int kBulkStages = 4;
constexpr int kBulkConsumers = 4;                 // consumer warps
constexpr int kBulkThreads = 32 * (kBulkConsumers + 1);
constexpr int kBulkMaxBC = 1024;                  // bytes of one B or C row (ngroups x N x element)

template <typename T, int N>
struct BulkCfg {
    static constexpr int ES = (int)sizeof(T);
    static constexpr int ST = kBulkCT * N * 4;    // state tile
    static constexpr int TOK = kBulkCT * ES;      // x, dt or z slice
    static constexpr int O_X = ST, O_DT = O_X + TOK, O_Z = O_DT + TOK, O_B = O_Z + TOK, O_C = O_B + kBulkMaxBC;
    static constexpr int STAGE = O_C + kBulkMaxBC;
    static constexpr int SMEM = kBulkStages * STAGE + 2 * kBulkStages * 8;
    static_assert(STAGE % 128 == 0 && (kBulkCT * N / 4) % (32 * kBulkConsumers) == 0, "stage layout");
};

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(reinterpret_cast<uint64_t>(dst)), "r"(src), "r"(bytes)
                 : "memory");
}

// Four consecutive elements (8 or 16 bytes, aligned) of B or C as floats.
__device__ __forceinline__ float4 ld_quad(const float* q) { return *reinterpret_cast<const float4*>(q); }
__device__ __forceinline__ float4 ld_quad(const __nv_bfloat16* q) {
    const uint2 v = *reinterpret_cast<const uint2*>(q);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xFFFF0000u));
}

template <typename T, int N, bool kFast>
__global__ void __launch_bounds__(kBulkThreads) state_update_bulk_kernel(UpdateArgs p, int rsplit, int ntile) {
    using CF = BulkCfg<T, N>;
    constexpr int L = N / 4;
    constexpr int QPT = kBulkCT * L / (32 * kBulkConsumers);   // state quads per consumer thread
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBulkStages * CF::STAGE);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kBulkStages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = (int)(blockIdx.x % (unsigned)ntile), rs = (int)(blockIdx.x / (unsigned)ntile);
    const int64_t d0 = (int64_t)tile * kBulkCT;
    const int nch = p.dim - d0 < kBulkCT ? (int)(p.dim - d0) : kBulkCT;
    const int64_t nrows = rs < p.batch ? (p.batch - 1 - rs) / rsplit + 1 : 0;
    const uint32_t bcb = (uint32_t)(p.ngroups * N * CF::ES);
    if (tid == 0) {
        for (int st = 0; st < kBulkStages; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, kBulkConsumers);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kBulkConsumers) {
        // ---- producer (one lane)
        if (lane != 0) return;
        const uint32_t base = smem_u32(sm);
        const uint32_t sbytes = (uint32_t)nch * N * 4, tbytes = (uint32_t)nch * CF::ES;
        const uint32_t tx = sbytes + (p.z ? 3 : 2) * tbytes + 2 * bcb;
        int64_t issued = 0;
        bool ok = true;
        // the wait test hook: block 0 never issues its first row's copies, so
        // its consumers wait that stage out and give up
        const bool hold = withhold_handoff((int)blockIdx.x, 0);
        for (int64_t m = 0; m < nrows && ok; ++m) {
            const int st = (int)(m % kBulkStages);
            const uint32_t sb = base + st * CF::STAGE;
            if (m >= kBulkStages) {
                // the row m - kBulkStages used this stage: written back by the
                // consumers -> store it, and wait until the store has read it
                const int64_t mp = m - kBulkStages;
                if (!mbar_wait(empty0 + 8 * st, (uint32_t)((mp / kBulkStages) & 1))) {
                    raise_error(1);
                    ok = false;
                    break;
                }
                const int64_t bp = rs + mp * rsplit;
                bulk_store(p.state + (bp * p.dim + d0) * N, sb, sbytes);
                bulk_commit();
                bulk_wait_read<0>();
            }
            if (m == 0 && hold) {
                issued = 1;
                continue;
            }
            const int64_t b = rs + m * rsplit, off = b * p.dim + d0;
            const uint32_t fb = full0 + 8 * st;
            mbar_expect_tx(fb, tx);
            bulk_load(sb, p.state + off * N, sbytes, fb);
            bulk_load(sb + CF::O_X, static_cast<const T*>(p.x) + off, tbytes, fb);
            bulk_load(sb + CF::O_DT, static_cast<const T*>(p.dt) + off, tbytes, fb);
            if (p.z) bulk_load(sb + CF::O_Z, static_cast<const T*>(p.z) + off, tbytes, fb);
            bulk_load(sb + CF::O_B, static_cast<const T*>(p.B) + b * p.ngroups * N, bcb, fb);
            bulk_load(sb + CF::O_C, static_cast<const T*>(p.C) + b * p.ngroups * N, bcb, fb);
            issued = m + 1;
        }
        // the last rows: store each once the consumers are done with it
        for (int64_t m = issued > kBulkStages ? issued - kBulkStages : 0; m < issued && ok; ++m) {
            const int st = (int)(m % kBulkStages);
            if (!mbar_wait(empty0 + 8 * st, (uint32_t)((m / kBulkStages) & 1))) {
                raise_error(1);
                ok = false;
                break;
            }
            bulk_store(p.state + ((rs + m * rsplit) * p.dim + d0) * N, base + st * CF::STAGE, sbytes);
            bulk_commit();
        }
        if (!ok) {
            // given up: let the loads already issued land before the CTA's
            // shared memory goes away (bounded)
            for (int64_t m = issued > kBulkStages ? issued - kBulkStages : 0; m < issued; ++m)
                mbar_wait(full0 + 8 * (int)(m % kBulkStages), (uint32_t)((m / kBulkStages) & 1));
        }
        bulk_wait_all();
        return;
    }

    // ---- consumers: thread quads q = tid + 128 j: channel q / L, quad q % L
    float4 a4[QPT];
    float Dd[QPT], bias[QPT];
    int grp[QPT];
#pragma unroll
    for (int j = 0; j < QPT; ++j) {
        const int q = tid + 32 * kBulkConsumers * j, c = q / L, g = q % L;
        const bool cok = c < nch;
        const int64_t d = d0 + c;
        a4[j] = cok ? __ldg(reinterpret_cast<const float4*>(p.A) + d * L + g) : make_float4(0.f, 0.f, 0.f, 0.f);
        a4[j] = make_float4(a4[j].x * kLog2e, a4[j].y * kLog2e, a4[j].z * kLog2e, a4[j].w * kLog2e);
        Dd[j] = (p.D && cok) ? __ldg(p.D + d) : 0.f;
        bias[j] = (p.dt_bias && cok) ? __ldg(p.dt_bias + d) : 0.f;
        grp[j] = cok ? (int)((uint32_t)d / (uint32_t)p.gch) : 0;
    }
    for (int64_t m = 0; m < nrows; ++m) {
        const int st = (int)(m % kBulkStages);
        // warp-uniform outcome (the row's outputs are summed by shuffles)
        const bool got = mbar_wait(full0 + 8 * st, (uint32_t)((m / kBulkStages) & 1));
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) raise_error(1);
            break;
        }
        unsigned char* stg = sm + st * CF::STAGE;
        float4* sst = reinterpret_cast<float4*>(stg);
        const T* tx = reinterpret_cast<const T*>(stg + CF::O_X);
        const T* tdt = reinterpret_cast<const T*>(stg + CF::O_DT);
        const T* tz = reinterpret_cast<const T*>(stg + CF::O_Z);
        const T* tb = reinterpret_cast<const T*>(stg + CF::O_B);
        const T* tc = reinterpret_cast<const T*>(stg + CF::O_C);
        const int64_t b = rs + m * rsplit;
#pragma unroll
        for (int j = 0; j < QPT; ++j) {
            const int q = tid + 32 * kBulkConsumers * j, c = q / L, g = q % L;
            const bool cok = c < nch;
            // the channel's terms (each of its L lanes computes them)
            const float xv = to_f32(tx[c]);
            float dl = to_f32(tdt[c]) + bias[j];
            if (p.softplus) dl = softplus_f<kFast>(dl);
            const float gate = p.z ? silu_f<kFast>(to_f32(tz[c])) : 1.f;
            const float4 bv = ld_quad(tb + grp[j] * N + 4 * g);
            const float4 cv = ld_quad(tc + grp[j] * N + 4 * g);
            const float4 h = sst[q];
            const float2 dl2 = splat2(dl), dx2 = splat2(dl * xv);
            const float2 e0 = mul2(dl2, make_float2(a4[j].x, a4[j].y)), e1 = mul2(dl2, make_float2(a4[j].z, a4[j].w));
            const float2 h0 = fma2(make_float2(decay_exp2<kFast>(e0.x), decay_exp2<kFast>(e0.y)),
                                   make_float2(h.x, h.y), mul2(dx2, make_float2(bv.x, bv.y)));
            const float2 h1 = fma2(make_float2(decay_exp2<kFast>(e1.x), decay_exp2<kFast>(e1.y)),
                                   make_float2(h.z, h.w), mul2(dx2, make_float2(bv.z, bv.w)));
            sst[q] = make_float4(h0.x, h0.y, h1.x, h1.y);
            const float2 c2 = fma2(make_float2(cv.z, cv.w), h1, mul2(make_float2(cv.x, cv.y), h0));
            float y = c2.x + c2.y;
#pragma unroll
            for (int o = 1; o < L; o <<= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
            if (g == 0 && cok)
                static_cast<T*>(p.out)[b * p.dim + d0 + c] = from_f32<T>((y + Dd[j] * xv) * gate);
        }
        // the updated tile goes back through the copy engine: order these
        // generic stores before its reads, then hand the stage over
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
    }
}

// Launch the bulk-copy step when its copies are legal and there are enough
// (tile, row) pairs to fill the GPU; false = not taken (use the other kernel).
template <typename T, int N>
bool launch_bulk(const UpdateArgs& a, int sms, cudaStream_t s, cudaError_t* err) {
    using CF = BulkCfg<T, N>;
    constexpr int es = (int)sizeof(T);
    const auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    const int64_t bcb = a.ngroups * N * es;
    if (!(al16(a.state) && al16(a.x) && al16(a.dt) && (!a.z || al16(a.z)) && al16(a.B) && al16(a.C) &&
          (a.dim * es) % 16 == 0 && bcb % 16 == 0 && bcb <= kBulkMaxBC))
        return false;
    const int64_t ntile = (a.dim + kBulkCT - 1) / kBulkCT;
    if (sms <= 0 || a.batch * ntile < 2 * (int64_t)sms) return false;
    // the ring's shared memory (set once per device), then the resident CTAs
    static DeviceMemo m_occ;
    int dev = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (!m_occ.get(dev, [&](int& r) {
            if (cudaFuncSetAttribute(state_update_bulk_kernel<T, N, es == 2>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM) != cudaSuccess)
                return false;
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, state_update_bulk_kernel<T, N, es == 2>,
                                                                 kBulkThreads, CF::SMEM) == cudaSuccess;
        }, &occ))
        return false;
    // every CTA owns one tile and every rsplit-th row: as many row splits as
    // the resident CTAs allow
    const int64_t rsplit = std::max<int64_t>(1, std::min<int64_t>(a.batch, (int64_t)sms * occ / ntile));
    const int64_t grid = ntile * rsplit;
    if (grid > 0x7fffffff) return false;
    state_update_bulk_kernel<T, N, es == 2><<<(unsigned)grid, kBulkThreads, CF::SMEM, s>>>(a, (int)rsplit, (int)ntile);
    *err = cudaGetLastError();
    return true;
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
cudaError_t launch_n(const UpdateArgs& a, int sms, cudaStream_t s) {
    cudaError_t err = cudaSuccess;
    if (launch_bulk<T, N>(a, sms, s, &err)) return err;
    // one vector load per quad of B / C needs both rows aligned to 4 elements
    const uintptr_t al = 4 * sizeof(T);
    const bool vec = (reinterpret_cast<uintptr_t>(a.B) % al) == 0 && (reinterpret_cast<uintptr_t>(a.C) % al) == 0;
    if (vec) return launch_v<T, N, true>(a, s);
    return launch_v<T, N, false>(a, s);
}

template <typename T>
cudaError_t launch_t(const UpdateArgs& a, int sms, cudaStream_t s) {
    if (a.batch > 65535LL * kRowsY) return cudaErrorInvalidValue;
    switch (a.dstate) {
        case 4: return launch_n<T, 4>(a, sms, s);
        case 8: return launch_n<T, 8>(a, sms, s);
        case 16: return launch_n<T, 16>(a, sms, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_state_update(const UpdateArgs& a, DType dt, int sms, cudaStream_t s) {
    if (dt == DType::F32) return launch_t<float>(a, sms, s);
    return launch_t<__nv_bfloat16>(a, sms, s);
}

int set_wait_test_update(int withhold, unsigned long long limit_ns) {
    if (cudaMemcpyToSymbol(g_withhold_flag, &withhold, sizeof(withhold)) != cudaSuccess) return -1;
    if (cudaMemcpyToSymbol(g_wait_limit_ns, &limit_ns, sizeof(limit_ns)) != cudaSuccess) return -1;
    return 0;
}

int read_update_device_error(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return -1;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return -1;
    }
    return (int)v;
}

}  // namespace ssm
