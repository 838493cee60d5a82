// sfu_peak.cu -- throughput probes for the arithmetic units the selective
// scan leans on: the special-function unit (ex2, lg2, rcp, tanh) and the float32
// pipe (packed f32x2 FMA).  Built into its own library (libssmpeak.so),
// separate from the scan library; the benchmark uses it to measure the
// denominators of the scan's arithmetic roofline on the GPU it runs on.
//
// Every probe runs `iters` iterations of U independent dependency chains per
// thread, with enough resident warps to hide latency, so the result is the
// unit's issue-limited throughput.  Each chain step is one instruction of the
// probed kind plus, for the SFU probes, one float32 add that keeps the value
// in a bounded range; the add goes to the float32 pipe and does not slow the
// SFU unless issue itself binds.
#include <cuda_runtime.h>

#include <cstdint>

#if defined(__GNUC__)
#define PK_API extern "C" __attribute__((visibility("default")))
#else
#define PK_API extern "C"
#endif

namespace {

constexpr int kU = 8;  // independent chains per thread
int g_threads = 256;   // block size of the next probe launch

__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2a(float x) {
    float y;
    asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcpa(float x) {
    float y;
    asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float tanha(float x) {
    float y;
    asm volatile("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// kind 0: ex2, 1: lg2, 2: rcp, 4: tanh.  x_{i+1} = f(x_i) - c keeps x in
// (-1, 0] for ex2 (2^x in (0.5, 1]), in [1, 2) for lg2 (log2 in [0, 1), + 1),
// in [1, 2] for rcp (1/x in [0.5, 1], + 1) and in (-0.75, 1.25) for tanh.
template <int kKind>
__global__ void __launch_bounds__(256) sfu_kernel(float* sink, int iters, float seed) {
    float v[kU];
#pragma unroll
    for (int i = 0; i < kU; ++i) v[i] = (kKind == 0 ? -0.25f : 1.25f) + seed * (threadIdx.x + i);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            if constexpr (kKind == 0) v[i] = ex2a(v[i]) - 1.0f;
            else if constexpr (kKind == 1) v[i] = lg2a(v[i]) + 1.0f;
            else if constexpr (kKind == 4) v[i] = tanha(v[i]) + 0.25f;
            else v[i] = rcpa(v[i]) + 1.0f;
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kU; ++i) s += v[i];
    if (s == 12345.678f) sink[threadIdx.x & 255] = s;  // never true; keeps the chains live
}

// Co-issue of the SFU and the float32 pipe: each step is one ex2 (kind 5) or
// one ex2 followed by K independent packed FMAs (kinds 6, 7: K = 1, 2), the
// mix of a recurrence step.  The result is counted in ex2 per second: on a
// GPU whose SFU and FMA pipes overlap perfectly, kinds 6 and 7 run at the
// ex2 rate as long as the packed FMAs (two FMA-pipe cycles each) fit in the
// SFU's cycles.
template <int K>
__global__ void __launch_bounds__(256) mix_kernel(float* sink, int iters, float seed) {
    float v[kU];
    unsigned long long p[kU][2];
    const float2 q = make_float2(0.9999f, seed);
    unsigned long long qq;
    asm("mov.b64 %0, {%1, %2};" : "=l"(qq) : "f"(q.x), "f"(q.y));
#pragma unroll
    for (int i = 0; i < kU; ++i) {
        v[i] = -0.25f + seed * (threadIdx.x + i);
        p[i][0] = p[i][1] = qq;
    }
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            v[i] = ex2a(v[i]) - 1.0f;
#pragma unroll
            for (int k = 0; k < K; ++k)
                asm volatile("fma.rn.f32x2 %0, %0, %1, %1;" : "+l"(p[i][k]) : "l"(qq));
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kU; ++i) {
        float2 a;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(p[i][0] ^ p[i][1]));
        s += v[i] + a.x;
    }
    if (s == 12345.678f) sink[threadIdx.x & 255] = s;
}

// Packed float32 FMA throughput: each step is one fma.rn.f32x2 (two FMAs).
__global__ void __launch_bounds__(256) ffma2_kernel(float* sink, int iters, float seed) {
    unsigned long long v[kU];
    const float a = 0.999f, b = 1e-3f;
    unsigned long long A, Bq;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a), "f"(a));
    asm("mov.b64 %0, {%1, %2};" : "=l"(Bq) : "f"(b), "f"(b));
#pragma unroll
    for (int i = 0; i < kU; ++i) {
        const float x = seed * (threadIdx.x + i);
        asm("mov.b64 %0, {%1, %2};" : "=l"(v[i]) : "f"(x), "f"(x));
    }
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kU; ++i) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(v[i]) : "l"(A), "l"(Bq));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kU; ++i) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v[i]));
        s += lo + hi;
    }
    if (s == 12345.678f) sink[threadIdx.x & 255] = s;
}


// The core of an in-warp time split of the scan, for measuring its cost: a
// lane owns all 16 states of one channel over a sub-chunk of T steps (lane =
// channel + 4 x sub-chunk, four channels and eight sub-chunks per warp, a
// chunk of 8T steps).  Per chunk: (1) each lane runs its T steps from a zero
// state, keeping the 16 T decays exp2(Delta A) in registers; (2) the
// sub-chunks' (decay product, local state) pairs are combined by an
// inclusive warp-shuffle scan (three levels), giving each lane the state
// entering its sub-chunk from the chunk's carry; (3) each lane re-sweeps its
// steps with the kept decays and sums C . h in-lane, one output per step.
// Per-step Delta, Delta u, B and C come from shared memory as in a staged
// kernel, laid out by lane (a warp's eight sub-chunks read eight consecutive
// 16-byte words, free of bank conflicts); no global memory is touched inside
// the loop, so the rate is the design's compute-and-shared-memory ceiling.
template <int T>
__global__ void __launch_bounds__(128) tsplit_kernel(float* sink, int iters) {
    constexpr int CH = 8 * T;   // steps per chunk
    // step t = sub * T + j of the chunk; [j][sub][channel] and [j][quad][sub]
    __shared__ float2 s_dd[T][8][4];
    __shared__ float4 s_b[T][4][8], s_c[T][4][8];
    __shared__ float s_y[4][T][32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < CH * 4; i += 128) {
        const int t = i / 4, q = i % 4, jj = t % T, sb = t / T;
        s_dd[jj][sb][q] = make_float2(1e-3f + 1e-3f * ((t * 7 + q) % 97), 1e-2f * (((t * 5 + q) % 21) - 10));
        s_b[jj][q][sb] = make_float4(0.1f * ((t + q) % 7) - 0.3f, 0.05f * ((t * 3 + q) % 9) - 0.2f, 0.1f, -0.1f);
        s_c[jj][q][sb] = make_float4(0.2f, -0.1f * ((t + 2 * q) % 5), 0.05f * ((t + q) % 3), 0.3f);
    }
    __syncthreads();
    const int ch = lane & 3, sub = lane >> 2;
    (void)CH;
    float2 A[8], carry[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        A[p] = make_float2(-1.4427f * (2 * p + 1) * 0.1f, -1.4427f * (2 * p + 2) * 0.1f);
        carry[p] = make_float2(0.f, 0.f);
    }
    const auto fma2 = [](float2 a, float2 b, float2 c) {
        unsigned long long d, pa, pb, pc;
        asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(pc) : "f"(c.x), "f"(c.y));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pa), "l"(pb), "l"(pc));
        float2 r;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
        return r;
    };
    const auto mul2 = [&](float2 a, float2 b) { return fma2(a, b, make_float2(0.f, 0.f)); };
    for (int it = 0; it < iters; ++it) {
        // (1) local sweep, decays kept
        float2 a[T][8], h[8];
        float sd = 0.f;
#pragma unroll
        for (int p = 0; p < 8; ++p) h[p] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < T; ++j) {
            const float2 dd = s_dd[j][sub][ch];
            sd += dd.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 bq = s_b[j][q][sub];
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int p = 2 * q + hlf;
                    const float2 e = mul2(make_float2(dd.x, dd.x), A[p]);
                    a[j][p] = make_float2(ex2a(e.x), ex2a(e.y));
                    const float2 b2 = hlf ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
                    h[p] = fma2(a[j][p], h[p], mul2(make_float2(dd.y, dd.y), b2));
                }
            }
        }
        // (2) decay product of the sub-chunk, then the inclusive scan over
        // the eight sub-chunks of each channel (lanes 4 apart)
        float2 P[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float2 e = mul2(make_float2(sd, sd), A[p]);
            P[p] = make_float2(ex2a(e.x), ex2a(e.y));
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float2 hp = make_float2(__shfl_up_sync(0xffffffffu, h[p].x, 4 * off),
                                              __shfl_up_sync(0xffffffffu, h[p].y, 4 * off));
                const float2 pp = make_float2(__shfl_up_sync(0xffffffffu, P[p].x, 4 * off),
                                              __shfl_up_sync(0xffffffffu, P[p].y, 4 * off));
                if (sub >= off) {
                    h[p] = fma2(P[p], hp, h[p]);
                    P[p] = mul2(P[p], pp);
                }
            }
        }
        // state entering this sub-chunk, from the chunk's carry; the carry
        // of the next chunk from sub-chunk 7
        float2 hin[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const float2 he = make_float2(__shfl_up_sync(0xffffffffu, h[p].x, 4), __shfl_up_sync(0xffffffffu, h[p].y, 4));
            const float2 pe = make_float2(__shfl_up_sync(0xffffffffu, P[p].x, 4), __shfl_up_sync(0xffffffffu, P[p].y, 4));
            hin[p] = sub == 0 ? carry[p] : fma2(pe, carry[p], he);
            const float2 fin = fma2(P[p], carry[p], h[p]);
            carry[p] = make_float2(__shfl_sync(0xffffffffu, fin.x, ch + 28), __shfl_sync(0xffffffffu, fin.y, ch + 28));
        }
        // (3) re-sweep with the kept decays; C . h in-lane
#pragma unroll
        for (int j = 0; j < T; ++j) {
            const float2 dd = s_dd[j][sub][ch];
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 bq = s_b[j][q][sub], cq = s_c[j][q][sub];
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int p = 2 * q + hlf;
                    const float2 b2 = hlf ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
                    const float2 c2 = hlf ? make_float2(cq.z, cq.w) : make_float2(cq.x, cq.y);
                    hin[p] = fma2(a[j][p], hin[p], mul2(make_float2(dd.y, dd.y), b2));
                    acc = fma2(c2, hin[p], acc);
                }
            }
            s_y[warp][j][lane] = acc.x + acc.y;
        }
    }
    __syncthreads();
    float s = s_y[warp][lane % T][lane];
#pragma unroll
    for (int p = 0; p < 8; ++p) s += carry[p].x + carry[p].y;
    if (s == 12345.678f) sink[tid] = s;
}
}  // namespace

// Same as ssmpk_probe but with an explicit block shape: `blocks_per_sm` x SM
// count blocks of `threads` threads (a multiple of 32, at most 256), for
// measuring how throughput depends on the number of warps per scheduler.
PK_API double ssmpk_probe_shape(int kind, int iters, int blocks_per_sm, int threads);

// Runs one probe and returns its throughput in operations per second
// (ex2 / lg2 / rcp / tanh results for kinds 0, 1, 2, 4, scalar FMAs for
// kind 3, ex2 results of the mixed steps for kinds 5, 6, 7), timed with CUDA
// events around a single launch of `blocks_per_sm` x SM-count blocks of 256
// threads.  Returns a negative value on any CUDA error.  Synchronises the
// device; a measurement tool, not part of the scan path.
PK_API double ssmpk_probe(int kind, int iters, int blocks_per_sm) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1.0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1.0;
    if (kind < 0 || kind > 7 || iters <= 0 || blocks_per_sm <= 0 || blocks_per_sm > 8) return -2.0;
    float* sink = nullptr;
    if (cudaMalloc(&sink, 256 * sizeof(float)) != cudaSuccess) return -1.0;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    const dim3 grid(sms * blocks_per_sm), block(g_threads);
    auto launch = [&]() {
        switch (kind) {
            case 0: sfu_kernel<0><<<grid, block>>>(sink, iters, 1e-7f); break;
            case 1: sfu_kernel<1><<<grid, block>>>(sink, iters, 1e-7f); break;
            case 2: sfu_kernel<2><<<grid, block>>>(sink, iters, 1e-7f); break;
            case 4: sfu_kernel<4><<<grid, block>>>(sink, iters, 1e-7f); break;
            case 5: mix_kernel<0><<<grid, block>>>(sink, iters, 1e-7f); break;
            case 6: mix_kernel<1><<<grid, block>>>(sink, iters, 1e-7f); break;
            case 7: mix_kernel<2><<<grid, block>>>(sink, iters, 1e-7f); break;
            default: ffma2_kernel<<<grid, block>>>(sink, iters, 1e-7f); break;
        }
    };
    launch();  // warm-up
    cudaEventRecord(e0);
    launch();
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    const cudaError_t err = cudaEventElapsedTime(&ms, e0, e1);
    const cudaError_t last = cudaGetLastError();
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(sink);
    if (err != cudaSuccess || last != cudaSuccess || ms <= 0.f) return -1.0;
    const double per_thread = double(iters) * kU * (kind == 3 ? 2 : 1);
    return per_thread * double(grid.x) * double(g_threads) / (ms * 1e-3);
}

PK_API double ssmpk_probe_shape(int kind, int iters, int blocks_per_sm, int threads) {
    if (threads <= 0 || threads > 256 || threads % 32 != 0) return -2.0;
    g_threads = threads;
    const double r = ssmpk_probe(kind, iters, blocks_per_sm);
    g_threads = 256;
    return r;
}

// Number of SMs of the current device (so callers can normalise per SM).
PK_API int ssmpk_sm_count(void) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

// The in-warp time-split core (tsplit_kernel) with sub-chunks of T = 2 or 4
// steps: returns scan elements (step x channel x state) per second over one
// launch of 8 x SM-count blocks of 128 threads (residency set by the
// kernel's registers), timed with CUDA events after a warm-up launch;
// negative on error.  A measurement tool, not part of the scan path.
PK_API double ssmpk_timesplit(int T, int iters) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1.0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1.0;
    if ((T != 2 && T != 4) || iters <= 0) return -2.0;
    float* sink = nullptr;
    if (cudaMalloc(&sink, 128 * sizeof(float)) != cudaSuccess) return -1.0;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    const dim3 grid(sms * 8), block(128);
    auto launch = [&]() {
        if (T == 2) tsplit_kernel<2><<<grid, block>>>(sink, iters);
        else tsplit_kernel<4><<<grid, block>>>(sink, iters);
    };
    launch();
    cudaEventRecord(e0);
    launch();
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    const cudaError_t err = cudaEventElapsedTime(&ms, e0, e1);
    const cudaError_t last = cudaGetLastError();
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(sink);
    if (err != cudaSuccess || last != cudaSuccess || ms <= 0.f) return -1.0;
    // per block and iteration: 4 warps x 4 channels x 8T steps x 16 states
    const double per_block = double(iters) * 4 * 4 * 8 * T * 16;
    return per_block * double(grid.x) / (ms * 1e-3);
}
