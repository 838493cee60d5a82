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
