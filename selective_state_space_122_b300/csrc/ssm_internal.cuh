// ssm_internal.cuh -- parameter blocks and device helpers shared by the
// library's kernels and its host entry points.  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

enum class DType : int { F32 = 0, BF16 = 1 };

// Arguments of one full-sequence scan; layouts as in ssm_scan.h.
struct ScanArgs {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    void* out;
    float* last_state;
    int64_t batch, dim, seqlen;
    int dstate;
    int softplus;
    const float* h0;        // initial state (batch, dim, dstate) f32, or null for zero
    // B and C per channel group: (batch, ngroups, dstate, seqlen); channel d
    // reads block b * ngroups + d / gch (gch = dim / ngroups channels per group)
    int64_t ngroups = 1;
    int64_t gch = 0;
};

// Arguments of one decode step; layouts as in ssm_scan.h.
struct UpdateArgs {
    float* state;
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* dt_bias;
    void* out;
    int64_t batch, dim;
    int dstate;
    int softplus;
    int64_t ngroups = 1;   // B, C: (batch, ngroups, dstate); channel d reads group d / gch
    int64_t gch = 0;
};

// One compiled layout of the scan kernel: G states per lane (the N / G
// lanes of a channel are adjacent), S warps per CTA, TL time lanes per warp,
// K steps per sub-chunk, CW channels per CTA.  S * TL > 1 splits every chunk
// of S * TL * K steps into sub-chunks combined with the associative scan.
struct ScanLayoutInfo {
    int G, S, TL, K, CW;
};

struct ScanPlan {
    int layout;  // index into the compiled layouts for this d_state
};

// TMA fast paths (scan_seg.cu): the staged-sequence padding (a multiple of
// 64 steps) and whether a call's pointers and sizes suit the tensor maps.
int64_t staged_lpad(int64_t seqlen);
bool tma_rows_supported(const ScanArgs& a, DType dt);
// Segmented direct scan (scan_seg.cu): needs staged B/C plus the segment
// hand-off state and flags (seg_workspace_bytes).
int64_t seg_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate, int elem_bytes,
                            int64_t ngroups);
cudaError_t launch_scan_seg(const ScanArgs& a, DType dt, void* workspace, int sms, cudaStream_t s);

// Depthwise causal conv1d (+ SiLU) and its decode step (conv1d.cu); layouts
// as in ssm_scan.h.  For the decode step, state_out is the state updated in
// place and state_in is unused.
struct ConvArgs {
    const void* x;
    const float* w;
    const float* bias;
    const float* state_in;
    void* out;
    float* state_out;
    int64_t batch, dim, seqlen;
    int width;
    int silu;
};
cudaError_t launch_conv1d_fwd(const ConvArgs& a, DType dt, cudaStream_t s);
cudaError_t launch_conv1d_update(const ConvArgs& a, DType dt, cudaStream_t s);

// Backward of the scan (scan_bwd.cu); layouts as in ssm_scan.h.  dD, dz and
// dbias may be null (not computed).  Workspace: the state entering every
// chunk (bwd_workspace_bytes).
struct BwdArgs {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    int softplus;
    const void* dout;
    void* du;
    void* ddelta;
    float* dA;
    float* dB;
    float* dC;
    float* dD;
    void* dz;
    float* dbias;
    int64_t batch, dim, seqlen;
    int dstate;
    int64_t ngroups = 1;   // B, C, dB, dC: (batch, ngroups, dstate, seqlen)
    int64_t gch = 0;       // channels per group (dim / ngroups)
    // scan from a given state whose final state enters the loss (all nullable):
    // h_{-1}, dL/d last_state in, dL/d h_{-1} out; (batch, dim, dstate) f32
    const float* h0 = nullptr;
    const float* dlast = nullptr;
    float* dh0 = nullptr;
};
int64_t bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate);
cudaError_t launch_scan_bwd(const BwdArgs& a, DType dt, void* workspace, int sms, cudaStream_t s);

// Tensor-memory scan (scan_tmem.cu): bf16 activations, 16 states.  Workspace:
// the staged one-hot MMA operands of B and C plus the segment hand-off state.
bool tmem_supported(const ScanArgs& a, DType dt);
int64_t tmem_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate, int64_t ngroups);
// variant 3: the warp-specialised kernel (four states per lane); otherwise
// two states per lane (8 consumer warps).
cudaError_t launch_scan_tmem(const ScanArgs& a, DType dt, void* workspace, int sms, cudaStream_t s, int variant);
int read_tmem_device_error(bool clear);
int read_device_error(bool clear);
// The wait test hook (ssm_debug_wait_test) in the segmented and the
// tensor-memory kernels' units: withhold flag and wait limit in ns; -1 on failure.
int set_wait_test_seg(int withhold, unsigned long long limit_ns);
int set_wait_test_tmem(int withhold, unsigned long long limit_ns);

// Every host-side check of a scan call (ssm_api.cu): returns SSM_OK or the
// ssm_status code the call would return, touching no device state.
int check_scan_call(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* delta_bias, const float* initial_state, const void* out,
                    const float* last_state, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                    int64_t ngroups, int dtype, const void* workspace, int64_t workspace_bytes);

int scan_layout_count(int dstate);
ScanLayoutInfo scan_layout_info(int dstate, int layout);
cudaError_t launch_scan_fwd(const ScanArgs& a, DType dt, const ScanPlan& plan, cudaStream_t s);
cudaError_t launch_state_update(const UpdateArgs& a, DType dt, int sms, cudaStream_t s);
// The decode unit's device error word (its bulk-copy pipeline's bounded waits)
// and its wait test hook (as set_wait_test_seg).
int read_update_device_error(bool clear);
int set_wait_test_update(int withhold, unsigned long long limit_ns);

// ---------------------------------------------------------------- device side

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// 2^x on the special-function unit (one MUFU.EX2; flushes denormal results).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// exp2 of the decay exponent.  kFast: the SFU instruction; otherwise the
// CUDA math library's exp2f (float32 inputs, where speed is secondary).
template <bool kFast>
__device__ __forceinline__ float decay_exp2(float x) {
    if constexpr (kFast) return ex2_approx(x);
    else return exp2f(x);
}

// softplus(x) = log(1 + e^x).  Above 20 the correction log1p(e^-x) is below
// 2.1e-9 and x itself is returned.
__device__ __forceinline__ float softplus_acc(float x) {
    return x > 20.f ? x : log1pf(expf(x));
}

// softplus on the special-function unit: e = 2^(x log2 e), then
// log1p(e) = ln2 * log2(1 + e), or, for e < 2^-6 where 1 + e would drop
// digits of e, the series e - e^2/2 + e^3/3 - e^4/4 (truncation < e^5/5,
// i.e. relative error < 2e-9).  Above 15 the correction log1p(e^-x) < 3.1e-7
// is dropped (relative error < 2.1e-8).
__device__ __forceinline__ float softplus_fast(float x) {
    const float e = ex2_approx(x * kLog2e);
    const float via_log = kLn2 * lg2_approx(1.f + e);
    const float series = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.33333334f), -0.5f), 1.f);
    const float r = e < 0.015625f ? series : via_log;
    return x > 15.f ? x : r;
}

// silu(z) = z / (1 + e^-z)
__device__ __forceinline__ float silu_acc(float zv) {
    return zv / (1.f + expf(-zv));
}

// silu on the special-function unit: one exp2 and one reciprocal.  For
// z < -88 the exponential overflows to +inf and the result is -0.
__device__ __forceinline__ float silu_fast(float zv) {
    return zv * rcp_approx(1.f + ex2_approx(-zv * kLog2e));
}

// ---------------------------------------------------------------- f32x2
// Packed two-lane float32 arithmetic (one instruction for two values).  Each
// helper is a single PTX instruction on 64-bit register pairs, with the pack
// and unpack as separate plain moves, so the register allocator can place the
// halves in the pair directly and the scheduler can move each instruction
// freely (no scoped asm blocks, which would pin the instruction order).

__device__ __forceinline__ unsigned long long pk2(float2 a) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
    return r;
}

__device__ __forceinline__ float2 up2(unsigned long long r) {
    float2 a;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
    return a;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)));
    return up2(d);
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)));
    return up2(d);
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
    return up2(d);
}

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// Component i (a compile-time constant after unrolling) of a float4 / float2.
__device__ __forceinline__ float comp(const float4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ float comp(const float2& v, int i) { return i == 0 ? v.x : v.y; }

// softplus of two values with packed arithmetic; same method and bounds as
// softplus_fast.
__device__ __forceinline__ float2 softplus_fast2(float2 x) {
    const float2 e = make_float2(ex2_approx(x.x * kLog2e), ex2_approx(x.y * kLog2e));
    const float2 ope = add2(e, splat2(1.f));
    const float2 via_log = mul2(splat2(kLn2), make_float2(lg2_approx(ope.x), lg2_approx(ope.y)));
    const float2 poly = fma2(e, fma2(e, fma2(e, splat2(-0.25f), splat2(0.33333334f)), splat2(-0.5f)),
                             splat2(1.f));
    const float2 series = mul2(e, poly);
    float2 r;
    r.x = x.x > 15.f ? x.x : (e.x < 0.015625f ? series.x : via_log.x);
    r.y = x.y > 15.f ? x.y : (e.y < 0.015625f ? series.y : via_log.y);
    return r;
}

// silu of two values: z / (1 + 2^(-z log2 e)).
__device__ __forceinline__ float2 silu_fast2(float2 z) {
    const float2 nz = mul2(z, splat2(-kLog2e));
    const float2 den = add2(make_float2(ex2_approx(nz.x), ex2_approx(nz.y)), splat2(1.f));
    return mul2(z, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
}

template <bool kFast>
__device__ __forceinline__ float2 softplus_f2(float2 x) {
    if constexpr (kFast) return softplus_fast2(x);
    else return make_float2(softplus_acc(x.x), softplus_acc(x.y));
}

template <bool kFast>
__device__ __forceinline__ float2 silu_f2(float2 z) {
    if constexpr (kFast) return silu_fast2(z);
    else return make_float2(silu_acc(z.x), silu_acc(z.y));
}

template <bool kFast>
__device__ __forceinline__ float softplus_f(float x) {
    if constexpr (kFast) return softplus_fast(x);
    else return softplus_acc(x);
}

template <bool kFast>
__device__ __forceinline__ float silu_f(float zv) {
    if constexpr (kFast) return silu_fast(zv);
    else return silu_acc(zv);
}

}  // namespace ssm
