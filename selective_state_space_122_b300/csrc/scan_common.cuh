// scan_common.cuh -- PTX wrappers (mbarrier, TMA, bulk copies, fences) and
// the per-element helpers shared by the scan kernels.
//
// Each translation unit that includes this header gets its own device error
// word (g_device_error): a kernel that gives up on a bounded wait sets a bit
// in it; the host reads and clears it through the unit's read function.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ssm_internal.cuh"

namespace ssm {
namespace {

static __device__ unsigned int g_device_error = 0;

// Limit of every bounded wait, in nanoseconds: 1 s unless the wait test hook
// (ssm_debug_wait_test) shortened it.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;
static __device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;
// Nonzero only under the wait test hook: the first segment of chain 0 keeps
// its hand-off flag unset, so the segment after it waits until the limit.
static __device__ int g_withhold_flag = 0;

__device__ __forceinline__ unsigned long long wait_limit_ns() {
    return *reinterpret_cast<volatile unsigned long long*>(&g_wait_limit_ns);
}
__device__ __forceinline__ bool withhold_handoff(int chain, int sgm) {
    return chain == 0 && sgm == 0 && *reinterpret_cast<volatile int*>(&g_withhold_flag) != 0;
}

// ------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

#ifndef SSM_WAIT_SPIN
#define SSM_WAIT_SPIN 0
#endif

// Wait for the phase with the given parity to complete; false after ~1 s.
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!(SSM_WAIT_SPIN ? mbar_test(bar, parity) : mbar_try(bar, parity)))
        if (globaltimer() - t0 > wait_limit_ns()) return false;
    return true;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (SSM_WAIT_SPIN ? mbar_test(bar, parity) : mbar_try(bar, parity)) return true;
    return mbar_wait_slow(bar, parity);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int c0, int c1, int c2, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int Nn>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(Nn) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void raise_error(unsigned int bit) { atomicOr(&g_device_error, bit); }

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void st_pair(T* p0, T* p1, float2 v);
template <>
__device__ __forceinline__ void st_pair<float>(float* p0, float* p1, float2 v) {
    *p0 = v.x;
    *p1 = v.y;
}
template <>
__device__ __forceinline__ void st_pair<__nv_bfloat16>(__nv_bfloat16* p0, __nv_bfloat16* p1, float2 v) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
    *p0 = b.x;
    *p1 = b.y;
}

// log1p(e) for e in [0, 1] as e * q(e), q a degree-7 polynomial fitted to
// log1p(e) / e on [0, 1] (least-squares iterated towards the minimax
// relative error; q(0) = 1 exactly).  Relative error below 4e-7 over the
// whole interval when evaluated in float32, so log1p(e) keeps every digit the
// bf16 inputs carry down to e -> 0, where ln2 * log2(1 + e) would lose
// them to the rounding of 1 + e.
__device__ __forceinline__ float2 log1p_unit2(float2 e) {
    float2 q = splat2(-8.778980002e-03f);
    q = fma2(q, e, splat2(4.498671740e-02f));
    q = fma2(q, e, splat2(-1.090230048e-01f));
    q = fma2(q, e, splat2(1.784721315e-01f));
    q = fma2(q, e, splat2(-2.453686744e-01f));
    q = fma2(q, e, splat2(3.328406513e-01f));
    q = fma2(q, e, splat2(-4.999817908e-01f));
    q = fma2(q, e, splat2(1.f));
    return mul2(q, e);
}

// softplus(x) = max(x, 0) + log1p(e^-|x|) for two values: one SFU exp2 each
// and the polynomial log1p above.  Relative error below 1e-6 for every x
// (the e^-|x| of ex2.approx and the polynomial); large |x| needs no special
// case (e underflows to 0 and the result is max(x, 0)).
__device__ __forceinline__ float2 softplus_poly2(float2 x) {
    const float2 e = make_float2(ex2_approx(-fabsf(x.x) * kLog2e), ex2_approx(-fabsf(x.y) * kLog2e));
    return add2(make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_unit2(e));
}

template <bool kFast>
__device__ __forceinline__ float2 softplus2_path(float2 x) {
    if constexpr (kFast) return softplus_poly2(x);
    else return make_float2(softplus_acc(x.x), softplus_acc(x.y));
}

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu(z) = z * sigmoid(z) = (z/2) * (1 + tanh(z/2)): one SFU operation.
// tanh.approx has an absolute error below 2^-10.9, so the gate is accurate to
// about 5e-4 * |z| / 2 -- below the rounding of a bfloat16 output.
template <bool kFast>
__device__ __forceinline__ float2 seg_silu2(float2 z) {
    if constexpr (kFast) {
        const float2 hz = mul2(z, splat2(0.5f));
        const float2 t = make_float2(tanh_approx(hz.x), tanh_approx(hz.y));
        return fma2(hz, t, hz);
    } else {
        return make_float2(silu_acc(z.x), silu_acc(z.y));
    }
}

}  // namespace
}  // namespace ssm
