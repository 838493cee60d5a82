// ssm_api.cu -- the library's C ABI (declared in include/ssm_scan.h):
// argument validation, work planning and kernel dispatch.  Nothing here
// allocates, copies or synchronises; every check runs on the host before the
// first launch, so a rejected call leaves every buffer untouched.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/ssm_scan.h"
#include "ssm_internal.cuh"

namespace {

constexpr int64_t kMaxElems = int64_t(1) << 40;
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// a * b > limit for positive a, b, without forming the (possibly overflowing) product
bool prod_exceeds(int64_t a, int64_t b, int64_t limit) { return a > limit / b; }

// batch * seqlen * dim above the element limit (all positive)
bool too_many_elems(int64_t batch, int64_t seqlen, int64_t dim) {
    return prod_exceeds(batch, seqlen, kMaxElems) || prod_exceeds(batch * seqlen, dim, kMaxElems);
}

struct Span {
    const void* p;
    int64_t bytes;
};

bool overlap(Span a, Span b) {
    if (!a.p || !b.p || a.bytes <= 0 || b.bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + (uintptr_t)b.bytes && b0 < a0 + (uintptr_t)a.bytes;
}

// Number of SMs of the current device (cached per device).
ssm_status sm_count(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return SSM_ERR_DEVICE;
    if (dev < kMaxDevices) {
        int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *out = c;
            return SSM_OK;
        }
    }
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
        return SSM_ERR_DEVICE;
    if (dev < kMaxDevices) g_sm_count[dev].store(c, std::memory_order_relaxed);
    *out = c;
    return SSM_OK;
}

// Kernel forced by ssm_force_scan_path (tests and benchmarks that compare the
// kernels); the default, path 0, is the library's own choice.
std::atomic<int> g_force_path{SSM_PATH_AUTO};
std::atomic<int> g_force_layout{-1};

// Pick a compiled scan layout.  Every channel walks the sequence in order,
// so a CTA's work is CW channels x L steps and its warps share it.  The
// score is the work of the busiest SM scheduler (warps are the unit a
// scheduler runs; a warp cannot migrate), times a per-layout cost factor:
// split layouts pay ~2 extra FP32 operations per (t, state) and layouts with
// few states per lane pay for the cross-lane y reduction.
int plan_layout(int64_t batch, int64_t dim, int N, int sms) {
    const int count = ssm::scan_layout_count(N);
    const int forced = g_force_layout.load(std::memory_order_relaxed);
    if (g_force_path.load(std::memory_order_relaxed) == SSM_PATH_GENERIC && forced >= 0 && forced < count)
        return forced;
    const double schedulers = 4.0 * sms;
    int best = 0;
    double best_t = 1e300;
    for (int l = 0; l < count; ++l) {
        const ssm::ScanLayoutInfo li = ssm::scan_layout_info(N, l);
        const int64_t ctas = batch * ((dim + li.CW - 1) / li.CW);
        const double warps = double(ctas) * li.S;
        const double per_warp = double(li.CW) / li.S;               // channels of work per warp
        const double busiest = std::ceil(warps / schedulers) * per_warp;
        double cost = (li.S * li.TL > 1) ? 1.15 : 1.0;
        const int R = N / li.G;
        cost *= 1.0 + 0.03 * (R > 1 ? R : 0);
        const double t = busiest * cost;
        if (t < best_t * 0.999) {
            best_t = t;
            best = l;
        }
    }
    return best;
}

bool dstate_ok(int64_t n) { return n == 4 || n == 8 || n == 16; }

// CUDA runtime error behind the calling thread's last SSM_ERR_LAUNCH.
thread_local cudaError_t t_last_launch = cudaSuccess;

ssm_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return SSM_OK;
    t_last_launch = e;
    return SSM_ERR_LAUNCH;
}

}  // namespace

extern "C" {

const char* ssm_status_string(int status) {
    switch (status) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_NULL: return "SSM_ERR_NULL: a required pointer is NULL";
        case SSM_ERR_SHAPE: return "SSM_ERR_SHAPE: a size is <= 0 or the problem is too large";
        case SSM_ERR_ALIGN: return "SSM_ERR_ALIGN: a pointer is misaligned";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED: d_state must be 4, 8 or 16";
        case SSM_ERR_DTYPE: return "SSM_ERR_DTYPE: dtype must be SSM_F32 or SSM_BF16";
        case SSM_ERR_ALIAS: return "SSM_ERR_ALIAS: an output overlaps an input";
        case SSM_ERR_LAUNCH: return "SSM_ERR_LAUNCH: the CUDA runtime rejected a launch";
        case SSM_ERR_DEVICE: return "SSM_ERR_DEVICE: no usable CUDA device";
        case SSM_ERR_SCRATCH:
            return "SSM_ERR_SCRATCH: the sizes need more scratch than ssm_scan_fwd_noalloc's fixed array holds";
        default: return "unknown ssm_status";
    }
}

int ssm_version(void) { return 101; }

ssm_status ssm_debug_wait_test(int withhold_flag, int64_t wait_limit_ns) {
    const unsigned long long ns = wait_limit_ns > 0 ? (unsigned long long)wait_limit_ns : 1000000000ull;
    const int w = withhold_flag ? 1 : 0;
    if (ssm::set_wait_test_seg(w, ns) != 0 || ssm::set_wait_test_tmem(w, ns) != 0 ||
        ssm::set_wait_test_update(w, ns) != 0)
        return SSM_ERR_DEVICE;
    return SSM_OK;
}

ssm_status ssm_force_scan_path(int path, int generic_layout) {
    if (path < SSM_PATH_AUTO || path > SSM_PATH_GENERIC) return SSM_ERR_SHAPE;
    g_force_layout.store(path == SSM_PATH_GENERIC ? generic_layout : -1, std::memory_order_relaxed);
    g_force_path.store(path, std::memory_order_relaxed);
    return SSM_OK;
}

const char* ssm_last_launch_error(void) {
    return t_last_launch == cudaSuccess ? "no launch error" : cudaGetErrorString(t_last_launch);
}

int64_t ssm_scan_workspace_bytes_grouped(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                         int64_t ngroups, int dtype) {
    if (dtype != SSM_F32 && dtype != SSM_BF16) return -1;
    if (dim <= 0 || dim >= (int64_t(1) << 31)) return -1;
    if (batch <= 0 || seqlen <= 0 || !dstate_ok(dstate) || batch > 65535 || seqlen > (int64_t(1) << 40))
        return -1;
    if (ngroups <= 0 || dim % ngroups != 0 || too_many_elems(batch, seqlen, dim)) return -1;
    int64_t need = ssm::seg_workspace_bytes(batch, dim, seqlen, (int)dstate, dtype == SSM_BF16 ? 2 : 4, ngroups);
    if (dtype == SSM_BF16) need = std::max(need, ssm::tmem_workspace_bytes(batch, dim, seqlen, (int)dstate, ngroups));
    return need;
}

int64_t ssm_scan_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int dtype) {
    return ssm_scan_workspace_bytes_grouped(batch, dim, seqlen, dstate, 1, dtype);
}

int ssm_device_error(int clear) {
    const int a = ssm::read_device_error(clear != 0);
    const int b = ssm::read_tmem_device_error(clear != 0);
    const int c = ssm::read_update_device_error(clear != 0);
    return (a < 0 || b < 0 || c < 0) ? -1 : (a | b | c);
}

}  // extern "C"

namespace ssm {

// Every host-side check of a (grouped) scan call: dtype, pointers, sizes,
// alignment and aliasing, in that order.  Nothing touches the device.
int check_scan_call(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* delta_bias, const float* initial_state, const void* out,
                    const float* last_state, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                    int64_t ngroups, int dtype, const void* workspace, int64_t workspace_bytes) {
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!u || !delta || !A || !B || !C || !out) return SSM_ERR_NULL;
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || dstate <= 0) return SSM_ERR_SHAPE;
    if (ngroups <= 0 || dim % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dstate_ok(dstate)) return SSM_ERR_UNSUPPORTED;
    if (batch > 65535 || dim >= (int64_t(1) << 31) || seqlen > (int64_t(1) << 40)) return SSM_ERR_SHAPE;
    if (too_many_elems(batch, seqlen, dim)) return SSM_ERR_SHAPE;
    const int64_t es = dtype == SSM_BF16 ? 2 : 4;
    const uintptr_t ea = (uintptr_t)es;
    if (!aligned(u, ea) || !aligned(delta, ea) || !aligned(B, ea) || !aligned(C, ea) ||
        !aligned(out, ea) || (z && !aligned(z, ea)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
        (delta_bias && !aligned(delta_bias, 4)) || (last_state && !aligned(last_state, 4)) ||
        (initial_state && !aligned(initial_state, 4)))
        return SSM_ERR_ALIGN;

    const int64_t x_bytes = batch * seqlen * dim * es;
    const int64_t bc_bytes = batch * ngroups * dstate * seqlen * es;
    const Span ins[] = {{u, x_bytes}, {delta, x_bytes}, {z, x_bytes}, {B, bc_bytes}, {C, bc_bytes},
                        {A, dim * dstate * 4}, {D, dim * 4}, {delta_bias, dim * 4}};
    const Span so{out, x_bytes}, sl{last_state, batch * dim * dstate * 4};
    for (const Span& s : ins)
        if (overlap(so, s) || overlap(sl, s)) return SSM_ERR_ALIAS;
    if (overlap(so, sl)) return SSM_ERR_ALIAS;
    // the initial state is an input; it may be the final-state array itself
    // (resume in place), but must not overlap any other output or input
    const Span sh{initial_state, batch * dim * dstate * 4};
    if (initial_state) {
        if (overlap(so, sh)) return SSM_ERR_ALIAS;
        if (overlap(sl, sh) && initial_state != last_state) return SSM_ERR_ALIAS;
        for (const Span& s : ins)
            if (overlap(sh, s)) return SSM_ERR_ALIAS;
    }

    if (workspace_bytes < 0 || (workspace && workspace_bytes == 0)) return SSM_ERR_SHAPE;
    if (workspace) {
        if (!aligned(workspace, 16)) return SSM_ERR_ALIGN;
        const Span sw{workspace, workspace_bytes};
        for (const Span& s : ins)
            if (overlap(sw, s)) return SSM_ERR_ALIAS;
        if (overlap(sw, so) || overlap(sw, sl) || overlap(sw, sh)) return SSM_ERR_ALIAS;
    }
    return SSM_OK;
}

}  // namespace ssm

extern "C" {

ssm_status ssm_scan_fwd_grouped(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const float* delta_bias, int softplus_flag,
                                const float* initial_state, void* out, float* last_state, int64_t batch,
                                int64_t dim, int64_t seqlen, int64_t dstate, int64_t ngroups, int dtype,
                                void* workspace, int64_t workspace_bytes, void* stream) {
    if (const int chk = ssm::check_scan_call(u, delta, A, B, C, D, z, delta_bias, initial_state, out, last_state,
                                             batch, dim, seqlen, dstate, ngroups, dtype, workspace, workspace_bytes);
        chk != SSM_OK)
        return static_cast<ssm_status>(chk);
    const int64_t es = dtype == SSM_BF16 ? 2 : 4;

    int sms = 0;
    if (ssm_status st = sm_count(&sms); st != SSM_OK) return st;

    ssm::ScanArgs a{u, delta, A, B, C, D, z, delta_bias, out, last_state,
                    batch, dim, seqlen, (int)dstate, softplus_flag ? 1 : 0, initial_state};
    a.ngroups = ngroups;
    a.gch = dim / ngroups;
    const ssm::DType dt = dtype == SSM_BF16 ? ssm::DType::BF16 : ssm::DType::F32;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The tensor-memory scan (two states per lane) runs whenever its
    // requirements hold (bf16, 16 states), else the segmented scan, else the
    // generic kernel; ssm_force_scan_path picks one of them instead.
    const int force = g_force_path.load(std::memory_order_relaxed);
    // (chains * 64 segments must stay a 32-bit task count)
    const bool fast_ok = workspace && ssm::tma_rows_supported(a, dt) &&
                         batch * ((dim + 127) / 128 * dstate) * 64 < (int64_t(1) << 31);
    const bool tmem_ok = fast_ok && ssm::tmem_supported(a, dt) &&
                         workspace_bytes >= ssm::tmem_workspace_bytes(batch, dim, seqlen, (int)dstate, ngroups);
    const bool seg_ok = fast_ok &&
                        workspace_bytes >= ssm::seg_workspace_bytes(batch, dim, seqlen, (int)dstate, (int)es, ngroups);
    if (force == SSM_PATH_TMEM2 || force == SSM_PATH_WS) {
        if (!tmem_ok) return SSM_ERR_UNSUPPORTED;
        return launch_status(ssm::launch_scan_tmem(a, dt, workspace, sms, st, force == SSM_PATH_WS ? 3 : 2));
    }
    if (force == SSM_PATH_SEG) {
        if (!seg_ok) return SSM_ERR_UNSUPPORTED;
        return launch_status(ssm::launch_scan_seg(a, dt, workspace, sms, st));
    }
    if (force == SSM_PATH_AUTO && tmem_ok)
        return launch_status(ssm::launch_scan_tmem(a, dt, workspace, sms, st, 2));
    if (force == SSM_PATH_AUTO && seg_ok) return launch_status(ssm::launch_scan_seg(a, dt, workspace, sms, st));
    ssm::ScanPlan plan{plan_layout(batch, dim, (int)dstate, sms)};
    return launch_status(ssm::launch_scan_fwd(a, dt, plan, st));
}

ssm_status ssm_scan_fwd_from_state(const void* u, const void* delta, const float* A, const void* B,
                                   const void* C, const float* D, const void* z, const float* delta_bias,
                                   int softplus_flag, const float* initial_state, void* out, float* last_state,
                                   int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int dtype,
                                   void* workspace, int64_t workspace_bytes, void* stream) {
    return ssm_scan_fwd_grouped(u, delta, A, B, C, D, z, delta_bias, softplus_flag, initial_state, out, last_state,
                                batch, dim, seqlen, dstate, 1, dtype, workspace, workspace_bytes, stream);
}

ssm_status ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                        const void* C, const float* D, const void* z, const float* delta_bias,
                        int softplus_flag, void* out, float* last_state, int64_t batch,
                        int64_t dim, int64_t seqlen, int64_t dstate, int dtype, void* workspace,
                        int64_t workspace_bytes, void* stream) {
    return ssm_scan_fwd_from_state(u, delta, A, B, C, D, z, delta_bias, softplus_flag, nullptr, out, last_state,
                                   batch, dim, seqlen, dstate, dtype, workspace, workspace_bytes, stream);
}

ssm_status ssm_conv1d_fwd(const void* x, const float* weight, const float* bias, int silu_flag,
                          const float* conv_state_in, void* out, float* conv_state_out, int64_t batch,
                          int64_t dim, int64_t seqlen, int64_t width, int dtype, void* stream) {
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!x || !weight || !out) return SSM_ERR_NULL;
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || width <= 0) return SSM_ERR_SHAPE;
    if (width > 4) return SSM_ERR_UNSUPPORTED;
    if (batch > 65535 || dim >= (int64_t(1) << 31) || seqlen > (int64_t(1) << 40)) return SSM_ERR_SHAPE;
    if (too_many_elems(batch, seqlen, dim)) return SSM_ERR_SHAPE;
    const int64_t es = dtype == SSM_BF16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(out, es) || !aligned(weight, 4) || (bias && !aligned(bias, 4)) ||
        (conv_state_in && !aligned(conv_state_in, 4)) || (conv_state_out && !aligned(conv_state_out, 4)))
        return SSM_ERR_ALIGN;
    const int64_t x_bytes = batch * seqlen * dim * es, st_bytes = batch * dim * (width - 1) * 4;
    const Span sx{x, x_bytes}, sw{weight, dim * width * 4}, sb{bias, dim * 4}, si{conv_state_in, st_bytes};
    const Span so{out, x_bytes}, sso{conv_state_out, st_bytes};
    for (const Span& s : {sx, sw, sb, si})
        if (overlap(so, s)) return SSM_ERR_ALIAS;
    for (const Span& s : {sx, sw, sb, so})
        if (overlap(sso, s)) return SSM_ERR_ALIAS;
    // the carried state may be updated in place, but not overlap partially
    if (overlap(si, sso) && conv_state_in != conv_state_out) return SSM_ERR_ALIAS;
    int sms = 0;
    if (ssm_status st = sm_count(&sms); st != SSM_OK) return st;
    ssm::ConvArgs a{x, weight, bias, conv_state_in, out, conv_state_out, batch, dim, seqlen, (int)width,
                    silu_flag ? 1 : 0};
    return launch_status(ssm::launch_conv1d_fwd(a, dtype == SSM_BF16 ? ssm::DType::BF16 : ssm::DType::F32,
                                                static_cast<cudaStream_t>(stream)));
}

ssm_status ssm_conv1d_update(float* conv_state, const void* x, const float* weight, const float* bias,
                             int silu_flag, void* out, int64_t batch, int64_t dim, int64_t width, int dtype,
                             void* stream) {
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!x || !weight || !out || (width > 1 && !conv_state)) return SSM_ERR_NULL;
    if (batch <= 0 || dim <= 0 || width <= 0) return SSM_ERR_SHAPE;
    if (width > 4) return SSM_ERR_UNSUPPORTED;
    if (prod_exceeds(batch, dim, kMaxElems / 16)) return SSM_ERR_SHAPE;
    const int64_t es = dtype == SSM_BF16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(out, es) || !aligned(weight, 4) || (bias && !aligned(bias, 4)) ||
        (conv_state && !aligned(conv_state, 4)))
        return SSM_ERR_ALIGN;
    const Span sx{x, batch * dim * es}, sw{weight, dim * width * 4}, sb{bias, dim * 4};
    const Span so{out, batch * dim * es}, ss{conv_state, batch * dim * (width - 1) * 4};
    for (const Span& s : {sx, sw, sb, ss})
        if (overlap(so, s)) return SSM_ERR_ALIAS;
    for (const Span& s : {sx, sw, sb})
        if (overlap(ss, s)) return SSM_ERR_ALIAS;
    int sms = 0;
    if (ssm_status st = sm_count(&sms); st != SSM_OK) return st;
    ssm::ConvArgs a{x, weight, bias, nullptr, out, conv_state, batch, dim, 1, (int)width, silu_flag ? 1 : 0};
    return launch_status(ssm::launch_conv1d_update(a, dtype == SSM_BF16 ? ssm::DType::BF16 : ssm::DType::F32,
                                                   static_cast<cudaStream_t>(stream)));
}

int64_t ssm_scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int dtype) {
    if (dtype != SSM_F32 && dtype != SSM_BF16) return -1;
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || !dstate_ok(dstate) || batch > 65535 || dim >= (int64_t(1) << 31) ||
        seqlen > (int64_t(1) << 40) || too_many_elems(batch, seqlen, dim))
        return -1;
    return std::max<int64_t>(16, ssm::bwd_workspace_bytes(batch, dim, seqlen, (int)dstate));
}

ssm_status ssm_scan_bwd_from_state(const void* u, const void* delta, const float* A, const void* B,
                                   const void* C, const float* D, const void* z, const float* delta_bias,
                                   int softplus_flag, const float* initial_state, const void* dout,
                                   const float* dlast, void* du, void* ddelta, float* dA, float* dB, float* dC,
                                   float* dD, void* dz, float* ddelta_bias, float* dinitial_state, int64_t batch,
                                   int64_t dim, int64_t seqlen, int64_t dstate, int64_t ngroups, int dtype,
                                   void* workspace, int64_t workspace_bytes, void* stream) {
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!u || !delta || !A || !B || !C || !dout || !du || !ddelta || !dA || !dB || !dC || !workspace)
        return SSM_ERR_NULL;
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || dstate <= 0) return SSM_ERR_SHAPE;
    if (ngroups <= 0 || dim % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dstate_ok(dstate)) return SSM_ERR_UNSUPPORTED;
    if (batch > 65535 || dim >= (int64_t(1) << 31) || seqlen > (int64_t(1) << 40)) return SSM_ERR_SHAPE;
    if (too_many_elems(batch, seqlen, dim)) return SSM_ERR_SHAPE;
    if (workspace_bytes < ssm::bwd_workspace_bytes(batch, dim, seqlen, (int)dstate)) return SSM_ERR_SHAPE;
    const int64_t es = dtype == SSM_BF16 ? 2 : 4;
    const uintptr_t ea = (uintptr_t)es;
    if (!aligned(u, ea) || !aligned(delta, ea) || !aligned(B, ea) || !aligned(C, ea) || !aligned(dout, ea) ||
        (z && !aligned(z, ea)) || !aligned(du, ea) || !aligned(ddelta, ea) || (dz && !aligned(dz, ea)) ||
        !aligned(A, 4) || (D && !aligned(D, 4)) || (delta_bias && !aligned(delta_bias, 4)) || !aligned(dA, 4) ||
        !aligned(dB, 4) || !aligned(dC, 4) || (dD && !aligned(dD, 4)) || (ddelta_bias && !aligned(ddelta_bias, 4)) ||
        !aligned(workspace, 16) || (initial_state && !aligned(initial_state, 16)) || (dlast && !aligned(dlast, 16)) ||
        (dinitial_state && !aligned(dinitial_state, 16)))
        return SSM_ERR_ALIGN;
    const int64_t x_bytes = batch * seqlen * dim * es, bc_bytes = batch * ngroups * dstate * seqlen * es;
    const int64_t gbc_bytes = batch * ngroups * dstate * seqlen * 4;
    const int64_t st_bytes = batch * dim * dstate * 4;
    const Span ins[] = {{u, x_bytes}, {delta, x_bytes}, {z, x_bytes}, {dout, x_bytes}, {B, bc_bytes},
                        {C, bc_bytes}, {A, dim * dstate * 4}, {D, dim * 4}, {delta_bias, dim * 4},
                        {initial_state, st_bytes}, {dlast, st_bytes}};
    const Span outs[] = {{du, x_bytes}, {ddelta, x_bytes}, {dz, x_bytes}, {dA, dim * dstate * 4},
                         {dB, gbc_bytes}, {dC, gbc_bytes}, {dD, dim * 4},
                         {ddelta_bias, dim * 4}, {workspace, workspace_bytes}, {dinitial_state, st_bytes}};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        for (const Span& s : ins)
            if (overlap(outs[i], s)) return SSM_ERR_ALIAS;
        for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
            if (overlap(outs[i], outs[j])) return SSM_ERR_ALIAS;
    }
    int sms = 0;
    if (ssm_status st = sm_count(&sms); st != SSM_OK) return st;
    ssm::BwdArgs a{u, delta, A, B, C, D, z, delta_bias, softplus_flag ? 1 : 0, dout, du, ddelta, dA, dB, dC,
                   D ? dD : nullptr, z ? dz : nullptr, delta_bias ? ddelta_bias : nullptr, batch, dim, seqlen,
                   (int)dstate};
    a.ngroups = ngroups;
    a.gch = dim / ngroups;
    a.h0 = initial_state;
    a.dlast = dlast;
    a.dh0 = dinitial_state;
    return launch_status(ssm::launch_scan_bwd(a, dtype == SSM_BF16 ? ssm::DType::BF16 : ssm::DType::F32, workspace,
                                              sms, static_cast<cudaStream_t>(stream)));
}

ssm_status ssm_scan_bwd_grouped(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const float* delta_bias, int softplus_flag,
                                const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC,
                                float* dD, void* dz, float* ddelta_bias, int64_t batch, int64_t dim,
                                int64_t seqlen, int64_t dstate, int64_t ngroups, int dtype, void* workspace,
                                int64_t workspace_bytes, void* stream) {
    return ssm_scan_bwd_from_state(u, delta, A, B, C, D, z, delta_bias, softplus_flag, nullptr, dout, nullptr, du,
                                   ddelta, dA, dB, dC, dD, dz, ddelta_bias, nullptr, batch, dim, seqlen, dstate,
                                   ngroups, dtype, workspace, workspace_bytes, stream);
}

ssm_status ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, int softplus_flag,
                        const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC, float* dD,
                        void* dz, float* ddelta_bias, int64_t batch, int64_t dim, int64_t seqlen,
                        int64_t dstate, int dtype, void* workspace, int64_t workspace_bytes, void* stream) {
    return ssm_scan_bwd_grouped(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dout, du, ddelta, dA, dB, dC,
                                dD, dz, ddelta_bias, batch, dim, seqlen, dstate, 1, dtype, workspace,
                                workspace_bytes, stream);
}

ssm_status ssm_state_update_grouped(float* state, const void* x, const void* dt, const float* A, const void* B,
                                    const void* C, const float* D, const void* z, const float* dt_bias, void* out,
                                    int64_t batch, int64_t dim, int64_t dstate, int64_t ngroups, int dt_softplus,
                                    int dtype, void* stream) {
    if (dtype != SSM_F32 && dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!state || !x || !dt || !A || !B || !C || !out) return SSM_ERR_NULL;
    if (batch <= 0 || dim <= 0 || dstate <= 0) return SSM_ERR_SHAPE;
    if (ngroups <= 0 || dim % ngroups != 0 || dim >= (int64_t(1) << 31)) return SSM_ERR_SHAPE;
    if (!dstate_ok(dstate)) return SSM_ERR_UNSUPPORTED;
    if (prod_exceeds(batch, dim, kMaxElems / 16)) return SSM_ERR_SHAPE;
    const int64_t es = dtype == SSM_BF16 ? 2 : 4;
    const uintptr_t ea = (uintptr_t)es;
    if (!aligned(state, 16) || !aligned(A, 16) || !aligned(x, ea) || !aligned(dt, ea) ||
        !aligned(B, ea) || !aligned(C, ea) || !aligned(out, ea) || (z && !aligned(z, ea)) ||
        (D && !aligned(D, 4)) || (dt_bias && !aligned(dt_bias, 4)))
        return SSM_ERR_ALIGN;

    const int64_t tok = batch * dim * es, bc = batch * ngroups * dstate * es;
    const Span ins[] = {{x, tok}, {dt, tok}, {z, tok}, {B, bc}, {C, bc},
                        {A, dim * dstate * 4}, {D, dim * 4}, {dt_bias, dim * 4}};
    const Span ss{state, batch * dim * dstate * 4}, so{out, tok};
    for (const Span& s : ins)
        if (overlap(ss, s) || overlap(so, s)) return SSM_ERR_ALIAS;
    if (overlap(ss, so)) return SSM_ERR_ALIAS;

    int sms = 0;
    if (ssm_status st = sm_count(&sms); st != SSM_OK) return st;

    ssm::UpdateArgs a{state, x, dt, A, B, C, D, z, dt_bias, out, batch, dim, (int)dstate,
                      dt_softplus ? 1 : 0};
    a.ngroups = ngroups;
    a.gch = dim / ngroups;
    return launch_status(ssm::launch_state_update(a, dtype == SSM_BF16 ? ssm::DType::BF16 : ssm::DType::F32, sms,
                                                  static_cast<cudaStream_t>(stream)));
}

ssm_status ssm_state_update(float* state, const void* x, const void* dt, const float* A,
                            const void* B, const void* C, const float* D, const void* z,
                            const float* dt_bias, void* out, int64_t batch, int64_t dim,
                            int64_t dstate, int dt_softplus, int dtype, void* stream) {
    return ssm_state_update_grouped(state, x, dt, A, B, C, D, z, dt_bias, out, batch, dim, dstate, 1, dt_softplus,
                                    dtype, stream);
}

}  // extern "C"
