// noalloc.cu -- ssm_scan_fwd_noalloc: the full-sequence scan for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the scan:
// code inside a framework whose allocator owns all device memory, code that
// runs where allocation is forbidden or would synchronise (an allocation-free
// hot loop), or plain C callers with no allocator of their own to hand a
// workspace from.  ssm_scan_fwd needs a caller-provided workspace for its
// fast path; this entry point instead uses a fixed scratch array that lives
// in the library itself, so it allocates nothing.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes
// (32 MiB).  Every GPU that loads the library holds it until the process
// exits.  In host code the array's name is only a host-side stand-in, so its
// device address is looked up once per device with cudaGetSymbolAddress
// (with that device current) and passed to the kernels.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/ssm_scan.h"
#include "ssm_internal.cuh"

namespace {

constexpr int64_t kNoAllocScratchBytes = int64_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device: looked up on
// the first call for that device, then cached.
ssm_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSM_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSM_ERR_DEVICE;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SSM_OK;
}

}  // namespace

extern "C" {

int64_t ssm_scan_noalloc_max_workspace_bytes(void) { return kNoAllocScratchBytes; }

ssm_status ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z, const float* delta_bias,
                                int softplus_flag, void* out, float* last_state, int64_t batch,
                                int64_t dim, int64_t seqlen, int64_t dstate, int dtype, void* stream) {
    // the scan's own checks first (dtype, pointers, sizes, alignment,
    // aliasing), so an invalid call gets the code ssm_scan_fwd would return;
    // only a valid call can be refused for its size
    if (const int chk = ssm::check_scan_call(u, delta, A, B, C, D, z, delta_bias, nullptr, out, last_state, batch,
                                             dim, seqlen, dstate, 1, dtype, nullptr, 0);
        chk != SSM_OK)
        return static_cast<ssm_status>(chk);
    const int64_t need = ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, dtype);
    if (need < 0) return SSM_ERR_SHAPE;
    if (need > kNoAllocScratchBytes) return SSM_ERR_SCRATCH;
    void* scratch = nullptr;
    if (ssm_status st = scratch_for_current_device(&scratch); st != SSM_OK) return st;
    return ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, out, last_state, batch, dim, seqlen,
                        dstate, dtype, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
