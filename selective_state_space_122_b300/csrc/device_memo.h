// device_memo.h -- a per-device, thread-safe memo for values a host entry
// point computes once per GPU: the launch attributes of a kernel are set with
// cudaFuncSetAttribute, which acts on the calling thread's current device, so
// "already set" is a fact about one device, not about the process.  Plain
// C++ (no CUDA types), so the bookkeeping is tested on the host.
#pragma once

#include <atomic>

namespace ssm {

constexpr int kMemoDevices = 64;

// One value per device ordinal; 0 means "not computed yet", so a memoised
// value must be nonzero.  Static instances are zero-initialised before any
// thread can reach them.
struct DeviceMemo {
    std::atomic<int> v[kMemoDevices];

    // The value for device `dev`: the memoised one, or compute(r) -> bool
    // run now (with `dev` current) and memoised when it succeeds with r != 0.
    // Concurrent first calls for one device may each run compute, so it must
    // be idempotent (setting a kernel attribute is).  Devices beyond the table
    // are served without memoising.  Returns false if compute failed.
    template <typename F>
    bool get(int dev, F&& compute, int* out) {
        if (dev < 0) return false;
        if (dev < kMemoDevices) {
            const int c = v[dev].load(std::memory_order_acquire);
            if (c != 0) {
                *out = c;
                return true;
            }
        }
        int r = 0;
        if (!compute(r) || r == 0) return false;
        if (dev < kMemoDevices) v[dev].store(r, std::memory_order_release);
        *out = r;
        return true;
    }

    bool known(int dev) const { return dev >= 0 && dev < kMemoDevices && v[dev].load(std::memory_order_acquire) != 0; }
};

}  // namespace ssm
