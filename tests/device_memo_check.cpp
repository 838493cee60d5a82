// Host check of the per-device memo that the library's launchers use to set
// kernel attributes once per GPU (compiled and run by test_device_memo.py).
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "device_memo.h"

static int failures = 0;
#define CHECK(c)                                                  \
    do {                                                          \
        if (!(c)) {                                               \
            std::printf("FAILED line %d: %s\n", __LINE__, #c);    \
            ++failures;                                           \
        }                                                         \
    } while (0)

int main() {
    static ssm::DeviceMemo memo;   // static storage: zero-initialised like the library's
    int calls[ssm::kMemoDevices] = {};
    auto compute_for = [&](int dev) {
        return [&, dev](int& r) {
            ++calls[dev];
            r = 100 + dev;
            return true;
        };
    };
    int out = 0;
    // each device computes once, independently of the others
    CHECK(!memo.known(0) && !memo.known(1));
    CHECK(memo.get(0, compute_for(0), &out) && out == 100);
    CHECK(memo.known(0) && !memo.known(1));
    CHECK(memo.get(0, compute_for(0), &out) && out == 100 && calls[0] == 1);
    CHECK(memo.get(1, compute_for(1), &out) && out == 101 && calls[1] == 1);
    CHECK(memo.get(1, compute_for(1), &out) && calls[1] == 1 && calls[0] == 1);
    // a failed computation is not memoised: the next call tries again
    int tries = 0;
    auto failing = [&](int& r) {
        ++tries;
        r = 7;
        return false;
    };
    CHECK(!memo.get(2, failing, &out) && !memo.known(2));
    CHECK(!memo.get(2, failing, &out) && tries == 2);
    auto zero = [&](int& r) {
        r = 0;
        return true;
    };
    CHECK(!memo.get(3, zero, &out) && !memo.known(3));   // zero is "not computed"
    CHECK(memo.get(2, compute_for(2), &out) && out == 102 && memo.known(2));
    // ordinals outside the table are served, not memoised; negative ones refused
    int far = 0;
    auto far_compute = [&](int& r) {
        ++far;
        r = 5;
        return true;
    };
    CHECK(memo.get(ssm::kMemoDevices, far_compute, &out) && out == 5);
    CHECK(memo.get(ssm::kMemoDevices, far_compute, &out) && far == 2);
    CHECK(!memo.get(-1, far_compute, &out) && far == 2);
    // concurrent first calls from many threads on several devices: every call
    // returns that device's value and the memo ends up set for each
    static ssm::DeviceMemo shared;
    std::atomic<int> computed[4] = {};
    std::atomic<int> wrong{0};
    std::vector<std::thread> threads;
    for (int t = 0; t < 16; ++t)
        threads.emplace_back([&, t] {
            for (int i = 0; i < 1000; ++i) {
                const int dev = (t + i) % 4;
                int v = 0;
                const bool ok = shared.get(dev, [&, dev](int& r) {
                    computed[dev].fetch_add(1);
                    r = 10 + dev;
                    return true;
                }, &v);
                if (!ok || v != 10 + dev) wrong.fetch_add(1);
            }
        });
    for (auto& th : threads) th.join();
    CHECK(wrong.load() == 0);
    for (int d = 0; d < 4; ++d) CHECK(shared.known(d) && computed[d].load() >= 1);
    std::printf("%s\n", failures ? "device memo check FAILED" : "device memo check passed");
    return failures ? 1 : 0;
}
