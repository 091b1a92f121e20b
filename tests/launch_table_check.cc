// Host-only check of the per-device launch tables (launch_table.h), driven by
// made-up devices and a fake attribute setter: a setting is applied once per
// (device, kernel), again for a larger value or after a failure, exactly once
// under racing threads, and a full table keeps applying without recording.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "launch_table.h"

static int fails = 0;
#define CHECK(c)                                                  \
    do {                                                          \
        if (!(c)) {                                               \
            std::printf("FAIL line %d: %s\n", __LINE__, #c);      \
            ++fails;                                              \
        }                                                         \
    } while (0)

int main() {
    static int kernel_a, kernel_b;
    const void *A = &kernel_a, *B = &kernel_b;
    {
        ck::OnceTable<const void *, 16> t;
        int calls = 0;
        auto set = [&] { ++calls; return true; };
        CHECK(t.ensure(0, A, 1000, set) && calls == 1);
        CHECK(t.ensure(0, A, 1000, set) && calls == 1);   // done on device 0
        CHECK(t.ensure(1, A, 1000, set) && calls == 2);   // device 1 has its own copy
        CHECK(t.ensure(1, A, 800, set) && calls == 2);
        CHECK(t.ensure(0, A, 2000, set) && calls == 3);   // a larger opt-in
        CHECK(t.ensure(0, A, 1500, set) && calls == 3);
        CHECK(t.ensure(0, B, 1000, set) && calls == 4);
        CHECK(t.size() == 3);
        int tries = 0;
        auto fail = [&] { ++tries; return false; };
        CHECK(!t.ensure(2, A, 1000, fail) && tries == 1);  // a failure is not recorded
        CHECK(!t.ensure(2, A, 1000, fail) && tries == 2);
        CHECK(t.ensure(2, A, 1000, set) && calls == 5);
        CHECK(t.size() == 4);
    }
    {
        // racing threads on four devices and two kernels: exactly one call each
        ck::OnceTable<const void *, 64> t;
        std::atomic<int> calls[4][2] = {};
        std::vector<std::thread> th;
        for (int w = 0; w < 8; ++w)
            th.emplace_back([&, w] {
                for (int i = 0; i < 2000; ++i) {
                    const int dev = (i + w) % 4, k = (i / 4 + w) % 2;
                    t.ensure(dev, k ? B : A, 4096, [&] { calls[dev][k]++; return true; });
                }
            });
        for (auto &x : th) x.join();
        for (int d = 0; d < 4; ++d)
            for (int k = 0; k < 2; ++k) CHECK(calls[d][k].load() == 1);
        CHECK(t.size() == 8);
    }
    {
        // a full table keeps applying (and succeeding) without recording
        ck::OnceTable<const void *, 1> t;
        int calls = 0;
        auto set = [&] { ++calls; return true; };
        CHECK(t.ensure(0, A, 1, set) && t.ensure(1, A, 1, set) && t.ensure(1, A, 1, set));
        CHECK(calls == 3 && t.size() == 1);
    }
    {
        ck::ValueCache<int, int, 8> c;
        int computed = 0;
        auto ok = [](int v) { return v > 0; };
        CHECK(c.get(0, 7, [&] { ++computed; return 3; }, ok) == 3);
        CHECK(c.get(0, 7, [&] { ++computed; return 5; }, ok) == 3 && computed == 1);
        CHECK(c.get(1, 7, [&] { ++computed; return 5; }, ok) == 5 && computed == 2);
        CHECK(c.get(2, 7, [&] { ++computed; return 0; }, ok) == 0);  // not recorded
        CHECK(c.get(2, 7, [&] { ++computed; return 4; }, ok) == 4 && computed == 4);
        CHECK(c.size() == 3);
    }
    if (fails == 0) std::printf("ok\n");
    return fails == 0 ? 0 : 1;
}
