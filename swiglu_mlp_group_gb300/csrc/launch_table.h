// launch_table.h -- the per-device tables behind the launch bookkeeping of
// launch_util.cu, in plain C++ (no CUDA) so that their logic is tested on
// the host with made-up devices.
//
//  - OnceTable: "do this once per (device, key)" for settings that belong to
//    each device's copy of a kernel (the dynamic shared-memory opt-in): the
//    action runs under the table's lock, is recorded only when it succeeds,
//    and runs again when a larger value is asked for.
//  - ValueCache: a value computed once per (device, key) (occupancy).
// Both are fixed-size and thread-safe; when full they keep working without
// recording (the action / computation then runs on every call).
#pragma once

#include <mutex>

namespace ck {

template <typename Key, int kMax>
class OnceTable {
  public:
    // Runs apply() unless (device, key) was recorded with a value >= v.
    // Returns true when it was, or when apply() returned true (then (device,
    // key, v) is recorded); false when apply() failed.
    template <typename Apply>
    bool ensure(int device, const Key &key, int v, Apply &&apply) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < n_; ++i)
            if (e_[i].device == device && e_[i].key == key && e_[i].value >= v) return true;
        if (!apply()) return false;
        for (int i = 0; i < n_; ++i)
            if (e_[i].device == device && e_[i].key == key) {
                e_[i].value = v;
                return true;
            }
        if (n_ < kMax) e_[n_++] = Entry{device, key, v};
        return true;
    }
    int size() {
        std::lock_guard<std::mutex> lock(mu_);
        return n_;
    }

  private:
    struct Entry {
        int device;
        Key key;
        int value;
    };
    std::mutex mu_;
    Entry e_[kMax];
    int n_ = 0;
};

template <typename Key, typename Value, int kMax>
class ValueCache {
  public:
    // The value recorded for (device, key), else compute()'s, recorded when
    // ok(value) holds.
    template <typename Compute, typename Ok>
    Value get(int device, const Key &key, Compute &&compute, Ok &&ok) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < n_; ++i)
            if (e_[i].device == device && e_[i].key == key) return e_[i].value;
        const Value v = compute();
        if (ok(v) && n_ < kMax) e_[n_++] = Entry{device, key, v};
        return v;
    }
    int size() {
        std::lock_guard<std::mutex> lock(mu_);
        return n_;
    }

  private:
    struct Entry {
        int device;
        Key key;
        Value value;
    };
    std::mutex mu_;
    Entry e_[kMax];
    int n_ = 0;
};

}  // namespace ck
