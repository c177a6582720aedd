// Per-device record of a kernel attribute that the launcher sets once.
//
// cudaFuncSetAttribute (the dynamic shared-memory limit above 48 KB, the
// carveout preference) acts on the device that is current when it is
// called.  A record kept once per process would let a launch on a second
// device skip the call and then fail for want of shared memory; this keeps
// one record per device instead.  The header uses no CUDA types so that
// its logic can be checked on a machine without a GPU.
#pragma once

#include <atomic>

namespace dcn {

template <int kMaxDevices = 64>
class PerDeviceValue {
public:
    // Calls set() unless `value` is already recorded for `device`; records
    // `value` when set() returns 0.  A device index outside the table is
    // never recorded, so set() then runs on every call.  Concurrent calls
    // may both run set(), which is harmless: it sets the same value.
    template <typename Set>
    int ensure(int device, int value, Set &&set) {
        const bool kept = device >= 0 && device < kMaxDevices;
        if (kept && v_[device].load(std::memory_order_acquire) == value) return 0;
        const int e = static_cast<int>(set());
        if (e == 0 && kept) v_[device].store(value, std::memory_order_release);
        return e;
    }

private:
    std::atomic<int> v_[kMaxDevices] = {};
};

}  // namespace dcn
