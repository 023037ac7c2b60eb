// per_device.h -- once-per-device set-up flags for the launch wrappers.
//
// Kernel function attributes (the dynamic shared-memory limit of the tensor-core GEMM, the
// preferred shared-memory carveout) belong to the context of the device that is current
// when they are set.  A process that drives several GPUs must therefore set them once per
// device, not once per process.  PerDeviceOnce keeps one flag per device ordinal; run()
// calls the set-up function for a device until it has succeeded once there.  Host threads
// may call it concurrently: the flags are atomic, and a set-up that two threads run at the
// same time is idempotent (the same attribute set to the same value).
//
// No CUDA dependency: the device ordinal and the set-up are passed in, so the logic is
// testable on a machine without a GPU.
#pragma once

#include <atomic>
#include <cstdint>

namespace ctr {

constexpr int kMaxDevicesTracked = 64;

class PerDeviceOnce {
  public:
    // Runs setup() (returning an error code E, where `ok` means success) unless it already
    // succeeded on `device`.  Ordinals outside [0, kMaxDevicesTracked) are never cached:
    // their set-up runs on every call.
    template <typename E, typename F>
    E run(int device, E ok, F &&setup) {
        const bool tracked = device >= 0 && device < kMaxDevicesTracked;
        if (tracked && done_[device].load(std::memory_order_acquire)) return ok;
        const E e = setup();
        if (tracked && e == ok) done_[device].store(1, std::memory_order_release);
        return e;
    }

    bool done(int device) const {
        return device >= 0 && device < kMaxDevicesTracked &&
               done_[device].load(std::memory_order_acquire) != 0;
    }

  private:
    std::atomic<uint8_t> done_[kMaxDevicesTracked] = {};
};

}  // namespace ctr
