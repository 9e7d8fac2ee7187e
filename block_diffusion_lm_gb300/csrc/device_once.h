// Per-device, once-only host set-up (plain C++, no CUDA types).
//
// Kernel attributes such as the dynamic shared-memory limit belong to a
// device (its context), not to the process: a process that drives two GPUs
// must set them on each.  PerDeviceOnce runs a set-up step once for every
// device ordinal, under a lock, so host threads that race a first launch on
// the same device run it once and all see its result; a step that failed is
// retried on the next call.
#pragma once

#include <cstdint>
#include <mutex>

namespace csbp {

class PerDeviceOnce {
 public:
  static constexpr int kMaxDevices = 64;

  // Runs `setup(device)` (returning true on success) unless it already
  // succeeded for this device; returns whether the device is set up.  A
  // device ordinal outside [0, kMaxDevices) is refused (false).
  template <class F>
  bool run(int device, F&& setup) {
    if (device < 0 || device >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[device]) return true;
    if (!setup(device)) return false;
    done_[device] = true;
    return true;
  }

  bool done(int device) {
    if (device < 0 || device >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu_);
    return done_[device];
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

}  // namespace csbp
