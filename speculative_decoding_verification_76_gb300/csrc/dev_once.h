// Per-device, thread-safe one-time host setup (no CUDA types: the logic is
// compiled and exercised on its own by a host-only test).
//
// A kernel's attributes (its dynamic shared-memory limit) and a __device__
// symbol's address belong to one device's context, not to the process: a
// process that drives several GPUs, or several host threads that launch on
// one, must set them up per device and without racing.  PerDeviceOnce keeps,
// for each device ordinal, whether a setup step succeeded and the value it
// produced.  The fast path is one atomic load; the first call on a device
// runs the setup under a mutex, and a failed setup is retried on the next
// call instead of being remembered.
#pragma once
#include <atomic>
#include <mutex>
#include <stdint.h>

template <typename T = int, int kMaxDev = 64>
class PerDeviceOnce {
 public:
  static_assert(kMaxDev <= 64, "one bit per device in a 64-bit word");

  // Calls setup(&value) for device `dev` unless an earlier call for that
  // device succeeded; returns 0 and stores the device's value in *out on
  // success, the setup's nonzero code on failure, -1 for an ordinal outside
  // [0, kMaxDev).
  template <class F>
  int run(int dev, F&& setup, T* out = nullptr) {
    if (dev < 0 || dev >= kMaxDev) return -1;
    const uint64_t bit = uint64_t(1) << dev;
    if (done_.load(std::memory_order_acquire) & bit) {
      if (out) *out = value_[dev];
      return 0;
    }
    std::lock_guard<std::mutex> lock(mu_);
    if (!(done_.load(std::memory_order_relaxed) & bit)) {
      T v{};
      const int rc = setup(&v);
      if (rc != 0) return rc;
      value_[dev] = v;
      done_.fetch_or(bit, std::memory_order_release);
    }
    if (out) *out = value_[dev];
    return 0;
  }

  bool done(int dev) const {
    return dev >= 0 && dev < kMaxDev && (done_.load(std::memory_order_acquire) >> dev) & 1;
  }

 private:
  std::atomic<uint64_t> done_{0};
  std::mutex mu_;
  T value_[kMaxDev] = {};
};
