// Per-device, thread-safe caches for launch set-up.
//
// CUDA applies a kernel's function attributes (its dynamic shared-memory
// limit, its cluster opt-in) to the current device only, and SM counts and
// occupancy differ between devices.  Each launcher therefore keeps such
// set-up in a PerDevice cache: one value per device ordinal, computed by the
// first caller on that device with the device current, read lock-free after
// that.  Host threads may launch concurrently.
#pragma once

#include <atomic>
#include <climits>
#include <mutex>

#include <cuda_runtime.h>

namespace qsa {

constexpr int kMaxDevices = 64;

class PerDevice {
 public:
  PerDevice() {
    for (auto &v : val_) v.store(kUnset, std::memory_order_relaxed);
  }

  // The cached value for the current device, computing it with init() on the
  // first call.  init() returns a value >= 0, or a negative value for a set-up
  // that failed; failures are not cached, so a later call tries again.
  template <typename F>
  int get(F &&init) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
      cudaGetLastError();
      return init();
    }
    int v = val_[dev].load(std::memory_order_acquire);
    if (v != kUnset) return v;
    std::lock_guard<std::mutex> lock(mu_);
    v = val_[dev].load(std::memory_order_relaxed);
    if (v == kUnset) {
      v = init();
      if (v >= 0) val_[dev].store(v, std::memory_order_release);
    }
    return v;
  }

 private:
  static constexpr int kUnset = INT_MIN;
  std::mutex mu_;
  std::atomic<int> val_[kMaxDevices];
};

// Sets a kernel's dynamic shared-memory limit once per device.  Returns
// cudaSuccess, or the error of the attempt (not cached).
template <typename K>
cudaError_t set_smem_once(PerDevice &cache, K kernel, size_t bytes) {
  const int r = cache.get([&]() -> int {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return -(int)e;
    }
    return 0;
  });
  return r >= 0 ? cudaSuccess : (cudaError_t)(-r);
}

// The current device's SM count (1 if the query fails).
inline int device_sm_count() {
  static PerDevice cache;
  const int n = cache.get([]() -> int {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      return -1;
    }
    return v;
  });
  return n > 0 ? n : 1;
}

}  // namespace qsa
