// optin.h - per-device opt-in of a kernel's dynamic shared memory (host side,
// internal to libdec).
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace dec {

// A kernel's dynamic shared-memory limit is an attribute of the pair
// (function, device): setting it while one device is current leaves every
// other device at the default.  Each launcher keeps one SmemOptIn per kernel
// instantiation, recording per device the largest size set so far; ensure()
// raises the limit before a launch that needs more.  The raise happens under
// a lock, so two threads making their first launches at once never lower a
// limit the other has set.  Once a device is configured the check is one
// atomic load.  With nonportable_cluster the kernel may also be launched in
// clusters of more than 8 CTAs on that device.
class SmemOptIn {
 public:
  static constexpr int kMaxDevices = 64;

  template <typename F>
  cudaError_t ensure(F* fn, int bytes, bool nonportable_cluster = false) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (set_[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    std::lock_guard<std::mutex> guard(mu_);
    const int have = set_[dev].load(std::memory_order_relaxed);
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && nonportable_cluster && have == 0)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) set_[dev].store(bytes, std::memory_order_release);
    return e;
  }

 private:
  std::atomic<int> set_[kMaxDevices] = {};
  std::mutex mu_;
};

}  // namespace dec
