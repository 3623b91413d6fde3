// vn_smem.h -- opting a kernel into more than 48 KB of dynamic shared memory.
//
// cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, n)
// acts on the kernel's copy for the current device, so a process that launches
// on several devices has to opt in on each of them. A launcher keeps one record
// per kernel with, per device, the largest size already set. The attribute is
// set under a lock and only ever raised, so a thread can never lower it below
// the size another thread has just checked for.
//
// Host-only code with no device code in it: the CPU tests compile this header
// with the host compiler against stand-ins for the two runtime calls it makes.
#pragma once

#include <atomic>
#include <cstddef>
#include <mutex>

#include <cuda_runtime_api.h>

namespace vn {

constexpr int kMaxDevices = 64;

// Per device, the largest dynamic shared-memory size set so far for one kernel
// (static storage: zero until the first opt-in).
using SmemRecord = std::atomic<size_t>[kMaxDevices];

inline std::mutex& smem_optin_mutex() {
  static std::mutex m;
  return m;
}

// Make `fn` launchable with `smem` bytes of dynamic shared memory on the current
// device; a no-op once a size at least as large has been set there.
inline cudaError_t ensure_dynamic_smem(const void* fn, size_t smem, SmemRecord& done) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire) >= smem) return cudaSuccess;
  std::lock_guard<std::mutex> lock(smem_optin_mutex());
  if (done[dev].load(std::memory_order_relaxed) >= smem) return cudaSuccess;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err == cudaSuccess) done[dev].store(smem, std::memory_order_release);
  return err;
}

}  // namespace vn
