// Per-device, thread-safe raising of a kernel's dynamic shared-memory limit.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

namespace pkv {

// Sets cudaFuncAttributeMaxDynamicSharedMemorySize of `kernel` to `bytes` on
// the current device, once per device: `done` (one per kernel) holds a bit
// for each device 0..63 already set (devices above 63 are set every call).
// Two threads making their first call at the same time may both set it,
// which is harmless.
template <class Kernel>
cudaError_t set_smem_limit_once(std::atomic<unsigned long long>& done, Kernel kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit) != 0ull) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (bit != 0ull) done.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

}  // namespace pkv
