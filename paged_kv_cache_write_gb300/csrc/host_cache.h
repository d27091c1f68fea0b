// Host-side cache of per-kernel launch set-up (dynamic shared-memory opt-in
// and occupancy), so repeated calls do not repeat driver queries.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

namespace pkv {

constexpr int kMaxCachedDevices = 16;

// One per kernel instantiation: per device, the last (smem, threads) set
// up and the resulting CTAs per SM, packed in one word so readers never see
// a torn entry.
struct KernelSetup {
  std::atomic<uint64_t> entry[kMaxCachedDevices];
  KernelSetup() {
    for (auto& e : entry) e.store(0);
  }
};

// Opt `kern` into `smem` bytes of dynamic shared memory on the current
// device and report its resident CTAs per SM for `threads` threads
// (per_sm may be null).  Driver calls happen once per device and size.
template <typename Kern>
cudaError_t kernel_setup(KernelSetup& ks, Kern kern, int smem, int threads, int* per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t key = (uint64_t(uint32_t(smem)) << 24) | (uint64_t(uint32_t(threads)) << 8);
  if (dev < kMaxCachedDevices) {
    const uint64_t v = ks.entry[dev].load(std::memory_order_acquire);
    if (v != 0 && (v & ~uint64_t(0xff)) == key) {
      if (per_sm) *per_sm = int(v & 0xff) - 1;
      return cudaSuccess;
    }
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
  if (e != cudaSuccess) return e;
  if (occ > 254) occ = 254;
  if (per_sm) *per_sm = occ;
  if (dev < kMaxCachedDevices) ks.entry[dev].store(key | uint64_t(occ + 1), std::memory_order_release);
  return cudaSuccess;
}

// SMs of the current device, looked up once per device (devices past
// kMaxCachedDevices are asked every time).  Entries are atomics, so threads
// calling on different devices neither race nor see each other's count.
inline int sm_count() {
  static std::atomic<int> cached[kMaxCachedDevices];  // static storage: starts at 0
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  const bool keep = dev >= 0 && dev < kMaxCachedDevices;
  if (keep) {
    const int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 0;
  }
  if (sms <= 0) sms = 1;
  if (keep) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

}  // namespace pkv
