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

// Clusters of C CTAs (threads each, smem bytes of dynamic shared memory)
// of `kern` that the current device can hold at once, from the runtime's
// occupancy query, cached per device and shape (the kernel's dynamic
// shared-memory opt-in must be set first).  0 on error.
struct ClusterOccupancy {
  static constexpr int kSlots = 256;
  std::atomic<uint64_t> entry[kMaxCachedDevices][kSlots];
  ClusterOccupancy() {
    for (auto& d : entry)
      for (auto& e : d) e.store(0);
  }
};

template <typename Kern>
int max_active_clusters(ClusterOccupancy& co, Kern kern, int C, int smem, int threads) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  // key: C (5 bits), smem / 16 (15 bits), threads / 32 (6 bits); value + 1 in 20 bits
  const uint64_t key = (uint64_t(C) << 21) | (uint64_t(smem / 16) << 6) | uint64_t(threads / 32);
  // open addressing: probe up to 16 slots from the key's hash
  const int h = static_cast<int>((key * 0x9E3779B97F4A7C15ull) >> 56);
  if (dev < kMaxCachedDevices) {
    for (int i = 0; i < 16; ++i) {
      const uint64_t v = co.entry[dev][(h + i) & (ClusterOccupancy::kSlots - 1)].load(
          std::memory_order_acquire);
      if (v == 0) break;
      if ((v >> 20) == key) return int(v & 0xfffff) - 1;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (n > 0xffffe) n = 0xffffe;
  if (dev < kMaxCachedDevices) {
    for (int i = 0; i < 16; ++i) {  // first free slot (racing writers may store it twice)
      uint64_t expect = 0;
      if (co.entry[dev][(h + i) & (ClusterOccupancy::kSlots - 1)].compare_exchange_strong(
              expect, (key << 20) | uint64_t(n + 1)))
        break;
    }
  }
  return n;
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
