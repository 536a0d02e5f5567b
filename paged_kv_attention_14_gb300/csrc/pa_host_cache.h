// pa_host_cache.h -- host-side caches that keep per-call launch overhead low.
//
// Every entry point launches a kernel whose set-up does not change between
// calls with the same buffers: the kernel's dynamic shared-memory limit and
// occupancy (per device), and the TMA tensor maps of the caches (per cache
// pointer and shape).  Computing them on every call cost a few microseconds
// of host time per call; these caches compute each once.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

namespace pa {

// Sets the kernel's dynamic shared-memory limit on the current device (once
// per device and kernel) and returns its occupancy in CTAs per SM for the
// given block size and shared memory (0 on failure).
inline int prepare_kernel(const void *fn, int threads, size_t smem) {
  struct Entry {
    int dev;
    const void *fn;
    int threads;
    size_t smem;
    int occ;
  };
  static Entry entries[256];
  static int count = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < count; ++i)
    if (entries[i].dev == dev && entries[i].fn == fn && entries[i].threads == threads && entries[i].smem == smem)
      return entries[i].occ;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem) != cudaSuccess) return 0;
  if (occ > 0 && count < 256) entries[count++] = Entry{dev, fn, threads, smem, occ};
  return occ;
}

// A small per-thread cache of encoded tensor maps.  Key: the device, the
// base pointer and the caller's shape words; a hit copies the stored map.
struct MapKey {
  int dev;
  const void *base;
  int64_t words[8];
};

template <int N = 16>
struct MapCache {
  MapKey keys[N];
  CUtensorMap maps[N];
  int used = 0, next = 0;

  bool find(const MapKey &k, CUtensorMap *out) const {
    for (int i = 0; i < used; ++i)
      if (memcmp(&keys[i], &k, sizeof k) == 0) {
        *out = maps[i];
        return true;
      }
    return false;
  }
  void put(const MapKey &k, const CUtensorMap &m) {
    keys[next] = k;
    maps[next] = m;
    next = (next + 1) % N;
    if (used < N) ++used;
  }
};

inline MapKey map_key(const void *base, int64_t w0, int64_t w1, int64_t w2, int64_t w3, int64_t w4 = 0,
                      int64_t w5 = 0, int64_t w6 = 0, int64_t w7 = 0) {
  MapKey k;
  memset(&k, 0, sizeof k);
  cudaGetDevice(&k.dev);
  k.base = base;
  const int64_t w[8] = {w0, w1, w2, w3, w4, w5, w6, w7};
  memcpy(k.words, w, sizeof w);
  return k;
}

}  // namespace pa
