// Per-device memo of a host-side query (an SM count, an occupancy figure):
// one slot per device ordinal, lock-free.  Threads that race on a first
// lookup all compute the same value and store it; readers see either 0
// ("not known yet") or that value, never a torn one.  Ordinals beyond the
// table are simply not memoised.
#pragma once

#include <atomic>
#include <stdint.h>

namespace pkvd {

constexpr int kMaxDevicesCached = 64;

template <typename V>
struct PerDeviceMemo {
  std::atomic<V> slot[kMaxDevicesCached] = {};

  // value for `dev` (0 when not yet known or out of range)
  V get(int dev) const {
    return (dev >= 0 && dev < kMaxDevicesCached) ? slot[dev].load(std::memory_order_acquire) : V(0);
  }
  void put(int dev, V v) {
    if (dev >= 0 && dev < kMaxDevicesCached) slot[dev].store(v, std::memory_order_release);
  }
};

}  // namespace pkvd
