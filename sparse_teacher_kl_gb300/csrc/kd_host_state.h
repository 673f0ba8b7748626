// Host-side state of the library that belongs to one device: kernel attributes,
// occupancy figures, SM counts.  Each value is set up once per device ordinal, on the
// first call made with that device current, and may be requested from several host
// threads at once.  Plain C++ (no CUDA types), so that its logic can be tested alone.
#pragma once

#include <atomic>
#include <mutex>

namespace kd {

constexpr int kMaxDevices = 64;

// One value of type T per device ordinal in [0, kMaxDevices).  get() returns 0 and the
// value, running `init(dev, &value)` first if that device has none yet; init returns 0
// on success, and anything else is passed back to the caller with nothing stored, so
// that a later call tries again.  Concurrent first calls for one device run init once:
// the others wait on the lock, then read the stored value.
template <class T>
class PerDevice {
 public:
  template <class F>
  int get(int dev, T* out, F&& init) {
    if (dev < 0 || dev >= kMaxDevices) return -1;
    if (ready_[dev].load(std::memory_order_acquire)) {
      *out = val_[dev];
      return 0;
    }
    std::lock_guard<std::mutex> lock(mu_);
    if (!ready_[dev].load(std::memory_order_relaxed)) {
      T v{};
      const int rc = init(dev, &v);
      if (rc != 0) return rc;
      val_[dev] = v;
      ready_[dev].store(true, std::memory_order_release);
    }
    *out = val_[dev];
    return 0;
  }

  // Forget the value of one device (the next get() sets it up again).
  void reset(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> lock(mu_);
    ready_[dev].store(false, std::memory_order_release);
  }

 private:
  std::mutex mu_;
  std::atomic<bool> ready_[kMaxDevices]{};
  T val_[kMaxDevices]{};
};

}  // namespace kd
