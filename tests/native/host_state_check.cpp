// Checks kd::PerDevice (sparse_teacher_kl_gb300/csrc/kd_host_state.h) from many host
// threads at once: each device's value is set up exactly once, a failed set-up is
// retried by the next call, other devices are unaffected, and ordinals outside the
// table are refused.  Prints "ok" and exits 0 on success.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "kd_host_state.h"

int main() {
  kd::PerDevice<int> table;
  constexpr int kDevices = 8, kThreads = 16, kRounds = 2000;
  std::atomic<int> inits[kDevices];
  for (auto& a : inits) a.store(0);
  std::atomic<int> failures_left{3};  // device 5 fails its first three set-ups
  std::atomic<int> bad{0};
  std::vector<std::thread> threads;
  for (int t = 0; t < kThreads; ++t) {
    threads.emplace_back([&, t] {
      for (int r = 0; r < kRounds; ++r) {
        const int dev = (t + r) % kDevices;
        int v = -1;
        const int rc = table.get(dev, &v, [&](int d, int* out) {
          if (d == 5 && failures_left.fetch_sub(1) > 0) return 7;
          inits[d].fetch_add(1);
          *out = 100 + d;
          return 0;
        });
        if (rc == 7 && dev == 5) continue;  // a failed set-up is reported, nothing stored
        if (rc != 0 || v != 100 + dev) bad.fetch_add(1);
      }
    });
  }
  for (auto& th : threads) th.join();
  for (int d = 0; d < kDevices; ++d)
    if (inits[d].load() != 1) {
      std::printf("device %d set up %d times\n", d, inits[d].load());
      return 1;
    }
  if (bad.load() != 0) {
    std::printf("%d wrong values\n", bad.load());
    return 1;
  }
  int v = 0;
  if (table.get(-1, &v, [](int, int*) { return 0; }) != -1 ||
      table.get(kd::kMaxDevices, &v, [](int, int*) { return 0; }) != -1) {
    std::printf("out-of-range ordinal accepted\n");
    return 1;
  }
  table.reset(3);
  int again = 0;
  table.get(3, &v, [&](int, int* out) { ++again; *out = 42; return 0; });
  if (again != 1 || v != 42) {
    std::printf("reset did not set up again\n");
    return 1;
  }
  std::printf("ok\n");
  return 0;
}
