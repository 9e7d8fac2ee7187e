// Exercises csbp::PerDeviceOnce, the once-per-device host set-up used by the
// attention launchers, with a stand-in set-up step (no CUDA): the step runs
// once per device ordinal, a failed step is retried, out-of-range ordinals
// are refused, and threads racing the first call on one device run it once.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "device_once.h"

int main() {
  csbp::PerDeviceOnce once;
  std::atomic<int> calls[4] = {};
  auto setup = [&](int dev) {
    calls[dev].fetch_add(1);
    return true;
  };
  // device 0 twice, device 1 once: two set-ups, one each
  bool a = once.run(0, setup), b = once.run(0, setup), c = once.run(1, setup);
  std::printf("first %d %d %d calls %d %d done2 %d\n", a, b, c, calls[0].load(), calls[1].load(),
              once.done(2));
  // a failing step leaves the device unconfigured and is retried
  int tries = 0;
  bool f1 = once.run(2, [&](int) { ++tries; return false; });
  bool f2 = once.run(2, [&](int) { ++tries; return true; });
  bool f3 = once.run(2, [&](int) { ++tries; return true; });
  std::printf("retry %d %d %d tries %d\n", f1, f2, f3, tries);
  // ordinals outside the table are refused without running the step
  int outside = 0;
  bool o1 = once.run(-1, [&](int) { ++outside; return true; });
  bool o2 = once.run(csbp::PerDeviceOnce::kMaxDevices, [&](int) { ++outside; return true; });
  std::printf("outside %d %d runs %d\n", o1, o2, outside);
  // 16 threads race the first call on device 3
  std::vector<std::thread> ts;
  std::atomic<int> ok{0};
  for (int i = 0; i < 16; ++i)
    ts.emplace_back([&] {
      if (once.run(3, setup)) ok.fetch_add(1);
    });
  for (auto& t : ts) t.join();
  std::printf("race calls %d ok %d\n", calls[3].load(), ok.load());
  return 0;
}
