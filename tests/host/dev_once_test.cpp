// Host-only test of PerDeviceOnce (the per-device, thread-safe setup record
// the library uses for kernel attributes and symbol addresses).  Built with
// g++ by tests/test_host_logic.py; prints "ok" and exits 0 on success.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>

#include "dev_once.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::fprintf(stderr, "check failed line %d: %s\n", __LINE__, #c); \
      return 1;                                               \
    }                                                         \
  } while (0)

int main() {
  // one setup per device, whatever the number of callers and threads
  PerDeviceOnce<int> once;
  std::atomic<int> calls[8];
  for (auto& c : calls) c = 0;
  std::vector<std::thread> th;
  for (int t = 0; t < 16; ++t)
    th.emplace_back([&, t] {
      for (int i = 0; i < 1000; ++i) {
        const int dev = (t + i) % 8;
        int v = -1;
        const int rc = once.run(dev, [&](int* out) { calls[dev]++; *out = 100 + dev; return 0; }, &v);
        if (rc != 0 || v != 100 + dev) std::abort();
      }
    });
  for (auto& x : th) x.join();
  for (int d = 0; d < 8; ++d) CHECK(calls[d].load() == 1);
  for (int d = 0; d < 8; ++d) CHECK(once.done(d));
  CHECK(!once.done(8));

  // a failed setup is not remembered: the next call retries it
  PerDeviceOnce<void*> addr;
  int tries = 0;
  void* p = nullptr;
  CHECK(addr.run(3, [&](void** o) { ++tries; return 7; }, &p) == 7);
  CHECK(!addr.done(3));
  static int target;
  CHECK(addr.run(3, [&](void** o) { ++tries; *o = &target; return 0; }, &p) == 0);
  CHECK(p == &target && tries == 2 && addr.done(3));
  CHECK(addr.run(3, [&](void** o) { ++tries; return 9; }, &p) == 0);  // cached: not rerun
  CHECK(p == &target && tries == 2);
  // another device keeps its own value
  static int other;
  CHECK(addr.run(5, [&](void** o) { *o = &other; return 0; }, &p) == 0 && p == &other);
  CHECK(addr.run(3, [&](void** o) { return 1; }, &p) == 0 && p == &target);

  // ordinals outside the record are refused, not aliased onto another device
  CHECK(addr.run(-1, [&](void** o) { return 0; }, &p) == -1);
  CHECK(addr.run(64, [&](void** o) { return 0; }, &p) == -1);
  std::printf("ok\n");
  return 0;
}
