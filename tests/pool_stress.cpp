// Stress test of the host worker pool (built by tests/test_lib_host.py with
// -fsanitize=thread): two threads issue thousands of short parallel_for calls
// on one shared pool, so a worker that still touches a caller's completion
// latch after the caller has returned shows up as a data race.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <functional>
#include <string>
#include <thread>

#include "mt_host.h"

int main() {
  mth::Pool pool;
  pool.start(8);
  std::atomic<long> total{0};
  auto work = [&](int seed) {
    for (int it = 0; it < 3000; ++it) {
      std::function<void(int64_t)> fn = [&](int64_t i) { total.fetch_add(i + seed, std::memory_order_relaxed); };
      std::string err;
      if (!pool.parallel_for(1 + (it % 5), fn, &err)) {
        std::printf("error %s\n", err.c_str());
        std::abort();
      }
    }
  };
  std::thread a(work, 1), b(work, 2);
  a.join();
  b.join();
  pool.stop();
  // sum over it of sum_{i < 1 + it % 5} (i + seed), for seed 1 and 2
  long expect = 0;
  for (int it = 0; it < 3000; ++it)
    for (int i = 0; i < 1 + it % 5; ++i) expect += 2 * i + 3;
  std::printf("%s %ld\n", total.load() == expect ? "ok" : "wrong", total.load());
  return total.load() == expect ? 0 : 1;
}
