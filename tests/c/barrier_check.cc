// The grid-barrier protocol of libdsa (barrier_protocol.h, the same template
// the top-k kernel instantiates with device atomics) run by host threads on
// std::atomic: every participant passes when all arrive; when one participant
// never arrives, every other one gives up after the limit, records the
// timeout and reports failure instead of waiting on.  Exits non-zero on the
// first failed check.
#include <atomic>
#include <chrono>
#include <cstdio>
#include <thread>
#include <vector>

#include "barrier_protocol.h"

namespace {

struct HostOps {
  std::atomic<uint32_t>* counter;
  std::atomic<uint32_t>* status;
  void fence() { std::atomic_thread_fence(std::memory_order_seq_cst); }
  void arrive() { counter->fetch_add(1u, std::memory_order_relaxed); }
  uint32_t count() { return counter->load(std::memory_order_acquire); }
  uint64_t now() {
    return (uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(
               std::chrono::steady_clock::now().time_since_epoch())
        .count();
  }
  void timeout() { status->fetch_or(1u); }
};

// Runs n participants; participant `skip` (or none, if -1) never arrives.
// Returns the number that passed; *status gets the timeout bit; *ms the
// longest wait.
int run(int n, int skip, uint64_t limit_ns, uint32_t* status, double* ms) {
  std::atomic<uint32_t> counter{0}, st{0};
  std::vector<int> passed(n, 0);
  std::vector<double> waited(n, 0.0);
  std::vector<std::thread> th;
  for (int i = 0; i < n; ++i) {
    th.emplace_back([&, i] {
      if (i == skip) return;
      HostOps ops{&counter, &st};
      const auto t0 = std::chrono::steady_clock::now();
      passed[i] = dsa::barrier_arrive_and_wait(ops, (uint32_t)n, limit_ns) ? 1 : 0;
      waited[i] = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    });
  }
  for (auto& t : th) t.join();
  int np = 0;
  *ms = 0.0;
  for (int i = 0; i < n; ++i) {
    np += passed[i];
    if (waited[i] > *ms) *ms = waited[i];
  }
  *status = st.load();
  return np;
}

#define CHECK(cond, what)          \
  do {                             \
    if (!(cond)) {                 \
      std::printf("FAIL %s\n", what); \
      return 1;                    \
    }                              \
    std::printf("ok %s\n", what);  \
  } while (0)

}  // namespace

int main() {
  uint32_t status = 0;
  double ms = 0.0;
  const uint64_t limit = 20ull * 1000 * 1000;   // 20 ms
  for (int rep = 0; rep < 20; ++rep) {
    const int np = run(8, -1, 5ull * 1000 * 1000 * 1000, &status, &ms);
    if (np != 8 || status != 0) {
      std::printf("FAIL all arrive (rep %d: %d passed, status %u)\n", rep, np, status);
      return 1;
    }
  }
  std::printf("ok all arrive: every participant passes, no timeout (20 reps)\n");
  const int np = run(8, 3, limit, &status, &ms);
  CHECK(np == 0, "one arrival dropped: no participant passes");
  CHECK(status == 1u, "one arrival dropped: the timeout is recorded");
  CHECK(ms >= 20.0 && ms < 2000.0, "one arrival dropped: each wait ends at the limit");
  std::printf("all ok\n");
  return 0;
}
