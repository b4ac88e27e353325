// The arrive-and-spin step of the library's grid barriers, written once over a
// small set of operations so that the device kernels and a host-thread test
// (tests/c/barrier_check.cc) run the same steps: publish this participant's
// writes, arrive, spin until every participant has arrived or the limit has
// passed, and on expiry raise the timeout and report failure instead of
// waiting on.  Plain C++: no CUDA headers needed.
//
// Ops provides:
//   fence()     order this participant's earlier writes before what follows
//   arrive()    add one to the barrier's counter (atomic)
//   count()     read the counter (acquire)
//   now()       a clock in nanoseconds
//   timeout()   record that a wait ran out (the device status bit)
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define DSA_PROTOCOL_FN __host__ __device__ __forceinline__
#else
#define DSA_PROTOCOL_FN inline
#endif

namespace dsa {

#if defined(__CUDACC__)
#pragma nv_exec_check_disable
#endif
template <class Ops>
DSA_PROTOCOL_FN bool barrier_arrive_and_wait(Ops& ops, uint32_t participants, uint64_t limit_ns) {
  ops.fence();
  ops.arrive();
  const uint64_t t0 = ops.now();
  while (ops.count() < participants) {
    if (ops.now() - t0 > limit_ns) {
      ops.timeout();
      return false;
    }
  }
  ops.fence();
  return true;
}

}  // namespace dsa
