// The library's bounded wait exercised on its own: one thread waits on an
// mbarrier phase that nothing completes. The wait gives up after the library's
// limit (kWaitLimitNs), ORs the timeout bit into the device error word and the
// kernel returns, touching nothing else. Every pipelined kernel waits through
// the same mbar_wait; this is how a test makes a wait run out without faulting
// or hanging the GPU.
#include "launch.h"
#include "pipeline.cuh"

namespace qkvp {

__global__ void qkvp_wait_selftest_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_init_fence();
  mbar_wait(&bar, 0, err);  // phase 0 never completes: nothing arrives on the barrier
}

const void* wait_selftest_kernel() { return reinterpret_cast<const void*>(&qkvp_wait_selftest_kernel); }

}  // namespace qkvp
