// Self-check of the bounded device wait that every tcgen05 kernel of this
// library uses (mbar_wait_budget in common.cuh): one CTA waits on an mbarrier
// phase that nothing completes, so the wait must give up, either when its
// %globaltimer budget runs out or when a peer warp raises the CTA's abort
// flag, set MC_STATUS_TIMEOUT and return, leaving the context usable.  Every
// loop here is bounded by %globaltimer.
#include "common.cuh"
#include "kernels.h"

namespace mc {

namespace {

__global__ void wait_selftest_kernel(unsigned long long budget_ns, unsigned long long abort_after_ns,
                                     int32_t* status, unsigned long long* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);          // one arrival completes phase 0; none comes
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    const bool ok = mbar_wait_budget(&bar, 0, &abort_flag, budget_ns);
    const unsigned long long t1 = globaltimer_ns();
    if (!ok) set_status(status, MC_STATUS_TIMEOUT);
    if (waited_ns) *waited_ns = t1 - t0;
    abort_flag = 1;              // the other warp stops waiting too
  } else if (threadIdx.x == 32 && abort_after_ns) {
    const unsigned long long t0 = globaltimer_ns();
    while (!abort_flag && globaltimer_ns() - t0 < abort_after_ns) {
    }
    abort_flag = 1;
  }
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long budget_ns, unsigned long long abort_after_ns,
                                 int32_t* status, unsigned long long* waited_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 64, 0, s>>>(budget_ns, abort_after_ns, status, waited_ns);
  return cudaGetLastError();
}

}  // namespace mc
