// eagle_selftest_wait: exercises the bounded waits every kernel of the step
// relies on, by waiting on a barrier that nothing completes.
//
// The step's kernels never trap and never spin forever: each mbarrier wait
// gives up after a wall-time limit, raises an abort flag, and the kernel
// reports EAGLE_ERR_TIMEOUT in the caller's status word before it drains its
// own copies and returns.  This kernel runs exactly those helpers (the
// CTA-local wait with its suspend hint, and the polling wait used for
// barriers that other CTAs of a cluster arrive on) on a freshly initialised
// barrier whose phase can never complete, with a short limit, and reports
// what they returned.  Nothing else is in flight: no copy, no MMA, no tensor
// memory.
#include "common.cuh"
#include "sm100.cuh"

namespace eagle {

using namespace sm100;

// One warp.  which = 0: the CTA-local wait (mbar_wait); 1: the cluster-scope
// polling wait (mbar_wait_cluster).  elapsed_ns (optional) receives the
// wall time the wait took before it gave up.
__global__ void __launch_bounds__(32) selftest_wait_kernel(uint64_t limit_ns, int which, int32_t *status,
                                                           uint64_t *elapsed_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none will come
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  const uint64_t t0 = globaltimer_ns();
  bool ok;
  if (which == 0) {
    ok = mbar_wait(&bar, 0, reinterpret_cast<volatile int *>(&abort_flag), limit_ns);
  } else {
    ok = mbar_wait_cluster(&bar, 0, limit_ns);
    if (!ok) abort_flag = 1;
  }
  const uint64_t t1 = globaltimer_ns();
  if (elapsed_ns) *elapsed_ns = t1 - t0;
  // a wait that gave up raised the abort flag: the kernels report that as
  // a timeout; a wait that succeeded would be a broken barrier
  if (!ok && abort_flag) report(status, EAGLE_ERR_TIMEOUT);
  else report(status, EAGLE_ERR_INVALID);
}

}  // namespace eagle

using namespace eagle;

extern "C" int eagle_selftest_wait(uint64_t limit_ns, int which, int32_t *status, uint64_t *elapsed_ns,
                                   eagle_stream_t stream) {
  if (!status || (which != 0 && which != 1)) return EAGLE_ERR_INVALID;
  if (limit_ns < 1000ull || limit_ns > 100000000ull) return EAGLE_ERR_INVALID;  // 1 us .. 100 ms
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, which, status, elapsed_ns);
  return cudaGetLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}
