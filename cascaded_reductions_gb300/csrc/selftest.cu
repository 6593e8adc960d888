// Self-tests of the on-device checks: the bounded waits the tensor-core
// kernels use, and (bounds-checked build) the index checks of every kernel.
//
// One thread waits on a shared-memory mbarrier that nothing ever arrives on,
// through the same tc::mbar_wait every pipeline wait in this library uses.
// The wait gives up after its limit (kWaitLimitNs), sets the CTA's abort
// flag, records RF_ERR_TIMEOUT in this translation unit's status word and
// the kernel returns normally: no fault, no trap, no hang, and the context
// stays usable.  The host reads the status through rf_device_error.

#include "tc_common.cuh"

namespace rf {
namespace {

__global__ void wait_timeout_kernel(int* __restrict__ waited_ms) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long t0 = tc::globaltimer_ns();
    const bool completed = tc::mbar_wait(&bar, 0, &abort_flag);   // nothing arrives
    const unsigned long long dt = tc::globaltimer_ns() - t0;
    *waited_ms = completed ? -1 : (int)(dt / 1000000ull);
  }
}

#ifdef RF_CHECK_BOUNDS
__device__ int g_selftest_sink[1];

// Presents the index n to the check of an n-element buffer: one past the
// end, so the check refuses it and records RF_ERR_BOUNDS.  The store it
// guards targets element 0, a valid address, so nothing faults even if the
// check were wrong.
__global__ void bounds_selftest_kernel(int n) {
  if (RF_IDX_OK(n, n)) g_selftest_sink[0] = 1;
}
#endif

}  // namespace

#ifdef RF_CHECK_BOUNDS
rf_status launch_selftest_bounds(cudaStream_t st) {
  bounds_selftest_kernel<<<1, 1, 0, st>>>(1);
  return launch_status();
}
#endif

rf_status launch_selftest_wait_timeout(int* waited_ms, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(waited_ms);
  return launch_status();
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
