// Test hook for the failure detection of the bounded device-side waits.
//
// Every spin-wait of the library (an mbarrier wait inside a CTA) gives up
// after a device-time limit, records DEV_ERR_TIMEOUT in the ctx's status word
// and lets its kernel return; mkv_check_device reports it.  This kernel runs
// that same wait on an mbarrier no thread ever arrives on, so a test can make
// the limit run out without any fault, trap or hang.
#include "mkv_internal.cuh"
#include "ptx.cuh"

namespace mkv {

__global__ void __launch_bounds__(32) wait_test_kernel(int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    // phase 0 never completes: only the limit ends this wait
    if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(err, DEV_ERR_TIMEOUT);
  }
}

cudaError_t launch_wait_test(int* err, uint64_t limit_ns, cudaStream_t st) {
  wait_test_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace mkv
