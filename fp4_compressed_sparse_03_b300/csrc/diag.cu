// Diagnostic for the failure-detection contract: one warp waits, through the same bounded
// mbarrier wait that every TMA- or tcgen05-fed kernel of this library uses, on a barrier
// phase that completes only if the caller asks for the arrival.  Without it the wait runs
// out after `limit` polls, raises CSA2_DEV_TIMEOUT in *dev_status and the kernel returns:
// nothing is in flight (no copy, no MMA, no TMEM), so the context stays usable.
#include "async.cuh"

namespace csa2 {

__global__ void __launch_bounds__(32, 1)
    bounded_wait_kernel(int arrive, uint32_t limit, int32_t* st) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort;
  if (threadIdx.x == 0) {
    abort = 0;
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncwarp();
  if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
  // Every lane polls; the first to give up raises `abort`, the rest see it within 1024
  // polls (or expire themselves).  The status bit is OR-ed, so repeats are harmless.
  (void)mbar_wait(&abort, &bar, 0, st, limit);
}

cudaError_t launch_bounded_wait(int arrive, uint32_t limit, int32_t* st, cudaStream_t s) {
  bounded_wait_kernel<<<1, 32, 0, s>>>(arrive, limit, st);
  return cudaGetLastError();
}

}  // namespace csa2
