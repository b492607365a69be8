// Self-test of the bounded waits every pipeline kernel uses: one CTA waits on an mbarrier that
// nothing ever arrives at.  The wait gives up when its polls run out, records its code in the
// device error flag and returns, so the kernel ends and the context stays usable.
#include "mi_internal.h"
#include "ptx.cuh"

namespace mi {

namespace {

__global__ void wait_timeout_selftest_kernel(int* err, uint32_t polls) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, DEV_TIMEOUT_SELFTEST, polls);
}

}  // namespace

cudaError_t wait_timeout_selftest_launch(int* err, unsigned long long limit_ns, cudaStream_t s) {
  // the same bounded wait as the pipelines, with as many polls as fit in limit_ns at the ~1.48 us
  // an unsuccessful poll takes
  const unsigned long long polls = limit_ns / 1476ull;
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err, (uint32_t)(polls > 0 ? (polls < kWaitPolls ? polls : kWaitPolls) : 1));
  return cudaGetLastError();
}

}  // namespace mi
