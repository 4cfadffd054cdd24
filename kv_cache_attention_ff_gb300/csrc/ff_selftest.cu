// Self-test of the bounded device waits: one CTA waits on an mbarrier that
// nothing completes, gives up after `limit_ns`, and reports through the same
// error word the library's kernels use.  No fault, no trap: the context stays
// usable and the host reads FF_ERR_DEVICE_TIMEOUT from ff_bank_error_poll.
#include "ff_internal.h"
#include "ff_ptx.cuh"

namespace ff {

__global__ void wait_probe_kernel(unsigned int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, &abort_flag, err, limit_ns);  // never completes: times out
  __syncthreads();
}

cudaError_t launch_wait_probe(unsigned int* err, unsigned long long limit_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace ff
