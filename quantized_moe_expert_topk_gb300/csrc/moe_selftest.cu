// moe_selftest.cu -- self-test of the failure detection: a bounded wait that
// is made to run out.  Every pipeline of this library waits on mbarriers with
// mbar_wait_bounded; on timeout the kernel records MOE_ERR_TIMEOUT in the
// device error word and returns instead of hanging.  This kernel waits, the
// same way, on a barrier that nothing completes, so that a test can check the
// timeout path and that the context stays usable afterwards.
#include "moe_common.cuh"
#include "moe_experts.h"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

__global__ void selftest_wait_kernel(int *err, long long limit_cycles) {
  __shared__ uint64_t bar;  // one arrival expected, none made
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, limit_cycles))
    record_device_error(err, MOE_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(int *err, long long limit_cycles, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit_cycles);
  return cudaGetLastError();
}

}  // namespace moe
