// selftest.cu — a kernel that waits on an mbarrier nothing ever completes,
// bounded by the caller's limit, to exercise the timeout path (status word
// set, kernel returns, context stays usable) without faulting or hanging.
#include "ra_internal.h"
#include "sm103.cuh"

namespace ra {
namespace {

__global__ void selftest_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtl ctl{status, &abort_flag, limit_ns};
  mbar_wait(smem_u32(&bar), 0, ctl, 99);  // nobody arrives: runs out after limit_ns
}

}  // namespace

cudaError_t launch_selftest_timeout(const Ctx& c, uint64_t* launches) {
  selftest_timeout_kernel<<<1, 32, 0, c.stream>>>(c.status, c.limit_ns);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace ra
