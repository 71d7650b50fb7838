// Self-test of the bounded waits the copy pipelines of this library use on their mbarriers.
#include "common.cuh"

namespace ssmtree {
namespace {

// One thread arms an mbarrier for one arrival that never comes and waits on it with the
// library's bounded wait (limit_ns of global time).  When the wait gives up it reports
// SSM_STATUS_TIMEOUT, as the kernels' copy pipelines do, and the kernel returns: the
// context stays usable.
__global__ void selftest_wait_kernel(int32_t* status, unsigned long long limit_ns) {
  __shared__ unsigned long long bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  if (!mbar_wait_ns(b, 0, limit_ns)) flag(status, SSM_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t* status, unsigned long long limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace ssmtree
