// Self-tests: the bounded waits the copy pipelines of this library use on their mbarriers,
// and the three SiLU forms the kernels evaluate.
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

// The SiLU forms of the kernels on n given inputs: out[0][i] the FMA-pipe form (polynomial
// 2^t, Newton reciprocal; the main verify kernel's x conv), out[1][i] the special-function
// intrinsic form (the B | C conv of the prep kernels), out[2][i] v / (1 + expf(-v)) with a
// rounded divide (commit, draft step).
__global__ void selftest_silu_kernel(const float* __restrict__ v, float* __restrict__ out, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float x = v[i];
    out[i] = silu_fma(x);
    out[n + i] = silu_fast(x);
    out[2 * n + i] = silu_f(x);
  }
}

}  // namespace

cudaError_t launch_selftest_silu(const float* v, float* out, long long n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  selftest_silu_kernel<<<(unsigned)blocks, 256, 0, s>>>(v, out, n);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int32_t* status, unsigned long long limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace ssmtree
