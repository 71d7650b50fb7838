// Row norms around the Mamba2 mixer.
//
// LightMamba page ("旋转辅助量化" and "为什么 Mamba 难加速"): the block has an RMSNorm
// before the input projection and a second one after the SSM, where the SSM output
// is multiplied by Z before the output projection.  Read here as Mamba2's gated form:
//     g[c] = y[c] · SiLU(z[c]),   out[c] = w[c] · g[c] / sqrt(mean_c g[c]² + eps)
// and, without z, the plain RMSNorm of the residual stream:
//     out[c] = w[c] · x[c] / sqrt(mean_c x[c]² + eps).
//
// rmsnorm_kernel: one CTA (256 threads) per row; each thread keeps its columns in
// registers (C ≤ 8192), the sum of squares is reduced with warp shuffles and one
// shared-memory pass, the row is written once as bf16 (the next projection's input).
#include "common.cuh"

namespace ssmtree {
namespace {

constexpr int NTHREADS = 256;
constexpr int NPER = 32;  // columns per thread: C ≤ 8192

__global__ void __launch_bounds__(NTHREADS) rmsnorm_kernel(int C, const float* __restrict__ x, long long ldx,
                                                           const uint16_t* __restrict__ z, long long ldz,
                                                           const float* __restrict__ w, float eps,
                                                           uint16_t* __restrict__ out, long long ldo) {
  __shared__ float part[NTHREADS / 32];
  const int row = blockIdx.x, tid = threadIdx.x;
  const float* xr = x + (size_t)row * ldx;
  const uint16_t* zr = z ? z + (size_t)row * ldz : nullptr;
  float v[NPER];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int c = tid + i * NTHREADS;
    float g = 0.f;
    if (c < C) {
      g = xr[c];
      if (zr) g *= silu_f(bf16f(zr[c]));
    }
    v[i] = g;
    ss = fmaf(g, g, ss);
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < NTHREADS / 32; ++i) tot += part[i];
  const float r = rsqrtf(tot / (float)C + eps);
  uint16_t* o = out + (size_t)row * ldo;
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int c = tid + i * NTHREADS;
    if (c < C) {
      uint32_t p;
      const float val = v[i] * r * w[c];
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p) : "f"(0.f), "f"(val));
      o[c] = (uint16_t)(p & 0xffffu);
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm(int M, int C, const float* x, long long ldx, const uint16_t* z, long long ldz,
                           const float* w, float eps, uint16_t* out, long long ldo, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  rmsnorm_kernel<<<(unsigned)M, NTHREADS, 0, s>>>(C, x, ldx, z, ldz, w, eps, out, ldo);
  return cudaGetLastError();
}

}  // namespace ssmtree
