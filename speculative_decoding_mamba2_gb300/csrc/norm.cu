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
// rmsnorm_vec4_kernel is the same with 16-byte loads when the shapes allow them.
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

// The same with 16-byte loads (4 columns per access) when C and the strides are multiples of 4.
constexpr int NPER4 = 8;  // float4 groups per thread: C <= 8192
__global__ void __launch_bounds__(NTHREADS) rmsnorm_vec4_kernel(int C, const float* __restrict__ x, long long ldx,
                                                                const uint16_t* __restrict__ z, long long ldz,
                                                                const float* __restrict__ w, float eps,
                                                                uint16_t* __restrict__ out, long long ldo) {
  __shared__ float part[NTHREADS / 32];
  const int row = blockIdx.x, tid = threadIdx.x, C4 = C / 4;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * ldx);
  const uint2* zr = z ? reinterpret_cast<const uint2*>(z + (size_t)row * ldz) : nullptr;
  float4 v[NPER4];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NPER4; ++i) {
    const int c = tid + i * NTHREADS;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < C4) {
      g = xr[c];
      if (zr) {
        const uint2 zz = zr[c];
        g.x *= silu_f(bf16_lo(zz.x));
        g.y *= silu_f(bf16_hi(zz.x));
        g.z *= silu_f(bf16_lo(zz.y));
        g.w *= silu_f(bf16_hi(zz.y));
      }
    }
    v[i] = g;
    ss = fmaf(g.x, g.x, fmaf(g.y, g.y, fmaf(g.z, g.z, fmaf(g.w, g.w, ss))));
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < NTHREADS / 32; ++i) tot += part[i];
  const float r = rsqrtf(tot / (float)C + eps);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  uint2* o = reinterpret_cast<uint2*>(out + (size_t)row * ldo);
#pragma unroll
  for (int i = 0; i < NPER4; ++i) {
    const int c = tid + i * NTHREADS;
    if (c < C4) {
      const float4 ww = w4[c];
      uint32_t lo, hi;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(v[i].y * r * ww.y), "f"(v[i].x * r * ww.x));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(v[i].w * r * ww.w), "f"(v[i].z * r * ww.z));
      o[c] = make_uint2(lo, hi);
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm(int M, int C, const float* x, long long ldx, const uint16_t* z, long long ldz,
                           const float* w, float eps, uint16_t* out, long long ldo, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const bool vec = C % 4 == 0 && ldx % 4 == 0 && ldo % 4 == 0 && (!z || ldz % 4 == 0) &&
                   (((uintptr_t)x | (uintptr_t)w) & 15) == 0 && (((uintptr_t)out | (uintptr_t)z) & 7) == 0;
  if (vec)
    rmsnorm_vec4_kernel<<<(unsigned)M, NTHREADS, 0, s>>>(C, x, ldx, z, ldz, w, eps, out, ldo);
  else
    rmsnorm_kernel<<<(unsigned)M, NTHREADS, 0, s>>>(C, x, ldx, z, ldz, w, eps, out, ldo);
  return cudaGetLastError();
}

}  // namespace ssmtree
