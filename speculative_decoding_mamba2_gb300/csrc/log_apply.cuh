// Applying logged draft updates to state rows held in registers (replay, draft-tree commit).
#pragma once

#include "common.cuh"

namespace ssmtree {

// 16 state rows, one float4 (4 consecutive d_state columns, 4·lane .. 4·lane+3) per lane and
// row, take `cnt` logged updates in order:
//     h <- a_t · h + u_t[row] · B_t[col],   u_t[row] = Δ_t · x_t[row],   a_t = exp(Δ_t · A),
// with the one-token draft step's two roundings per element (as ssm_update), so applying the
// log reproduces the stepped state bit for bit.  u: shared [t][ustride], rows r0 .. r0+15;
// B: shared [t][kN]; decay: shared, step t at decay[t * dstride].
__device__ __forceinline__ void apply_logged_updates(float4 (&hr)[16], int cnt, const float* u, int ustride,
                                                     int r0, const float* B, const float* decay, int dstride,
                                                     int lane) {
  // packed pairs (fma.rn.f32x2 / mul.rn.f32x2): the same two roundings per element, half the
  // instructions
  unsigned long long p01[16], p23[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    p01[r] = pack2(hr[r].x, hr[r].y);
    p23[r] = pack2(hr[r].z, hr[r].w);
  }
  for (int t = 0; t < cnt; ++t) {
    const float4 b = reinterpret_cast<const float4*>(B + t * kN)[lane];
    const unsigned long long b01 = pack2(b.x, b.y), b23 = pack2(b.z, b.w);
    const float a = decay[t * dstride];
    const unsigned long long a2 = pack2(a, a);
    const float* ut = u + t * ustride + r0;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const unsigned long long u2 = pack2(ut[r], ut[r]);
      p01[r] = ffma2(a2, p01[r], fmul2(u2, b01));
      p23[r] = ffma2(a2, p23[r], fmul2(u2, b23));
    }
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float2 x01 = unpack2(p01[r]), x23 = unpack2(p23[r]);
    hr[r] = make_float4(x01.x, x01.y, x23.x, x23.y);
  }
}

}  // namespace ssmtree
