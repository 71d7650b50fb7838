// Verification of a chain-shaped draft tree (parent[v] = v - 1), of any length.
//
// SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践") §3.2: the tree
// is walked in order, each node updated from its parent's state, the parent's
// state released once its child is done.  For a chain that walk needs exactly
// one live state, so one CTA per (instance, head) keeps its 64 x 128 state slice
// in registers (256 threads, 32 elements each: row p = thread/4, columns
// 32*(thread%4) .. +32) for the whole chain.  The nodes stream through shared
// memory in segments of 16: conv + SiLU of the segment's x (this head) and B, C
// channels from the pre-conv rows (the three rows before the segment come from
// the previous nodes, or from the conv ring for the first segment), Δ and the
// decay exp(Δ·A); then, node by node,
//     h = exp(Δ_v·A)·h + (Δ_v·x_v[p])·B_v[k],   y_v[p] = Σ_k C_v[k]·h[p][k] + D·x_v[p]
// with the four partial sums of a row combined by quad shuffles.  h0 is read
// once, no per-node state touches memory.
#include "common.cuh"

namespace ssmtree {
namespace {

constexpr int CT = 256;          // threads: 64 rows x 4 column quarters
constexpr int SEG = 16;          // nodes per segment
constexpr int QS = kN / 4;       // 32 columns per thread
constexpr int BSTR = kN + 16;    // B/C rows padded so the four quarters hit different banks

__device__ __forceinline__ int bc_col(int k) { return k + (k / QS) * 4; }

__global__ void __launch_bounds__(CT) chain_verify_kernel(VerifyArgs a) {
  __shared__ __align__(16) float Bs[SEG][BSTR];
  __shared__ __align__(16) float Cs[SEG][BSTR];
  __shared__ float xs[SEG][kP];
  __shared__ float dls[SEG], decs[SEG];

  const int tid = threadIdx.x;
  const int h = blockIdx.x % a.H;
  const int inst = blockIdx.x / a.H;
  const int layer = inst % a.L;
  const int n = a.n;
  const int d_inner = a.H * kP, conv_dim = d_inner + 2 * kN, R = a.R;
  const int p = tid >> 2, qq = tid & 3;
  const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  const int head = a.ring_head[inst];
  const float A = neg_exp(a.A_log[(size_t)layer * a.H + h]);
  const float bias = a.dt_bias[(size_t)layer * a.H + h];
  const float Dh = a.D[(size_t)layer * a.H + h];
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float* cb = a.conv_b + (size_t)layer * conv_dim;

  // this thread's state: row p of head h, columns 32*qq .. 32*qq+31
  float st[QS];
  {
    const float4* src =
        reinterpret_cast<const float4*>(a.h0 + (((size_t)inst * a.H + h) * kP + p) * kN + qq * QS);
#pragma unroll
    for (int i = 0; i < QS / 4; ++i) {
      const float4 v = src[i];
      st[4 * i] = v.x;
      st[4 * i + 1] = v.y;
      st[4 * i + 2] = v.z;
      st[4 * i + 3] = v.w;
    }
  }
  // pre-conv value of channel c at chain position j (j < 0: ring position head + j)
  auto pre = [&](int j, int c) -> float {
    if (j >= 0) return bf16f(xbc[(size_t)j * conv_dim + c]);
    return bf16f(ring[(size_t)ring_pos(head, j, R) * conv_dim + c]);
  };
  // conv jobs of a segment: x channels of this head (64) and B, C (256), one channel per thread
  const int c_x = h * kP + (tid & (kP - 1));  // threads 0..63 do x
  const int c_bc = d_inner + tid;              // every thread does one B|C channel
  const float4 wx = cw[c_x], wbc = cw[c_bc];
  const float bx = cb[c_x], bbc = cb[c_bc];

  for (int s0 = 0; s0 < n; s0 += SEG) {
    const int cnt = min(SEG, n - s0);
    __syncthreads();  // previous segment's tables consumed
    {
      float r0 = pre(s0 - 3, c_bc), r1 = pre(s0 - 2, c_bc), r2 = pre(s0 - 1, c_bc);
      float* dst = tid < kN ? &Bs[0][bc_col(tid)] : &Cs[0][bc_col(tid - kN)];
      for (int j = 0; j < cnt; ++j) {
        const float r3 = pre(s0 + j, c_bc);
        dst[j * BSTR] = silu_f(conv4_acc(wbc, bbc, r0, r1, r2, r3));
        r0 = r1;
        r1 = r2;
        r2 = r3;
      }
    }
    if (tid < kP) {
      float r0 = pre(s0 - 3, c_x), r1 = pre(s0 - 2, c_x), r2 = pre(s0 - 1, c_x);
      for (int j = 0; j < cnt; ++j) {
        const float r3 = pre(s0 + j, c_x);
        xs[j][tid] = silu_f(conv4_acc(wx, bx, r0, r1, r2, r3));
        r0 = r1;
        r1 = r2;
        r2 = r3;
      }
    } else if (tid < kP + cnt) {
      const int j = tid - kP;
      const float d = softplus_f(bf16f(a.dt[((size_t)inst * n + s0 + j) * a.H + h]) + bias);
      dls[j] = d;
      decs[j] = decay_of(d, A);
    }
    __syncthreads();
    for (int j = 0; j < cnt; ++j) {
      const float dec = decs[j];
      const float xv = xs[j][p];
      const float u = __fmul_rn(dls[j], xv);
      const float4* b4 = reinterpret_cast<const float4*>(&Bs[j][qq * (QS + 4)]);
      const float4* c4 = reinterpret_cast<const float4*>(&Cs[j][qq * (QS + 4)]);
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;  // four independent partial sums
#pragma unroll
      for (int i = 0; i < QS / 4; ++i) {
        const float4 bv = b4[i], cv = c4[i];
        st[4 * i] = ssm_update(dec, st[4 * i], u, bv.x);
        st[4 * i + 1] = ssm_update(dec, st[4 * i + 1], u, bv.y);
        st[4 * i + 2] = ssm_update(dec, st[4 * i + 2], u, bv.z);
        st[4 * i + 3] = ssm_update(dec, st[4 * i + 3], u, bv.w);
        acc0 = fmaf(cv.x, st[4 * i], acc0);
        acc1 = fmaf(cv.y, st[4 * i + 1], acc1);
        acc2 = fmaf(cv.z, st[4 * i + 2], acc2);
        acc3 = fmaf(cv.w, st[4 * i + 3], acc3);
      }
      float acc = (acc0 + acc1) + (acc2 + acc3);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (qq == 0) a.y[((size_t)inst * n + s0 + j) * d_inner + h * kP + p] = fmaf(Dh, xv, acc);
    }
  }
}

}  // namespace

cudaError_t launch_chain_verify(const VerifyArgs& a, cudaStream_t s) {
  const long long blocks = (long long)a.n_seq * a.L * a.H;
  if (blocks == 0) return cudaSuccess;
  chain_verify_kernel<<<(unsigned)blocks, CT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ssmtree
