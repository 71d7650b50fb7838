// Draft side: one-token draft step with its light log, and replay from that log.
//
// SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践") §3.1: the draft
// model stores only the small intermediates (Δ, A, B, X) instead of whole
// states and recovers its state from them; §2.3: the draft is memory bound.
// A is a per-head constant in Mamba2, so a log row is {Δ [H], B [N], x
// [d_inner]}, all post-conv fp32.  Replay applies the logged updates with the
// exact fp32 operation sequence of the step kernel (decay_of, __fmul_rn,
// ssm_update), so it reproduces the stepped state bit for bit.
#include "common.cuh"
#include "log_apply.cuh"

namespace ssmtree {
namespace {

constexpr int DG = 4;            // heads per CTA
constexpr int DROWS = DG * kP;   // 256 state rows
constexpr int DTHREADS = 256;

__global__ void __launch_bounds__(DTHREADS) draft_step_kernel(DraftArgs a) {
  __shared__ __align__(16) float Bs[kN];
  __shared__ __align__(16) float Cs[kN];
  __shared__ float xs[DROWS];
  __shared__ float dls[DG], decs[DG], Dh[DG];

  const int tid = threadIdx.x;
  const int n_groups = (a.H + DG - 1) / DG;
  const int grp = blockIdx.x % n_groups;
  const int inst = blockIdx.x / n_groups;
  const int layer = inst % a.L;
  const int h_begin = grp * DG;
  const int heads = min(DG, a.H - h_begin);
  const int d_inner = a.H * kP;
  const int conv_dim = d_inner + 2 * kN;
  const int R = a.R;
  const int pos = a.ring_head[inst] + a.step;

  const uint16_t* xt = a.xBC_t + (size_t)inst * conv_dim;
  uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  const uint16_t* r0 = ring + (size_t)ring_pos(pos, -3, R) * conv_dim;
  const uint16_t* r1 = ring + (size_t)ring_pos(pos, -2, R) * conv_dim;
  const uint16_t* r2 = ring + (size_t)ring_pos(pos, -1, R) * conv_dim;
  uint16_t* rw = ring + (size_t)ring_pos(pos, 0, R) * conv_dim;
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float* cb = a.conv_b + (size_t)layer * conv_dim;
  float* lx = a.log_x + ((size_t)inst * a.log_cap + a.step) * d_inner;
  float* lB = a.log_B + ((size_t)inst * a.log_cap + a.step) * kN;

  // conv + SiLU of the one position: this group's x channels, and B, C
  for (int job = tid; job < DROWS + 2 * kN; job += DTHREADS) {
    int c;
    if (job < DROWS) {
      if (job >= heads * kP) continue;
      c = h_begin * kP + job;
    } else {
      c = d_inner + (job - DROWS);  // every group needs B and C; group 0 also writes them out
    }
    const uint16_t cur = xt[c];
    const float post = conv4_silu(cw[c], cb[c], bf16f(r0[c]), bf16f(r1[c]), bf16f(r2[c]), bf16f(cur));
    if (job < DROWS) {
      xs[job] = post;
      lx[c] = post;
      rw[c] = cur;
    } else {
      const int j = job - DROWS;
      if (j < kN) Bs[j] = post;
      else Cs[j - kN] = post;
      if (grp == 0) {
        rw[c] = cur;
        if (j < kN) lB[j] = post;
      }
    }
  }
  if (tid < DG) {
    float d = 0.f, e = 1.f, dd = 0.f;
    if (tid < heads) {
      const int h = h_begin + tid;
      d = softplus_f(bf16f(a.dt_t[(size_t)inst * a.H + h]) + a.dt_bias[(size_t)layer * a.H + h]);
      e = decay_of(d, neg_exp(a.A_log[(size_t)layer * a.H + h]));
      dd = a.D[(size_t)layer * a.H + h];
      a.log_delta[((size_t)inst * a.log_cap + a.step) * a.H + h] = d;
    }
    dls[tid] = d;
    decs[tid] = e;
    Dh[tid] = dd;
  }
  if (grp == 0 && tid == 0) a.log_len[inst] = a.step + 1;
  __syncthreads();

  // state rows: one warp per row, each lane 4 consecutive d_state elements
  const int warp = tid >> 5, lane = tid & 31;
  const float4 b4 = reinterpret_cast<const float4*>(Bs)[lane];
  const float4 c4 = reinterpret_cast<const float4*>(Cs)[lane];
  const float* hin = a.h_in + ((size_t)inst * a.H + h_begin) * kP * kN;
  float* hout = a.h_out + ((size_t)inst * a.H + h_begin) * kP * kN;
  const int rows = heads * kP;
  constexpr int U = 4;                       // rows per step of a warp
  constexpr int STRIDE = (DTHREADS / 32) * U;
  float4 nx[U];                              // the warp's next U rows, loaded one step ahead
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (warp * U + u < rows) nx[u] = reinterpret_cast<const float4*>(hin + (size_t)(warp * U + u) * kN)[lane];
  for (int r0w = warp * U; r0w < rows; r0w += STRIDE) {
    float4 hv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      hv[u] = nx[u];
      if (r0w + STRIDE + u < rows) nx[u] = reinterpret_cast<const float4*>(hin + (size_t)(r0w + STRIDE + u) * kN)[lane];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = r0w + u;
      if (row >= rows) continue;
      const int g = row / kP;
      const float uu = __fmul_rn(dls[g], xs[row]);
      const float dec = decs[g];
      float4 h = hv[u];
      h.x = ssm_update(dec, h.x, uu, b4.x);
      h.y = ssm_update(dec, h.y, uu, b4.y);
      h.z = ssm_update(dec, h.z, uu, b4.z);
      h.w = ssm_update(dec, h.w, uu, b4.w);
      reinterpret_cast<float4*>(hout + (size_t)row * kN)[lane] = h;
      float s = c4.x * h.x;
      s = fmaf(c4.y, h.y, s);
      s = fmaf(c4.z, h.z, s);
      s = fmaf(c4.w, h.w, s);
      s = warp_sum(s);
      if (lane == 0) a.y[(size_t)inst * d_inner + h_begin * kP + row] = fmaf(Dh[g], xs[row], s);
    }
  }
}

// ---------------------------------------------------------------------------
// replay: each warp holds 16 state rows of one head in registers (a float4 of 4 columns
// per lane and row, all 16 loads in flight while the log is staged); a pass stages up to
// RT logged steps in shared memory (u = Δ·x per step and row, the decay per step and
// head, B per step) and applies them with the draft step's operations
// (apply_logged_updates)
// ---------------------------------------------------------------------------
constexpr int RW = 4;               // warps per CTA
constexpr int RTHREADS = RW * 32;
constexpr int RH = 1;               // heads per CTA
constexpr int RROWS = RH * kP;      // 64 state rows, 16 per warp
constexpr int RT = 16;              // logged steps per pass

__device__ __forceinline__ int replay_k(const ReplayArgs& a, int inst, bool report) {
  const int seq = inst / a.L;
  int k = a.k[seq];
  const int lim = max(0, min(a.log_len[inst], a.log_cap));
  if (k < 0 || k > lim) {
    if (report) flag(a.status, SSM_STATUS_K_RANGE);
    k = k < 0 ? 0 : lim;
  }
  return k;
}

__global__ void __launch_bounds__(RTHREADS, 4) replay_kernel(ReplayArgs a) {
  __shared__ float us[RT][RROWS];  // u = Δ_t·x_t[row]
  __shared__ float decs[RT][RH];
  __shared__ __align__(16) float Bs[RT][kN];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_groups = (a.H + RH - 1) / RH;
  const int grp = blockIdx.x % n_groups;
  const int inst = blockIdx.x / n_groups;
  const int layer = inst % a.L;
  const int h_begin = grp * RH;
  const int heads = min(RH, a.H - h_begin);
  const int rows = heads * kP;
  const int d_inner = a.H * kP;
  const int k = replay_k(a, inst, grp == 0 && tid == 0);
  if (k == 0) return;
  float* hs = a.h + ((size_t)inst * a.H + h_begin) * kP * kN;
  const int row0 = warp * (RROWS / RW);  // this warp's 16 rows, all of one head
  const int g = row0 / kP;
  const bool mine = g < heads;
  float4 hr[16];
  if (mine) {
#pragma unroll
    for (int r = 0; r < 16; ++r) hr[r] = reinterpret_cast<const float4*>(hs + (size_t)(row0 + r) * kN)[lane];
  }
  const float A_g = neg_exp(a.A_log[(size_t)layer * a.H + h_begin + min(tid % RH, heads - 1)]);
  for (int t0 = 0; t0 < k; t0 += RT) {
    const int cnt = min(RT, k - t0);
    if (t0 > 0) __syncthreads();  // the previous pass is done with us, decs, Bs
    // every log value of the pass in flight at once: Δ and x for (row, step) pairs, B rows,
    // then the products and decays into shared memory
    static_assert(RTHREADS == 2 * RROWS, "two threads per row, each half of the steps");
    const int r = tid % RROWS, th = tid / RROWS;
    float dl[RT / 2], xv[RT / 2];
#pragma unroll
    for (int j = 0; j < RT / 2; ++j) {
      const int t = th + 2 * j;
      dl[j] = 0.f;
      xv[j] = 0.f;
      if (t < cnt && r < rows) {
        const size_t lrow = (size_t)inst * a.log_cap + t0 + t;
        dl[j] = a.log_delta[lrow * a.H + h_begin + r / kP];
        xv[j] = a.log_x[lrow * d_inner + h_begin * kP + r];
      }
    }
    float4 bv[RT * (kN / 4) / RTHREADS];
#pragma unroll
    for (int q = 0; q < RT * (kN / 4) / RTHREADS; ++q) {
      const int i = tid + q * RTHREADS, t = i / (kN / 4), c4 = i - t * (kN / 4);
      bv[q] = t < cnt ? reinterpret_cast<const float4*>(a.log_B + ((size_t)inst * a.log_cap + t0 + t) * kN)[c4]
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int dt_ = tid / RH, dg = tid - dt_ * RH;
    float dd = 0.f;
    if (tid < cnt * RH && dg < heads) dd = a.log_delta[((size_t)inst * a.log_cap + t0 + dt_) * a.H + h_begin + dg];
#pragma unroll
    for (int j = 0; j < RT / 2; ++j) {
      const int t = th + 2 * j;
      if (t < cnt) us[t][r] = __fmul_rn(dl[j], xv[j]);
    }
#pragma unroll
    for (int q = 0; q < RT * (kN / 4) / RTHREADS; ++q) {
      const int i = tid + q * RTHREADS, t = i / (kN / 4), c4 = i - t * (kN / 4);
      reinterpret_cast<float4*>(Bs[t])[c4] = bv[q];
    }
    if (tid < cnt * RH) decs[dt_][dg] = dg < heads ? decay_of(dd, A_g) : 1.f;
    __syncthreads();
    if (mine) apply_logged_updates(hr, cnt, &us[0][0], RROWS, row0, &Bs[0][0], &decs[0][g], RH, lane);
  }
  if (mine) {
#pragma unroll
    for (int r = 0; r < 16; ++r) reinterpret_cast<float4*>(hs + (size_t)(row0 + r) * kN)[lane] = hr[r];
  }
}

// head += k, log_len = 0 (after every replay CTA has read log_len)
__global__ void replay_finish_kernel(ReplayArgs a, int n_inst) {
  const int inst = blockIdx.x * blockDim.x + threadIdx.x;
  if (inst >= n_inst) return;
  const int k = replay_k(a, inst, false);
  a.ring_head[inst] += k;
  a.log_len[inst] = 0;
}

}  // namespace

cudaError_t launch_draft_step(const DraftArgs& a, cudaStream_t s) {
  const int n_groups = (a.H + DG - 1) / DG;
  const long long inst = (long long)a.n_seq * a.L;
  if (inst == 0) return cudaSuccess;
  draft_step_kernel<<<(unsigned)(n_groups * inst), DTHREADS, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_replay(const ReplayArgs& a, cudaStream_t s) {
  const int n_groups = (a.H + RH - 1) / RH;
  const long long inst = (long long)a.n_seq * a.L;
  if (inst == 0) return cudaSuccess;
  replay_kernel<<<(unsigned)(n_groups * inst), RTHREADS, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  replay_finish_kernel<<<(unsigned)((inst + 255) / 256), 256, 0, s>>>(a, (int)inst);
  return cudaGetLastError();
}

}  // namespace ssmtree
