// Accept walk, commit (selective recompute of the accepted path) and the conv
// ring advance.
//
// SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践"):
//   §1.2  the target verifies the draft's tokens;
//   §2.1  after a rejection the state must go back to the last accepted token;
//   §3.1  the target recomputes only the affected path (dependency analysis),
//         which is the accepted root-to-node path;
//   §3.2  the conv state lives in a ring buffer.
#include "common.cuh"

namespace ssmtree {
namespace {

// ---------------------------------------------------------------------------
// accept: one warp per sequence, greedy walk over the breadth-first tree
// ---------------------------------------------------------------------------
__global__ void accept_kernel(AcceptArgs a) {
  const int lane = threadIdx.x & 31;
  const int seq = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (seq >= a.n_seq) return;
  const int n = a.n;
  const ssm_node* lay = a.layout + (size_t)seq * n;
  const int32_t* tok = a.tok + (size_t)seq * n;
  const int32_t* tgt = a.tgt + (size_t)seq * n;
  int32_t* path = a.path + (size_t)seq * a.max_path;
  int cur = 0, len = 1;
  if (lane == 0) path[0] = 0;
  for (;;) {
    const ssm_node r = lay[cur];
    int cb = r.child_begin, cc = r.child_count;
    if (cc <= 0) break;
    if (cb <= cur || cb + cc > n) {  // children must follow their parent
      if (lane == 0) flag(a.status, SSM_STATUS_BAD_LAYOUT);
      break;
    }
    const int want = tgt[cur];
    int found = -1;
    for (int base = 0; base < cc && found < 0; base += 32) {
      const bool hit = base + lane < cc && tok[cb + base + lane] == want;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) found = cb + base + __ffs(m) - 1;
    }
    if (found < 0) break;
    if (len == a.max_path) {
      if (lane == 0) flag(a.status, SSM_STATUS_WALK_TRUNCATED);
      break;
    }
    if (lane == 0) path[len] = found;
    ++len;
    cur = found;
  }
  for (int j = len + lane; j < a.max_path; j += 32) path[j] = -1;
  if (lane == 0) {
    a.path_len[seq] = len;
    a.bonus[seq] = tgt[cur];
  }
}

// ---------------------------------------------------------------------------
// commit: h <- state after the accepted path, re-run from h0 (in place)
// ---------------------------------------------------------------------------
constexpr int CG = 8;            // heads per CTA
constexpr int CROWS = CG * kP;   // 512 state rows
constexpr int PC = 16;           // path nodes per sweep
constexpr int CTHREADS = 256;

// validated accepted path of one sequence into shared memory; returns its length
__device__ int load_path(const CommitArgs& a, int seq, int* pth) {
  __shared__ int s_len;
  if (threadIdx.x == 0) {
    int len = a.path_len[seq];
    bool bad = false;
    if (len < 1 || len > a.max_path) {
      bad = true;
      len = len < 1 ? 1 : a.max_path;
    }
    const int32_t* p = a.path + (size_t)seq * a.max_path;
    const ssm_node* lay = a.layout + (size_t)seq * a.n;
    int prev = -1, good = 0;
    for (int j = 0; j < len; ++j) {
      const int v = p[j];
      const bool ok = (j == 0) ? v == 0 : (v > prev && v < a.n && lay[v].parent == prev);
      if (!ok) {
        bad = true;
        break;
      }
      pth[j] = v;
      prev = v;
      ++good;
    }
    if (good == 0) {
      pth[0] = 0;
      good = 1;
    }
    if (bad) flag(a.status, SSM_STATUS_PATH_RANGE);
    s_len = good;
  }
  __syncthreads();
  return s_len;
}

__global__ void __launch_bounds__(CTHREADS) commit_kernel(CommitArgs a) {
  __shared__ int pth[SSM_MAX_PATH];
  __shared__ __align__(16) float Bs[PC][kN];
  __shared__ __align__(16) float xs[PC][CROWS];
  __shared__ float dls[PC][CG];
  __shared__ float decs[PC][CG];
  __shared__ float Es[CG];
  __shared__ int taps[PC][3];

  const int tid = threadIdx.x;
  const int n_groups = (a.H + CG - 1) / CG;
  const int grp = blockIdx.x % n_groups;
  const int inst = blockIdx.x / n_groups;
  const int seq = inst / a.L;
  const int layer = inst % a.L;
  const int h_begin = grp * CG;
  const int heads = min(CG, a.H - h_begin);
  const int d_inner = a.H * kP;
  const int conv_dim = d_inner + 2 * kN;
  const int len = load_path(a, seq, pth);

  const uint16_t* xbc = a.xBC + (size_t)inst * a.n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * a.R * conv_dim;
  const int head = a.ring_head[inst];
  const ssm_node* lay = a.layout + (size_t)seq * a.n;
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float* cb = a.conv_b + (size_t)layer * conv_dim;
  float* hs = a.h + ((size_t)inst * a.H + h_begin) * kP * kN;
  const int n4 = heads * kP * kN / 4;  // float4 elements of this group's state

  for (int j0 = 0; j0 < len; j0 += PC) {
    const int cnt = min(PC, len - j0);
    if (j0 > 0) __syncthreads();  // previous sweep done with the shared tables
    if (tid < cnt * 3) {
      const int j = tid / 3, d = tid % 3;
      int t = lay[pth[j0 + j]].tap[d];
      if (t >= a.n || t < -3) t = -1;
      taps[j][d] = t;
    }
    __syncthreads();
    // conv + SiLU of the path nodes: B (all N) and this group's x channels
    for (int job = tid; job < CROWS + kN; job += CTHREADS) {
      int c;
      float* dst;
      int stride;
      if (job < CROWS) {
        if (job >= heads * kP) continue;
        c = h_begin * kP + job;
        dst = &xs[0][job];
        stride = CROWS;
      } else {
        c = d_inner + (job - CROWS);
        dst = &Bs[0][job - CROWS];
        stride = kN;
      }
      const float4 w = cw[c];
      const float b = cb[c];
      for (int j = 0; j < cnt; ++j)
        dst[j * stride] = node_conv(xbc, ring, head, a.R, conv_dim, taps[j], pth[j0 + j], c, w, b);
    }
    if (tid < cnt * CG) {
      const int j = tid / CG, g = tid % CG;
      float d = 0.f, e = 1.f;
      if (g < heads) {
        const int h = h_begin + g;
        const int v = pth[j0 + j];
        d = softplus_f(bf16f(a.dt[((size_t)inst * a.n + v) * a.H + h]) + a.dt_bias[(size_t)layer * a.H + h]);
        e = decay_of(d, neg_exp(a.A_log[(size_t)layer * a.H + h]));
      }
      dls[j][g] = d;
      decs[j][g] = e;
    }
    __syncthreads();
    // longer sweeps take their nodes as one rank-cnt update (the folded commit's form):
    //     h' = E·h + Σ_j (w_j·x_j[p])·B_j[n],  w_j = Δ_j·Π_{i>j} a_i,  E = Π_j a_j  (per head),
    // one FMA per node and element instead of a multiply and an FMA; short ones (the common
    // accepted paths of a few nodes) keep the node-by-node update, which needs no extra pass
    const bool folded = cnt > 4;
    if (folded && tid < CG) {
      float run = 1.f;
      for (int j = cnt - 1; j >= 0; --j) {
        dls[j][tid] *= run;  // w_j
        run *= decs[j][tid];
      }
      Es[tid] = run;
    }
    if (folded) {
      __syncthreads();
      for (int i = tid; i < cnt * CROWS; i += CTHREADS) {
        const int j = i / CROWS, r = i - j * CROWS;
        xs[j][r] *= dls[j][r / kP];  // u_j[p] = w_j·x_j[p]
      }
      __syncthreads();
    }
    // sweep the state slice
    for (int e0 = tid; e0 < n4; e0 += CTHREADS * 4) {
      float4 hv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * CTHREADS;
        if (e < n4) hv[u] = reinterpret_cast<const float4*>(hs)[e];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * CTHREADS;
        if (e >= n4) continue;
        const int row = e / (kN / 4);  // g*P + p
        const int g = row / kP;
        const int nn = (e % (kN / 4)) * 4;
        float4 h4 = hv[u];
        if (folded) {
          const float E = Es[g];
          h4 = make_float4(E * h4.x, E * h4.y, E * h4.z, E * h4.w);
          for (int j = 0; j < cnt; ++j) {
            const float uu = xs[j][row];
            const float4 b4 = *reinterpret_cast<const float4*>(&Bs[j][nn]);
            h4.x = fmaf(uu, b4.x, h4.x);
            h4.y = fmaf(uu, b4.y, h4.y);
            h4.z = fmaf(uu, b4.z, h4.z);
            h4.w = fmaf(uu, b4.w, h4.w);
          }
        } else {
          for (int j = 0; j < cnt; ++j) {
            const float uu = __fmul_rn(dls[j][g], xs[j][row]);
            const float dec = decs[j][g];
            const float4 b4 = *reinterpret_cast<const float4*>(&Bs[j][nn]);
            h4.x = ssm_update(dec, h4.x, uu, b4.x);
            h4.y = ssm_update(dec, h4.y, uu, b4.y);
            h4.z = ssm_update(dec, h4.z, uu, b4.z);
            h4.w = ssm_update(dec, h4.w, uu, b4.w);
          }
        }
        reinterpret_cast<float4*>(hs)[e] = h4;
      }
    }
  }
}

// conv ring: the last min(len, 3) path rows go to positions head+len-3 .. head+len-1,
// then the head advances by len (separate launch: every commit CTA has read the old head)
__global__ void ring_advance_kernel(CommitArgs a) {
  __shared__ int s_len, s_head;
  __shared__ int nodes3[3];
  const int inst = blockIdx.x;
  const int seq = inst / a.L;
  const int d_inner = a.H * kP;
  const int conv_dim = d_inner + 2 * kN;
  if (threadIdx.x == 0) {
    int len = a.path_len[seq];
    len = len < 1 ? 1 : (len > a.max_path ? a.max_path : len);
    const int32_t* p = a.path + (size_t)seq * a.max_path;
    const ssm_node* lay = a.layout + (size_t)seq * a.n;
    int prev = -1, good = 0;
    for (int j = 0; j < len; ++j) {  // same validation as the state commit
      const int v = p[j];
      const bool ok = (j == 0) ? v == 0 : (v > prev && v < a.n && lay[v].parent == prev);
      if (!ok) break;
      prev = v;
      ++good;
    }
    if (good == 0) good = 1;
    s_len = good;
    s_head = a.ring_head[inst];
    for (int j = 0; j < 3; ++j) {
      const int jj = good - 3 + j;
      nodes3[j] = jj >= 0 ? (jj == 0 ? 0 : p[jj]) : -1;
    }
  }
  __syncthreads();
  const uint16_t* xbc = a.xBC + (size_t)inst * a.n * conv_dim;
  uint16_t* ring = a.ring + (size_t)inst * a.R * conv_dim;
  for (int j = 0; j < 3; ++j) {
    const int v = nodes3[j];
    if (v < 0) continue;
    const int pos = ring_pos(s_head, s_len - 3 + j, a.R);
    // rows are conv_dim * 2 bytes = 16-byte multiples (conv_dim = 64*H + 256)
    const uint4* src = reinterpret_cast<const uint4*>(xbc + (size_t)v * conv_dim);
    uint4* dst = reinterpret_cast<uint4*>(ring + (size_t)pos * conv_dim);
    for (int c = threadIdx.x; c < conv_dim / 8; c += blockDim.x) dst[c] = src[c];
  }
  __syncthreads();
  if (threadIdx.x == 0) a.ring_head[inst] = s_head + s_len;
}

}  // namespace

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
  if (a.n_seq == 0) return cudaSuccess;
  const int warps = 4;
  accept_kernel<<<(a.n_seq + warps - 1) / warps, warps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s) {
  const int n_groups = (a.H + CG - 1) / CG;
  const long long inst = (long long)a.n_seq * a.L;
  if (inst == 0) return cudaSuccess;
  commit_kernel<<<(unsigned)(n_groups * inst), CTHREADS, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ring_advance_kernel<<<(unsigned)inst, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ssmtree
