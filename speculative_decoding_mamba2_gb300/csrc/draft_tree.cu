// Draft-side tree drafting: one depth level of the draft tree per call, every node from its
// branch state rebuilt out of the light log, and the commit of the accepted path from the log.
//
// SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践"): §3.1 the draft keeps only the
// small intermediates (Δ, A, B, X) and recovers its state from them; §3.2 a tree node's
// children continue from that node's state; §2.3 the draft side is memory bound.  A draft
// tree grows one depth level at a time (level d+1's tokens come from level d's outputs), so
// a call processes the nodes of one depth.  No branch state is ever stored: for node v with
// root-to-node path m_0 .. m_d = v and S_m = Σ_{j on the path, up to m} Δ_j·A,
//   y_v = e^{S_v} (C_v · h_ckpt) + Σ_k e^{S_v − S_{m_k}} Δ_{m_k} (B_{m_k} · C_v) x_{m_k} + D·x_v,
// which reads the committed state once per level, whatever the number of branches, and
// writes no state.  The ancestors' Δ, B, x are the log rows their own level wrote.
//
// draft_tree_level_kernel: one CTA per (instance, pair of heads).  Each thread loads its
// share of the pair's 128 state rows (8 lanes per row, 16 columns each) into registers
// first, so the loads are in flight while the CTA sets up the level: the frontier list
// and the union of the frontier's paths (shared memory), the ancestors' logged x and Δ,
// the frontier's conv + SiLU (x of the pair's channels, B, C), Δ and their log rows, the
// cumulative log-decays S, the B·C products along each path (one warp per pair) and
// the per-row path sums.  The C_v · h contraction then runs from registers, FB = 8 nodes
// per pass; the 8 lanes of a row end with one node's sum each after a 7-shuffle
// reduce-scatter.
//
// draft_tree_commit_kernel: one CTA per (instance, pair of heads), one warp per state row at
// a time (4 columns per lane), the path's updates applied in path order with the same fp32
// operations as the one-token draft step, so on a chain it reproduces the stepped state bit
// for bit.  draft_tree_ring_kernel then writes the path's last three pre-conv rows into the
// ring and advances the head.
#include "draft_tree.cuh"

namespace ssmtree {
namespace {

constexpr int TG = 2;                            // heads per CTA
constexpr int TROWS = TG * kP;                   // 128 state rows
constexpr int TTHREADS = 256;                    // 8 lanes per row: 32 rows per sweep
constexpr int TSWEEPS = TROWS / (TTHREADS / 8);  // 4
constexpr int FB = 8;                            // frontier nodes per pass
constexpr int MAXN = SSM_MAX_NODES;              // 64
constexpr int MAXP = SSM_MAX_DEPTH + 1;          // 16 nodes on a root-to-node path

struct LevelSmem {
  int par[MAXN], dep[MAXN], tap[MAXN][3], slot[MAXN], front[MAXN];
  int nf;
  int pslot[FB][MAXP], pnode[FB][MAXP], plen[FB];
  float A[TG], Dh[TG];
  float du[MAXN][TG];        // Δ of every node on a frontier path (by slot)
  float su[MAXN][TG];        // S: cumulative Δ·A from the root to the node, inclusive
  float coef[FB][MAXP][TG];  // e^{S_v − S_m} Δ_m (B_m · C_v)
  float E[FB][TG];           // e^{S_v}
  float bc[FB][MAXP];        // B_m · C_v
  __align__(16) float Cf[FB][kN];
  __align__(16) float Bf[FB][kN];
  float base[FB][TROWS];     // Σ_k coef·x_{m_k}[row] + D·x_v[row]
  float xu[MAXN][TROWS];     // post-conv x of the pair's channels, by slot
};

// 8 partial sums per lane, over the 8 lanes o = 0..7 of an aligned lane group: returns
// the full sum of value o (recursive halving: 4 + 2 + 1 shuffles).
__device__ __forceinline__ float reduce_scatter8(const float (&v)[FB], int o) {
  const bool b2 = o & 4, b1 = o & 2, b0 = o & 1;
  float s4[4], s2[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b2 ? v[4 + i] : v[i];
    const float send = b2 ? v[i] : v[4 + i];
    s4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b1 ? s4[2 + i] : s4[i];
    const float send = b1 ? s4[i] : s4[2 + i];
    s2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  const float keep = b0 ? s2[1] : s2[0];
  const float send = b0 ? s2[0] : s2[1];
  return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__global__ void __launch_bounds__(TTHREADS, 2) draft_tree_level_kernel(DraftTreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  LevelSmem& s = *reinterpret_cast<LevelSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, o = tid & 7, rsub = tid >> 3;
  const int n_groups = (a.H + TG - 1) / TG;
  const int grp = blockIdx.x % n_groups;
  const long long inst = blockIdx.x / n_groups;
  const int seq = (int)(inst / a.L), layer = (int)(inst % a.L);
  const int h_begin = grp * TG, heads = min(TG, a.H - h_begin), rows = heads * kP;
  const int n = a.n, d_inner = a.H * kP, conv_dim = d_inner + 2 * kN;
  const size_t node0 = (size_t)inst * n;  // first node row of this instance (xBC, dt, log, y)

  // this thread's state values: rows rsub + 32 i, columns 4 o + 32 j
  const float* hb = a.h + ((size_t)inst * a.H + h_begin) * kP * kN;
  float4 hv[TSWEEPS][4];
#pragma unroll
  for (int i = 0; i < TSWEEPS; ++i) {
    const int row = rsub + 32 * i;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      hv[i][j] = row < rows ? __ldg(reinterpret_cast<const float4*>(hb + (size_t)row * kN) + o + 8 * j)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const ssm_node* lay = a.layout + (size_t)seq * n;
  for (int v = tid; v < n; v += TTHREADS) {
    const ssm_node r = lay[v];
    s.par[v] = r.parent;
    s.dep[v] = r.depth;
    s.tap[v][0] = r.tap[0];
    s.tap[v][1] = r.tap[1];
    s.tap[v][2] = r.tap[2];
    s.slot[v] = -1;
  }
  if (tid < TG) {
    const bool on = tid < heads;
    s.A[tid] = on ? neg_exp(a.A_log[(size_t)layer * a.H + h_begin + tid]) : 0.f;
    s.Dh[tid] = on ? a.D[(size_t)layer * a.H + h_begin + tid] : 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    // records in range (parents and taps earlier nodes, depths consistent), the level's
    // nodes in node order, and every node on their paths numbered in node order
    bool ok = s.par[0] == -1 && s.dep[0] == 0;
    int nf = 0;
    for (int v = 0; v < n && ok; ++v) {
      const int p = s.par[v];
      if (v > 0 && (p < 0 || p >= v || s.dep[v] != s.dep[p] + 1)) ok = false;
      for (int t = 0; t < 3; ++t) {
        const int src = s.tap[v][t];
        if (src >= v || src < -3) ok = false;
      }
      if (ok && s.dep[v] == a.level) s.front[nf++] = v;
    }
    if (ok) {
      for (int f = 0; f < nf; ++f)
        for (int v = s.front[f]; v >= 0; v = s.par[v]) s.slot[v] = 0;
      int nu = 0;
      for (int v = 0; v < n; ++v)
        if (s.slot[v] >= 0) s.slot[v] = nu++;
    } else {
      flag(a.status, SSM_STATUS_BAD_LAYOUT);
    }
    s.nf = ok ? nf : 0;
  }
  __syncthreads();
  const int nf = s.nf;
  if (nf == 0) return;

  // ancestors on the frontier's paths: their logged x (this pair's channels) and Δ
  for (int i = tid; i < n * TROWS; i += TTHREADS) {
    const int v = i / TROWS, r = i - v * TROWS;
    const int sl = s.slot[v];
    if (sl < 0 || s.dep[v] >= a.level) continue;
    s.xu[sl][r] = r < rows ? a.log_x[(node0 + v) * d_inner + h_begin * kP + r] : 0.f;
  }
  for (int i = tid; i < n * TG; i += TTHREADS) {
    const int v = i / TG, g = i - v * TG;
    const int sl = s.slot[v];
    if (sl < 0 || s.dep[v] >= a.level) continue;
    s.du[sl][g] = g < heads ? a.log_delta[(node0 + v) * a.H + h_begin + g] : 0.f;
  }
  __syncthreads();
  if (tid < TG) {  // S of the ancestors, parents first
    for (int v = 0; v < n; ++v) {
      const int sl = s.slot[v];
      if (sl < 0 || s.dep[v] >= a.level) continue;
      const int p = s.par[v];
      s.su[sl][tid] = (p >= 0 ? s.su[s.slot[p]][tid] : 0.f) + s.du[sl][tid] * s.A[tid];
    }
  }

  const uint16_t* xbc = a.xBC + node0 * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * a.R * conv_dim;
  const int head = a.ring_head[inst];
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float* cb = a.conv_b + (size_t)layer * conv_dim;
  constexpr int JOBS = TROWS + 2 * kN;  // per node: the pair's x channels, then B and C

  for (int f0 = 0; f0 < nf; f0 += FB) {
    const int fc = min(FB, nf - f0);
    // conv + SiLU of the pass's nodes, their Δ, and their log rows
    for (int job = tid; job < FB * JOBS; job += TTHREADS) {
      const int f = job / JOBS, cl = job - f * JOBS;
      if (f >= fc) {
        if (cl >= TROWS + kN) s.Cf[f][cl - TROWS - kN] = 0.f;
        continue;
      }
      const int v = s.front[f0 + f];
      int c;
      if (cl < TROWS) {
        if (cl >= rows) {
          s.xu[s.slot[v]][cl] = 0.f;
          continue;
        }
        c = h_begin * kP + cl;
      } else {
        c = d_inner + (cl - TROWS);
      }
      const float post = node_conv(xbc, ring, head, a.R, conv_dim, s.tap[v], v, c, cw[c], cb[c]);
      if (cl < TROWS) {
        s.xu[s.slot[v]][cl] = post;
        a.log_x[(node0 + v) * d_inner + c] = post;
      } else {
        const int j = cl - TROWS;
        if (j < kN) {
          s.Bf[f][j] = post;
          if (grp == 0) a.log_B[(node0 + v) * kN + j] = post;
        } else {
          s.Cf[f][j - kN] = post;
        }
      }
    }
    if (tid < FB * TG) {
      const int f = tid / TG, g = tid - f * TG;
      if (f < fc) {
        const int v = s.front[f0 + f];
        float d = 0.f;
        if (g < heads) {
          const int h = h_begin + g;
          d = softplus_f(bf16f(a.dt[(node0 + v) * a.H + h]) + a.dt_bias[(size_t)layer * a.H + h]);
          a.log_delta[(node0 + v) * a.H + h] = d;
        }
        s.du[s.slot[v]][g] = d;
      }
    }
    __syncthreads();
    if (tid < FB * TG) {  // S of the pass's nodes (their parents are ancestors)
      const int f = tid / TG, g = tid - f * TG;
      if (f < fc) {
        const int v = s.front[f0 + f], p = s.par[v], sl = s.slot[v];
        s.su[sl][g] = (p >= 0 ? s.su[s.slot[p]][g] : 0.f) + s.du[sl][g] * s.A[g];
      }
    }
    if (tid < FB) {  // each pass node's path, root first
      int len = 0;
      if (tid < fc) {
        const int v = s.front[f0 + tid];
        len = s.dep[v] + 1;
        int u = v;
        for (int k = len - 1; k >= 0; --k) {
          s.pnode[tid][k] = u;
          s.pslot[tid][k] = s.slot[u];
          u = s.par[u];
        }
      }
      s.plen[tid] = len;
    }
    __syncthreads();
    // B_m · C_v along each path: one warp per (node, path position)
    for (int q = warp; q < FB * MAXP; q += TTHREADS / 32) {
      const int f = q / MAXP, k = q - f * MAXP;
      if (f >= fc || k >= s.plen[f]) continue;
      float4 b4;
      if (k == s.plen[f] - 1)
        b4 = reinterpret_cast<const float4*>(s.Bf[f])[lane];
      else
        b4 = __ldg(reinterpret_cast<const float4*>(a.log_B + (node0 + s.pnode[f][k]) * kN) + lane);
      const float4 c4 = reinterpret_cast<const float4*>(s.Cf[f])[lane];
      float d = b4.x * c4.x;
      d = fmaf(b4.y, c4.y, d);
      d = fmaf(b4.z, c4.z, d);
      d = fmaf(b4.w, c4.w, d);
      d = warp_sum(d);
      if (lane == 0) s.bc[f][k] = d;
    }
    __syncthreads();
    {
      static_assert(FB * MAXP * TG == TTHREADS, "one coefficient per thread");
      const int f = tid / (MAXP * TG), rem = tid - f * (MAXP * TG), k = rem / TG, g = rem - k * TG;
      if (f < fc && k < s.plen[f]) {
        const int sv = s.pslot[f][s.plen[f] - 1], sm = s.pslot[f][k];
        s.coef[f][k][g] = expf(s.su[sv][g] - s.su[sm][g]) * s.du[sm][g] * s.bc[f][k];
      }
      if (tid < FB * TG) {
        const int ff = tid / TG, gg = tid - ff * TG;
        if (ff < fc) s.E[ff][gg] = expf(s.su[s.slot[s.front[f0 + ff]]][gg]);
      }
    }
    __syncthreads();
    for (int i = tid; i < FB * TROWS; i += TTHREADS) {
      const int f = i / TROWS, r = i - f * TROWS;
      float b = 0.f;
      if (f < fc && r < rows) {
        const int g = r / kP, len = s.plen[f];
        for (int k = 0; k < len; ++k) b = fmaf(s.coef[f][k][g], s.xu[s.pslot[f][k]][r], b);
        b = fmaf(s.Dh[g], s.xu[s.pslot[f][len - 1]][r], b);
      }
      s.base[f][r] = b;
    }
    __syncthreads();
    // y_v = e^{S_v} (C_v · h_ckpt) + base, from the state values held in registers; each
    // C float4 is read once and used for all of the thread's rows
    float acc[TSWEEPS][FB];
#pragma unroll
    for (int i = 0; i < TSWEEPS; ++i)
#pragma unroll
      for (int f = 0; f < FB; ++f) acc[i][f] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int f = 0; f < FB; ++f) {
        const float4 c = reinterpret_cast<const float4*>(s.Cf[f])[o + 8 * j];
#pragma unroll
        for (int i = 0; i < TSWEEPS; ++i) {
          acc[i][f] = fmaf(hv[i][j].x, c.x, acc[i][f]);
          acc[i][f] = fmaf(hv[i][j].y, c.y, acc[i][f]);
          acc[i][f] = fmaf(hv[i][j].z, c.z, acc[i][f]);
          acc[i][f] = fmaf(hv[i][j].w, c.w, acc[i][f]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < TSWEEPS; ++i) {
      const int row = rsub + 32 * i;
      const float sum = reduce_scatter8(acc[i], o);
      if (o < fc && row < rows) {
        const int g = row / kP, v = s.front[f0 + o];
        a.y[(node0 + v) * d_inner + h_begin * kP + row] = fmaf(s.E[o][g], sum, s.base[o][row]);
      }
    }
    __syncthreads();  // the next pass rewrites Cf, Bf, xu of its nodes, base
  }
}

// ---------------------------------------------------------------------------
// commit of the accepted path from the log
// ---------------------------------------------------------------------------
constexpr int CH = 2;               // heads per CTA
constexpr int CROWS = CH * kP;      // 128 state rows, 16 per warp
constexpr int CTHREADS = 256;
constexpr int CT = 16;              // path nodes per pass

// Length of the valid prefix of a sequence's accepted path: path[0] = 0, then each entry a
// child of the one before, at most max_path entries; anything else is flagged.
__device__ int tree_path_len(const DraftTreeCommitArgs& a, int seq, bool report) {
  int len = a.path_len[seq];
  bool bad = false;
  if (len < 0 || len > a.max_path) {
    bad = true;
    len = len < 0 ? 0 : a.max_path;
  }
  const int32_t* p = a.path + (size_t)seq * a.max_path;
  const ssm_node* lay = a.layout + (size_t)seq * a.n;
  int prev = -1, good = 0;
  for (int j = 0; j < len; ++j) {
    const int v = p[j];
    const bool ok = j == 0 ? v == 0 : (v > prev && v < a.n && lay[v].parent == prev);
    if (!ok) {
      bad = true;
      break;
    }
    prev = v;
    ++good;
  }
  if (bad && report) flag(a.status, SSM_STATUS_PATH_RANGE);
  return good;
}

__global__ void __launch_bounds__(CTHREADS) draft_tree_commit_kernel(DraftTreeCommitArgs a) {
  __shared__ float us[CT][CROWS];  // Δ_t·x_t[row]
  __shared__ float decs[CT][CH];
  __shared__ int nodes[CT];
  __shared__ int s_len;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_groups = (a.H + CH - 1) / CH;
  const int grp = blockIdx.x % n_groups;
  const long long inst = blockIdx.x / n_groups;
  const int seq = (int)(inst / a.L), layer = (int)(inst % a.L);
  const int h_begin = grp * CH, heads = min(CH, a.H - h_begin), rows = heads * kP;
  const int d_inner = a.H * kP;
  const size_t node0 = (size_t)inst * a.n;
  if (tid == 0) s_len = tree_path_len(a, seq, grp == 0 && layer == 0);
  __syncthreads();
  const int len = s_len;
  float* hs = a.h + ((size_t)inst * a.H + h_begin) * kP * kN;
  const int row0 = warp * (CROWS / 8);
  const int g = row0 / kP;

  for (int t0 = 0; t0 < len; t0 += CT) {
    const int cnt = min(CT, len - t0);
    if (t0 > 0) __syncthreads();  // the previous pass is done with nodes, us, decs
    if (tid < cnt) nodes[tid] = a.path[(size_t)seq * a.max_path + t0 + tid];
    __syncthreads();
    for (int i = tid; i < cnt * CROWS; i += CTHREADS) {
      const int t = i / CROWS, r = i - t * CROWS;
      float u = 0.f;
      if (r < rows) {
        const size_t lr = node0 + nodes[t];
        u = __fmul_rn(a.log_delta[lr * a.H + h_begin + r / kP], a.log_x[lr * d_inner + h_begin * kP + r]);
      }
      us[t][r] = u;
    }
    if (tid < cnt * CH) {
      const int t = tid / CH, gg = tid - t * CH;
      float e = 1.f;
      if (gg < heads) {
        const int h = h_begin + gg;
        e = decay_of(a.log_delta[(node0 + nodes[t]) * a.H + h], neg_exp(a.A_log[(size_t)layer * a.H + h]));
      }
      decs[t][gg] = e;
    }
    float4 bt[CT];
#pragma unroll
    for (int t = 0; t < CT; ++t)
      bt[t] = t < cnt ? __ldg(reinterpret_cast<const float4*>(a.log_B + (node0 + nodes[t]) * kN) + lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    if (g < heads) {
      float4 nx = reinterpret_cast<const float4*>(hs + (size_t)row0 * kN)[lane];
      for (int r = row0; r < row0 + CROWS / 8; ++r) {  // one row in work, the next in flight
        float4 h = nx;
        if (r + 1 < row0 + CROWS / 8) nx = reinterpret_cast<const float4*>(hs + (size_t)(r + 1) * kN)[lane];
#pragma unroll
        for (int t = 0; t < CT; ++t) {
          if (t < cnt) {
            const float u = us[t][r], dec = decs[t][g];
            h.x = ssm_update(dec, h.x, u, bt[t].x);
            h.y = ssm_update(dec, h.y, u, bt[t].y);
            h.z = ssm_update(dec, h.z, u, bt[t].z);
            h.w = ssm_update(dec, h.w, u, bt[t].w);
          }
        }
        reinterpret_cast<float4*>(hs + (size_t)r * kN)[lane] = h;
      }
    }
  }
}

// the path's last three pre-conv rows into the ring, head += len
__global__ void draft_tree_ring_kernel(DraftTreeCommitArgs a) {
  __shared__ int s_len, s_head, rows3[3];
  const long long inst = blockIdx.x;
  const int seq = (int)(inst / a.L);
  const int conv_dim = a.H * kP + 2 * kN;
  if (threadIdx.x == 0) {
    const int len = tree_path_len(a, seq, false);
    s_len = len;
    s_head = a.ring_head[inst];
    for (int j = 0; j < 3; ++j) {
      const int jj = len - 3 + j;
      rows3[j] = jj >= 0 ? a.path[(size_t)seq * a.max_path + jj] : -1;
    }
  }
  __syncthreads();
  const uint16_t* xbc = a.xBC + (size_t)inst * a.n * conv_dim;
  uint16_t* ring = a.ring + (size_t)inst * a.R * conv_dim;
  for (int j = 0; j < 3; ++j) {
    const int v = rows3[j];
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

cudaError_t launch_draft_tree_level(const DraftTreeArgs& a, cudaStream_t s) {
  const long long inst = (long long)a.n_seq * a.L;
  if (inst == 0) return cudaSuccess;
  const int n_groups = (a.H + TG - 1) / TG;
  const int smem = (int)sizeof(LevelSmem);
  cudaError_t e = cudaFuncSetAttribute(draft_tree_level_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  draft_tree_level_kernel<<<(unsigned)(inst * n_groups), TTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_draft_tree_commit(const DraftTreeCommitArgs& a, cudaStream_t s) {
  const long long inst = (long long)a.n_seq * a.L;
  if (inst == 0) return cudaSuccess;
  const int n_groups = (a.H + CH - 1) / CH;
  draft_tree_commit_kernel<<<(unsigned)(inst * n_groups), CTHREADS, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  draft_tree_ring_kernel<<<(unsigned)inst, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ssmtree
