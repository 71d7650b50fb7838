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
// draft_tree_bc_kernel (one CTA per instance): one warp finds the level's nodes and the nodes
// on their paths; B of the ancestors (their logged values) and B | C of the level's nodes
// (conv taps, conv + SiLU; B logged) are loaded in rounds with every load of a round in
// flight; the CTA writes C_v and the products B_{m_k} · C_v along every level node's path to
// the workspace.  This part is the same for every head, so it is done once per instance.
// draft_tree_prep_kernel (one CTA per instance and block of 4 heads, a dependent grid of the
// B | C kernel, so its loads overlap that kernel): x of the block's 256 channels for 8
// ancestors (logged) and 4 level nodes (conv + SiLU, logged) per round, Δ, S; then, once the
// products are complete, e^{S_v} for its heads and the path sum
// Σ_k e^{S_v − S_{m_k}} Δ_{m_k} (B_{m_k} · C_v) x_{m_k} + D·x_v for its rows.
// draft_tree_level_kernel (persistent, two CTAs per SM, launched as a dependent grid of the
// prep): each CTA walks a contiguous run of (instance, head) items and keeps the next three
// heads' 64 committed state rows in flight (bulk copies into a ring of shared-memory stages);
// per head, the C_v · h contraction runs from the stage, 8 nodes per pass, the 8 lanes of a
// row ending with one node's sum each after a 7-shuffle reduce-scatter:
// y_v = e^{S_v} (C_v · h) + path sum.
//
// draft_tree_commit_kernel (one CTA per instance and head): each warp holds 16 state
// rows in registers (16 loads in flight per lane) and applies the path's logged updates in
// path order with the one-token draft step's fp32 operations (apply_logged_updates), so on a
// chain it reproduces the stepped state bit for bit.  draft_tree_ring_kernel then writes the
// path's last three pre-conv rows into the ring and advances the head.
#include "draft_tree.cuh"
#include "log_apply.cuh"

namespace ssmtree {
namespace {

constexpr int TTHREADS = 256;                    // prep kernel
constexpr int FB = 8;                            // level nodes per pass
constexpr int MAXN = SSM_MAX_NODES;              // 64
constexpr int MAXP = SSM_MAX_DEPTH + 1;          // 16 nodes on a root-to-node path
static_assert(MAXN <= 64, "level_setup covers 64 nodes with one warp");

// The level's nodes and every node on their root-to-node paths, for one sequence.
struct LevelSetup {
  int par[MAXN], dep[MAXN], tap[MAXN][3];
  int slot[MAXN];   // node -> position among the nodes on the level's paths (node order), or -1
  int snode[MAXN];  // slot -> node
  int front[MAXN];  // the level's nodes, in node order
  int nf, nu;
};

// One warp: loads the records, checks that every parent and tap is an earlier node and the
// depths agree, and lists the level's nodes and the nodes on their paths.  A record that
// fails leaves nf = 0 (and sets SSM_STATUS_BAD_LAYOUT when `report`).
__device__ __forceinline__ void level_setup(LevelSetup& s, const ssm_node* lay, int n, int level, int32_t* status, bool report) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu, lt = (1u << lane) - 1u;
  bool ok = true;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int v = lane + 32 * k;
    if (v < n) {
      const ssm_node r = lay[v];
      s.par[v] = r.parent;
      s.dep[v] = r.depth;
      s.slot[v] = -1;
      ok = ok && (v == 0 ? (r.parent == -1 && r.depth == 0) : (r.parent >= 0 && r.parent < v));
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        s.tap[v][t] = r.tap[t];
        ok = ok && r.tap[t] < v && r.tap[t] >= -3;
      }
    }
  }
  ok = __all_sync(full, ok);
  __syncwarp();
  if (ok) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int v = lane + 32 * k;
      if (v < n && v > 0) ok = ok && s.dep[v] == s.dep[s.par[v]] + 1;
    }
    ok = __all_sync(full, ok);
  }
  if (!ok) {
    if (lane == 0) {
      if (report) flag(status, SSM_STATUS_BAD_LAYOUT);
      s.nf = 0;
      s.nu = 0;
    }
    return;
  }
  const unsigned m0 = __ballot_sync(full, lane < n && s.dep[lane] == level);
  const unsigned m1 = __ballot_sync(full, lane + 32 < n && s.dep[lane + 32] == level);
  if ((m0 >> lane) & 1u) s.front[__popc(m0 & lt)] = lane;
  if ((m1 >> lane) & 1u) s.front[__popc(m0) + __popc(m1 & lt)] = lane + 32;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int v = lane + 32 * k;
    if (v < n && s.dep[v] == level)
      for (int u = v; u >= 0; u = s.par[u]) s.slot[u] = 0;  // same value from every lane
  }
  __syncwarp();
  const unsigned p0 = __ballot_sync(full, lane < n && s.slot[lane] >= 0);
  const unsigned p1 = __ballot_sync(full, lane + 32 < n && s.slot[lane + 32] >= 0);
  if ((p0 >> lane) & 1u) {
    const int sl = __popc(p0 & lt);
    s.slot[lane] = sl;
    s.snode[sl] = lane;
  }
  if ((p1 >> lane) & 1u) {
    const int sl = __popc(p0) + __popc(p1 & lt);
    s.slot[lane + 32] = sl;
    s.snode[sl] = lane + 32;
  }
  if (lane == 0) {
    s.nf = __popc(m0) + __popc(m1);
    s.nu = __popc(p0) + __popc(p1);
  }
}

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

constexpr int PG = 4;             // heads per prep CTA
constexpr int PROWS = PG * kP;    // 256 channels (x rows) per prep CTA
static_assert(2 * kN == TTHREADS, "one B | C channel per thread of the B | C kernel");

// Workspace of one instance (floats): C rows [n][kN], e^{S_v} [n][H], path sums [n][d_inner],
// B·C products [n][MAXP] (node v's row: B_{m_k} · C_v for its path nodes m_0 .. m_d = v),
// indexed by node; only the level's nodes are written.  Each section (and so each instance)
// starts on a 128-byte boundary, for the 16-byte vector accesses.
__host__ __device__ inline size_t ws_pad(size_t f) { return (f + 31) & ~(size_t)31; }
__host__ __device__ inline size_t ws_E_off(int n) { return ws_pad((size_t)n * kN); }
__host__ __device__ inline size_t ws_P_off(int n, int H) { return ws_E_off(n) + ws_pad((size_t)n * H); }
__host__ __device__ inline size_t ws_D_off(int n, int H) { return ws_P_off(n, H) + ws_pad((size_t)n * H * kP); }
__host__ __device__ inline size_t ws_floats_per_inst(int n, int H) { return ws_D_off(n, H) + ws_pad((size_t)n * MAXP); }

// pre-conv row of tap source src of one instance: an earlier node of the tree, or the ring row
// src positions before the committed head hm
__device__ __forceinline__ const uint16_t* tap_row_of(const uint16_t* xbc, const uint16_t* ring, int hm, int R,
                                                      int conv_dim, int src) {
  if (src >= 0) return xbc + (size_t)src * conv_dim;
  int p = hm + src;
  if (p < 0) p += R;
  return ring + (size_t)p * conv_dim;
}

// Shared-memory layout of draft_tree_bc_kernel (byte offsets, multiples of 128).
struct BcLayout {
  int Bu, Cf, pslot, plen, total;
};
__host__ __device__ inline BcLayout bc_layout(int n) {
  auto up = [](int b) { return (b + 127) & ~127; };
  BcLayout L;
  int o = up((int)sizeof(LevelSetup));
  L.Bu = o;    o += up(n * kN * 4);      // B, by slot
  L.Cf = o;    o += up(n * kN * 4);      // C, by position
  L.pslot = o; o += up(n * MAXP * 4);    // path slots, root first, by position
  L.plen = o;  o += up(n * 4);
  L.total = o;
  return L;
}

// Root-to-node paths of the level's nodes as slots (threads over positions).
__device__ __forceinline__ void level_paths(const LevelSetup& ls, int* pslot, int* plen) {
  for (int f = threadIdx.x; f < ls.nf; f += blockDim.x) {
    int u = ls.front[f];
    const int len = ls.dep[u] + 1;
    for (int k = len - 1; k >= 0; --k) {
      pslot[f * MAXP + k] = ls.slot[u];
      u = ls.par[u];
    }
    plen[f] = len;
  }
}

// One CTA per instance: the per-instance part of a level, done once rather than by each head
// block.  B of the ancestors (their logged values) and B | C of the level's nodes (four conv
// taps each, conv + SiLU; B logged), C rows to the workspace, then the B·C products along
// every level node's path.  Checks and reports the layout.
__global__ void __launch_bounds__(TTHREADS) draft_tree_bc_kernel(DraftTreeArgs a, float* ws) {
  extern __shared__ __align__(128) unsigned char smem[];
  LevelSetup& ls = *reinterpret_cast<LevelSetup*>(smem);
  const int n = a.n;
  const BcLayout Lo = bc_layout(n);
  float* Bu = reinterpret_cast<float*>(smem + Lo.Bu);
  float* Cf = reinterpret_cast<float*>(smem + Lo.Cf);
  int* pslot = reinterpret_cast<int*>(smem + Lo.pslot);
  int* plen = reinterpret_cast<int*>(smem + Lo.plen);
  // the head blocks may start once every CTA here runs; they wait for this grid's completion
  // before they read the products
  launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long inst = blockIdx.x;
  const int seq = (int)(inst / a.L), layer = (int)(inst % a.L);
  const int H = a.H, d_inner = H * kP, conv_dim = d_inner + 2 * kN;
  const size_t node0 = (size_t)inst * n;
  int hm = a.ring_head[inst] % a.R;
  if (hm < 0) hm += a.R;
  if (warp == 0) level_setup(ls, a.layout + (size_t)seq * n, n, a.level, a.status, true);
  __syncthreads();
  const int nf = ls.nf, nu = ls.nu, na = nu - nf;  // slots [0, na): the ancestors; then the level
  if (nf == 0) return;
  const uint16_t* xbc = a.xBC + node0 * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * a.R * conv_dim;
  const float4* cw4 = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const int cb = d_inner + tid;  // B (tid < kN) or C channel of this thread
  const float4 wb = cw4[cb];
  const float bb = a.conv_b[(size_t)layer * conv_dim + cb];
  float* wsi = ws + (size_t)inst * ws_floats_per_inst(n, H);
  // every load of a round in flight: B of 8 ancestors, four taps of 4 level nodes
  for (int r0 = 0; 8 * r0 < na || 4 * r0 < nf; ++r0) {
    float ab[8], lb[4][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int sl = 8 * r0 + i;
      if (sl < na && tid < kN) ab[i] = __ldg(a.log_B + (node0 + ls.snode[sl]) * kN + tid);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int f = 4 * r0 + i;
      if (f < nf) {
        const int v = ls.front[f];
        lb[i][0] = bf16f(__ldg(tap_row_of(xbc, ring, hm, a.R, conv_dim, ls.tap[v][2]) + cb));
        lb[i][1] = bf16f(__ldg(tap_row_of(xbc, ring, hm, a.R, conv_dim, ls.tap[v][1]) + cb));
        lb[i][2] = bf16f(__ldg(tap_row_of(xbc, ring, hm, a.R, conv_dim, ls.tap[v][0]) + cb));
        lb[i][3] = bf16f(__ldg(xbc + (size_t)v * conv_dim + cb));
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int sl = 8 * r0 + i;
      if (sl < na && tid < kN) Bu[sl * kN + tid] = ab[i];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int f = 4 * r0 + i;
      if (f < nf) {
        const int v = ls.front[f];
        const float val = conv4_silu(wb, bb, lb[i][0], lb[i][1], lb[i][2], lb[i][3]);
        if (tid < kN) {
          Bu[(na + f) * kN + tid] = val;
          a.log_B[(node0 + v) * kN + tid] = val;
        } else {
          Cf[f * kN + tid - kN] = val;
          wsi[(size_t)v * kN + tid - kN] = val;
        }
      }
    }
  }
  level_paths(ls, pslot, plen);
  __syncthreads();
  // B_{m_k} · C_v: one warp per (level node, path index)
  float* wsD = wsi + ws_D_off(n, H);
  for (int q = warp; q < nf * MAXP; q += TTHREADS / 32) {
    const int f = q / MAXP, k = q - f * MAXP;
    if (k >= plen[f]) continue;
    const float4 b4 = reinterpret_cast<const float4*>(Bu + pslot[f * MAXP + k] * kN)[lane];
    const float4 c4 = reinterpret_cast<const float4*>(Cf + f * kN)[lane];
    float d = b4.x * c4.x;
    d = fmaf(b4.y, c4.y, d);
    d = fmaf(b4.z, c4.z, d);
    d = fmaf(b4.w, c4.w, d);
    d = warp_sum(d);
    if (lane == 0) wsD[(size_t)ls.front[f] * MAXP + k] = d;
  }
}

struct PrepFixed {
  LevelSetup ls;
  float A[PG], Dh[PG];
};

// Shared-memory layout of draft_tree_prep_kernel for trees of n nodes (byte offsets, each a
// multiple of 128).  Slots index the nodes on the level's paths, positions the level's nodes.
struct PrepLayout {
  int xu, coef, du, su, pslot, plen, total;
};
__host__ __device__ inline PrepLayout prep_layout(int n) {
  auto up = [](int b) { return (b + 127) & ~127; };
  PrepLayout L;
  int o = up((int)sizeof(PrepFixed));
  L.xu = o;    o += up(n * PROWS * 4);       // x of the block's channels, by slot
  L.coef = o;  o += up(n * MAXP * PG * 4);   // e^{S_v − S_m} Δ_m (B_m · C_v), by position and path index
  L.du = o;    o += up(n * PG * 4);          // Δ, by slot
  L.su = o;    o += up(n * PG * 4);          // S = Σ Δ·A from the root, inclusive, by slot
  L.pslot = o; o += up(n * MAXP * 4);        // path slots, root first, by position
  L.plen = o;  o += up(n * 4);
  L.total = o;
  return L;
}

// One CTA per instance and block of 4 heads, launched as a dependent grid of
// draft_tree_bc_kernel: x of the block's channels for the ancestors (logged) and the level's
// nodes (conv + SiLU, logged), Δ (logged for the level), S along the paths; then, once the
// B·C products are complete, e^{S_v} and the path coefficients of its heads and the path sums
// of its rows.
__global__ void __launch_bounds__(TTHREADS, 3) draft_tree_prep_kernel(DraftTreeArgs a, float* ws) {
  extern __shared__ __align__(128) unsigned char smem[];
  PrepFixed& s = *reinterpret_cast<PrepFixed*>(smem);
  const int n = a.n;
  const PrepLayout Lo = prep_layout(n);
  float* xu = reinterpret_cast<float*>(smem + Lo.xu);
  float* coef = reinterpret_cast<float*>(smem + Lo.coef);
  float* du = reinterpret_cast<float*>(smem + Lo.du);
  float* su = reinterpret_cast<float*>(smem + Lo.su);
  int* pslot = reinterpret_cast<int*>(smem + Lo.pslot);
  int* plen = reinterpret_cast<int*>(smem + Lo.plen);
  // the level kernel may be scheduled once every prep CTA runs; it waits for this grid's
  // completion before it reads anything written here
  launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_blocks = (a.H + PG - 1) / PG;
  const int blk = blockIdx.x % n_blocks;
  const long long inst = blockIdx.x / n_blocks;
  const int seq = (int)(inst / a.L), layer = (int)(inst % a.L);
  const int h_begin = blk * PG, heads = min(PG, a.H - h_begin), rows = heads * kP;
  const int H = a.H, d_inner = H * kP, conv_dim = d_inner + 2 * kN;
  const size_t node0 = (size_t)inst * n;

  int hm = a.ring_head[inst] % a.R;  // ring position of the committed head (loaded with the layout)
  if (hm < 0) hm += a.R;
  if (warp == 0) level_setup(s.ls, a.layout + (size_t)seq * n, n, a.level, a.status, false);
  if (warp == 1 && lane < PG) {
    const bool on = lane < heads;
    s.A[lane] = on ? neg_exp(a.A_log[(size_t)layer * H + h_begin + lane]) : 0.f;
    s.Dh[lane] = on ? a.D[(size_t)layer * H + h_begin + lane] : 0.f;
  }
  __syncthreads();
  const int nf = s.ls.nf, nu = s.ls.nu, na = nu - nf;  // slots [0, na): the ancestors; then the level
  if (nf == 0) return;
  const uint16_t* xbc = a.xBC + node0 * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * a.R * conv_dim;

  // ---- x of the block's channels, in rounds with every load of a round in flight: 8
  // ancestors (one logged value each) and 4 level nodes (four taps each, through the conv +
  // SiLU, logged here); Δ for each slot ----
  {
    const float4* cw4 = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
    const float* cbv = a.conv_b + (size_t)layer * conv_dim;
    const bool live = tid < rows;
    const int cx = h_begin * kP + tid;  // x channel of this thread
    const float4 wx = live ? cw4[cx] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float bx = live ? cbv[cx] : 0.f;
    float dval = 0.f;  // Δ: one (slot, head) per thread
    int d_sl = -1, d_g = 0;
    bool d_conv = false;
    if (tid < nu * PG) {
      d_sl = tid / PG;
      d_g = tid - d_sl * PG;
      const int v = s.ls.snode[d_sl];
      if (d_g < heads) {
        const int h = h_begin + d_g;
        if (d_sl < na) {
          dval = __ldg(a.log_delta + (node0 + v) * H + h);
        } else {
          d_conv = true;
          dval = bf16f(__ldg(a.dt + (node0 + v) * H + h)) + a.dt_bias[(size_t)layer * H + h];
        }
      }
    }
    for (int r0 = 0; 8 * r0 < na || 4 * r0 < nf; ++r0) {
      float ax[8];     // ancestors 8 r0 .. 8 r0 + 7: logged x
      float lx[4][4];  // level nodes 4 r0 .. 4 r0 + 3: taps of x
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int sl = 8 * r0 + i;
        if (sl < na && live) ax[i] = __ldg(a.log_x + (node0 + s.ls.snode[sl]) * d_inner + cx);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = 4 * r0 + i;
        if (f < nf && live) {
          const int v = s.ls.front[f];
          lx[i][0] = bf16f(__ldg(tap_row_of(xbc, ring, hm, a.R, conv_dim, s.ls.tap[v][2]) + cx));
          lx[i][1] = bf16f(__ldg(tap_row_of(xbc, ring, hm, a.R, conv_dim, s.ls.tap[v][1]) + cx));
          lx[i][2] = bf16f(__ldg(tap_row_of(xbc, ring, hm, a.R, conv_dim, s.ls.tap[v][0]) + cx));
          lx[i][3] = bf16f(__ldg(xbc + (size_t)v * conv_dim + cx));
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int sl = 8 * r0 + i;
        if (sl < na) xu[sl * PROWS + tid] = live ? ax[i] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = 4 * r0 + i;
        if (f < nf) {
          float x = 0.f;
          if (live) {
            x = conv4_silu(wx, bx, lx[i][0], lx[i][1], lx[i][2], lx[i][3]);
            a.log_x[(node0 + s.ls.front[f]) * d_inner + cx] = x;
          }
          xu[(na + f) * PROWS + tid] = x;
        }
      }
    }
    if (d_sl >= 0) {
      if (d_conv) {
        dval = softplus_f(dval);
        a.log_delta[(node0 + s.ls.snode[d_sl]) * H + h_begin + d_g] = dval;
      }
      du[d_sl * PG + d_g] = dval;
    }
  }
  __syncthreads();
  // S of every slot (walking its path to the root) and each level node's path as slots
  for (int i = tid; i < nu * PG; i += TTHREADS) {
    const int sl = i / PG, g = i - sl * PG;
    float acc = 0.f;
    for (int u = s.ls.snode[sl]; u >= 0; u = s.ls.par[u]) acc = fmaf(du[s.ls.slot[u] * PG + g], s.A[g], acc);
    su[sl * PG + g] = acc;
  }
  level_paths(s.ls, pslot, plen);
  __syncthreads();
  float* wsi = ws + (size_t)inst * ws_floats_per_inst(n, H);
  float* wsE = wsi + ws_E_off(n);            // [n][H]
  float* wsP = wsi + ws_P_off(n, H);         // [n][d_inner]
  const float* wsD = wsi + ws_D_off(n, H);   // [n][MAXP], written by draft_tree_bc_kernel
  // e^{S_v}
  for (int i = tid; i < nf * PG; i += TTHREADS) {
    const int f = i / PG, g = i - f * PG;
    if (g < heads) wsE[(size_t)s.ls.front[f] * H + h_begin + g] = expf(su[pslot[f * MAXP + plen[f] - 1] * PG + g]);
  }
  grid_dependency_wait();  // the B·C products
  // path coefficients: one (node, path index, head) per thread
  for (int i = tid; i < nf * MAXP * PG; i += TTHREADS) {
    const int f = i / (MAXP * PG), r = i - f * (MAXP * PG), k = r / PG, g = r - k * PG;
    if (k >= plen[f]) continue;
    const int sm = pslot[f * MAXP + k], sv = pslot[f * MAXP + plen[f] - 1];
    coef[(f * MAXP + k) * PG + g] =
        expf(su[sv * PG + g] - su[sm * PG + g]) * du[sm * PG + g] * __ldcg(wsD + (size_t)s.ls.front[f] * MAXP + k);
  }
  __syncthreads();
  // path sums of the block's rows: Σ_k coef_k x_{m_k}[row] + D x_v[row]
  if (tid < rows) {
    const int g = tid / kP;
    for (int f = 0; f < nf; ++f) {
      const int len = plen[f];
      float b = 0.f;
      for (int k = 0; k < len; ++k) b = fmaf(coef[(f * MAXP + k) * PG + g], xu[pslot[f * MAXP + k] * PROWS + tid], b);
      b = fmaf(s.Dh[g], xu[pslot[f * MAXP + len - 1] * PROWS + tid], b);
      wsP[(size_t)s.ls.front[f] * d_inner + h_begin * kP + tid] = b;
    }
  }
}

// F partial sums per lane (F = 1, 2, 4 or 8), over the 8 lanes o = 0..7 of an aligned lane
// group: lane o ends with the full sum of value o mod F (full sums over the lane bits above
// log2 F, then recursive halving over the bits below).
template <int F>
__device__ __forceinline__ float reduce_rows(float (&v)[F], int o) {
  if constexpr (F == 8) {
    return reduce_scatter8(v, o);
  } else {
    constexpr int LOGF = F == 1 ? 0 : (F == 2 ? 1 : 2);
#pragma unroll
    for (int m = 4; m >= F; m >>= 1)  // lane bits that do not select a value: plain sums
#pragma unroll
      for (int i = 0; i < F; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], m);
    if constexpr (LOGF == 0) {
      return v[0];
    } else if constexpr (LOGF == 1) {
      const bool b0 = o & 1;
      const float keep = b0 ? v[1] : v[0];
      const float send = b0 ? v[0] : v[1];
      return keep + __shfl_xor_sync(0xffffffffu, send, 1);
    } else {
      const bool b1 = o & 2, b0 = o & 1;
      float s2[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float keep = b1 ? v[2 + i] : v[i];
        const float send = b1 ? v[i] : v[2 + i];
        s2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
      }
      const float keep = b0 ? s2[1] : s2[0];
      const float send = b0 ? s2[0] : s2[1];
      return keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
  }
}

constexpr int MTHREADS = 256;                    // level kernel: 8 lanes per row, 32 rows per sweep
constexpr int MSWEEPS = kP / (MTHREADS / 8);      // 2 sweeps cover one head's 64 rows
constexpr int MSTAGES = 3;                        // heads' state rows in flight per CTA

struct MainFixed {
  unsigned long long bar[MSTAGES];  // completion of each stage's state-row copy
  LevelSetup ls;
  int seq_ready;                    // the sequence whose layout ls holds
  int ok;                           // the current stage's copy has landed
  int issued;                       // items whose copies have been issued
};
__host__ __device__ inline int main_h_offset() { return (int)((sizeof(MainFixed) + 127) & ~(size_t)127); }
__host__ __device__ inline int level_smem_bytes() { return main_h_offset() + MSTAGES * kP * kN * 4; }

// One pass of the contraction for up to F level nodes (fc of them live) of one head: 8 lanes
// per state row, 16 columns each (rows rsub + 32 i), C rows through the cache; the lanes of a
// row end with one node's sum each, and lane o < fc writes y of node o.
template <int F>
__device__ __forceinline__ void level_pass(const DraftTreeArgs& a, const int* front, int fc, const float* hsm,
                                           const float* wsi, const float* wsE, const float* wsP, size_t node0, int hh) {
  const int tid = threadIdx.x, o = tid & 7, rsub = tid >> 3;
  const int H = a.H, d_inner = H * kP;
  float acc[MSWEEPS][F];
#pragma unroll
  for (int i = 0; i < MSWEEPS; ++i)
#pragma unroll
    for (int f = 0; f < F; ++f) acc[i][f] = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float4 hr[MSWEEPS];
#pragma unroll
    for (int i = 0; i < MSWEEPS; ++i) hr[i] = reinterpret_cast<const float4*>(hsm + (rsub + 32 * i) * kN)[o + 8 * j];
#pragma unroll
    for (int f = 0; f < F; ++f) {
      const float4 cc = f < fc ? __ldg(reinterpret_cast<const float4*>(wsi + (size_t)front[f] * kN) + o + 8 * j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < MSWEEPS; ++i) {
        acc[i][f] = fmaf(hr[i].x, cc.x, acc[i][f]);
        acc[i][f] = fmaf(hr[i].y, cc.y, acc[i][f]);
        acc[i][f] = fmaf(hr[i].z, cc.z, acc[i][f]);
        acc[i][f] = fmaf(hr[i].w, cc.w, acc[i][f]);
      }
    }
  }
  const bool writer = o < fc;
  const int v = writer ? front[o] : 0;
  const float e = writer ? __ldg(wsE + (size_t)v * H + hh) : 0.f;
#pragma unroll
  for (int i = 0; i < MSWEEPS; ++i) {
    const int row = rsub + 32 * i;
    const float sum = reduce_rows<F>(acc[i], o);
    if (writer) {
      const size_t yo = (node0 + v) * d_inner + (size_t)hh * kP + row;
      a.y[yo] = fmaf(e, sum, __ldg(wsP + (size_t)v * d_inner + (size_t)hh * kP + row));
    }
  }
}

// Persistent: CTA c takes the contiguous run of (instance, head) items
// [c·items/G, (c+1)·items/G), G = the grid, and keeps the next MSTAGES heads' 64 state rows in
// flight (bulk copies into a ring of shared-memory stages, one mbarrier each) while it
// computes the current one, so the memory pipe never waits for the compute.
__global__ void __launch_bounds__(MTHREADS, 2) draft_tree_level_kernel(DraftTreeArgs a, const float* ws) {
  extern __shared__ __align__(128) unsigned char smem[];
  MainFixed& s = *reinterpret_cast<MainFixed*>(smem);
  float* stages = reinterpret_cast<float*>(smem + main_h_offset());
  const int n = a.n;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H;
  const long long items = (long long)a.n_seq * a.L * H;
  const long long it0 = blockIdx.x * items / gridDim.x, it1 = (blockIdx.x + 1) * items / gridDim.x;
  const int count = (int)(it1 - it0);
  constexpr uint32_t kBytes = kP * kN * 4;

  auto issue = [&](int k) {  // the k-th item of this CTA into stage k mod MSTAGES
    const long long it = it0 + k;
    const uint32_t bar = smem_u32(&s.bar[k % MSTAGES]);
    mbar_arrive_expect_tx(bar, kBytes);
    bulk_load(smem_u32(stages + (size_t)(k % MSTAGES) * kP * kN), a.h + (size_t)it * kP * kN, kBytes, bar);
  };
  if (tid == 0) {
    for (int st = 0; st < MSTAGES; ++st) mbar_init(smem_u32(&s.bar[st]), 1);
    fence_barrier_init();
    for (int k = 0; k < MSTAGES && k < count; ++k) issue(k);
    s.issued = count < MSTAGES ? count : MSTAGES;
    s.seq_ready = -1;
  }
  __syncthreads();
  grid_dependency_wait();  // the prep grid's workspace rows and log rows
  int k_fail = -1;
  for (int k = 0; k < count; ++k) {
    const long long it = it0 + k;
    const long long inst = it / H;
    const int hh = (int)(it - inst * H);
    const int seq = (int)(inst / a.L);
    if (seq != s.seq_ready) {  // this sequence's level nodes (uniform across the CTA)
      __syncthreads();
      if (warp == 0) {
        level_setup(s.ls, a.layout + (size_t)seq * n, n, a.level, a.status, false);
        if (tid == 0) s.seq_ready = seq;
      }
      __syncthreads();
    }
    const int nf = s.ls.nf;
    const float* hsm = stages + (size_t)(k % MSTAGES) * kP * kN;
    if (tid == 0) s.ok = mbar_wait(smem_u32(&s.bar[k % MSTAGES]), (uint32_t)((k / MSTAGES) & 1));
    __syncthreads();
    if (!s.ok) {  // uniform across the CTA
      k_fail = k;
      break;
    }
    const size_t node0 = (size_t)inst * n;
    const float* wsi = ws + (size_t)inst * ws_floats_per_inst(n, H);
    const float* wsE = wsi + ws_E_off(n);
    const float* wsP = wsi + ws_P_off(n, H);
    // y_v = e^{S_v} (C_v · h_ckpt) + path sum, up to 8 level nodes per pass, the pass's
    // arithmetic sized to its node count (1, 2, 4 or 8)
    for (int f0 = 0; f0 < nf; f0 += FB) {
      const int fc = min(FB, nf - f0);
      if (fc == 1)
        level_pass<1>(a, s.ls.front + f0, fc, hsm, wsi, wsE, wsP, node0, hh);
      else if (fc == 2)
        level_pass<2>(a, s.ls.front + f0, fc, hsm, wsi, wsE, wsP, node0, hh);
      else if (fc <= 4)
        level_pass<4>(a, s.ls.front + f0, fc, hsm, wsi, wsE, wsP, node0, hh);
      else
        level_pass<8>(a, s.ls.front + f0, fc, hsm, wsi, wsE, wsP, node0, hh);
    }
    __syncthreads();  // every thread is done with this stage
    if (tid == 0 && k + MSTAGES < count) {
      issue(k + MSTAGES);
      s.issued = k + MSTAGES + 1;
    }
  }
  if (k_fail >= 0 && tid == 0) {  // give the copies still in flight a last bounded wait before exiting
    flag(a.status, SSM_STATUS_TIMEOUT);
    for (int kk = k_fail; kk < s.issued; ++kk) mbar_wait(smem_u32(&s.bar[kk % MSTAGES]), (uint32_t)((kk / MSTAGES) & 1));
  }
}

// ---------------------------------------------------------------------------
// commit of the accepted path from the log
// ---------------------------------------------------------------------------
constexpr int CH = 1;               // heads per CTA
constexpr int CROWS = CH * kP;      // 64 state rows, 16 per warp
constexpr int CTHREADS = 128;
constexpr int CT = 16;              // path nodes per pass

// Length of the valid prefix of a sequence's accepted path (path[0] = 0, then each entry a
// child of the one before, at most max_path entries), checked by a whole warp at once;
// anything else is flagged when `report`.  Every lane returns the same value.
__device__ int tree_path_len(const DraftTreeCommitArgs& a, int seq, bool report) {
  const int lane = threadIdx.x & 31;
  int len = a.path_len[seq];
  bool bad = false;
  if (len < 0 || len > a.max_path) {
    bad = true;
    len = len < 0 ? 0 : a.max_path;
  }
  const int32_t* p = a.path + (size_t)seq * a.max_path;
  const ssm_node* lay = a.layout + (size_t)seq * a.n;
  int good = len;
  for (int base = 0; base < len; base += 32) {
    const int j = base + lane;
    bool ok = true;
    if (j < len) {
      const int v = p[j];
      if (j == 0) {
        ok = v == 0;
      } else {
        const int prev = p[j - 1];
        ok = v > prev && prev >= 0 && v < a.n && lay[v].parent == prev;
      }
    }
    const unsigned fail = __ballot_sync(0xffffffffu, !ok);
    if (fail) {
      good = base + __ffs(fail) - 1;
      bad = true;
      break;
    }
  }
  if (bad && report && lane == 0) flag(a.status, SSM_STATUS_PATH_RANGE);
  return good;
}

__global__ void __launch_bounds__(CTHREADS, 4) draft_tree_commit_kernel(DraftTreeCommitArgs a) {
  __shared__ float us[CT][CROWS];  // Δ_t·x_t[row]
  __shared__ float decs[CT][CH];
  __shared__ __align__(16) float Bs[CT][kN];
  __shared__ int nodes[SSM_MAX_PATH];
  __shared__ int s_len;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_groups = (a.H + CH - 1) / CH;
  const int grp = blockIdx.x % n_groups;
  const long long inst = blockIdx.x / n_groups;
  const int seq = (int)(inst / a.L), layer = (int)(inst % a.L);
  const int h_begin = grp * CH, heads = min(CH, a.H - h_begin), rows = heads * kP;
  const int d_inner = a.H * kP;
  const size_t node0 = (size_t)inst * a.n;
  float* hs = a.h + ((size_t)inst * a.H + h_begin) * kP * kN;
  const int row0 = warp * (CROWS / (CTHREADS / 32));
  const int g = row0 / kP;
  const bool mine = g < heads;
  // the warp's 16 rows, all in flight while the path is checked and the log staged
  float4 hr[16];
  if (mine) {
#pragma unroll
    for (int r = 0; r < 16; ++r) hr[r] = reinterpret_cast<const float4*>(hs + (size_t)(row0 + r) * kN)[lane];
  }
  if (warp == 0) {
    const int len = tree_path_len(a, seq, grp == 0 && layer == 0);
    for (int j = lane; j < len; j += 32) nodes[j] = a.path[(size_t)seq * a.max_path + j];
    if (lane == 0) s_len = len;
  }
  __syncthreads();
  const int len = s_len;
  if (len == 0) return;
  const float A_g = neg_exp(a.A_log[(size_t)layer * a.H + h_begin + min(tid % CH, heads - 1)]);
  for (int t0 = 0; t0 < len; t0 += CT) {
    const int cnt = min(CT, len - t0);
    if (t0 > 0) __syncthreads();  // the previous pass is done with us, decs, Bs
    // every log value of the pass in flight at once: Δ and x for (row, step) pairs, B rows,
    // then the products and decays into shared memory
    static_assert(CTHREADS == 2 * CROWS, "two threads per row, each half of the steps");
    const int r = tid % CROWS, th = tid / CROWS;
    float dl[CT / 2], xv[CT / 2];
#pragma unroll
    for (int j = 0; j < CT / 2; ++j) {
      const int t = th + 2 * j;
      dl[j] = 0.f;
      xv[j] = 0.f;
      if (t < cnt && r < rows) {
        const size_t lr = node0 + nodes[t0 + t];
        dl[j] = a.log_delta[lr * a.H + h_begin + r / kP];
        xv[j] = a.log_x[lr * d_inner + h_begin * kP + r];
      }
    }
    float4 bv[CT * (kN / 4) / CTHREADS];
#pragma unroll
    for (int q = 0; q < CT * (kN / 4) / CTHREADS; ++q) {
      const int i = tid + q * CTHREADS, t = i / (kN / 4), c4 = i - t * (kN / 4);
      bv[q] = t < cnt ? reinterpret_cast<const float4*>(a.log_B + (node0 + nodes[t0 + t]) * kN)[c4]
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float dd = 0.f;
    const int dt_ = tid / CH, dg = tid - dt_ * CH;
    if (tid < cnt * CH && dg < heads) dd = a.log_delta[(node0 + nodes[t0 + dt_]) * a.H + h_begin + dg];
#pragma unroll
    for (int j = 0; j < CT / 2; ++j) {
      const int t = th + 2 * j;
      if (t < cnt) us[t][r] = __fmul_rn(dl[j], xv[j]);
    }
#pragma unroll
    for (int q = 0; q < CT * (kN / 4) / CTHREADS; ++q) {
      const int i = tid + q * CTHREADS, t = i / (kN / 4), c4 = i - t * (kN / 4);
      reinterpret_cast<float4*>(Bs[t])[c4] = bv[q];
    }
    if (tid < cnt * CH) decs[dt_][dg] = dg < heads ? decay_of(dd, A_g) : 1.f;
    __syncthreads();
    if (mine) apply_logged_updates(hr, cnt, &us[0][0], CROWS, row0, &Bs[0][0], &decs[0][g], CH, lane);
  }
  if (mine) {
#pragma unroll
    for (int r = 0; r < 16; ++r) reinterpret_cast<float4*>(hs + (size_t)(row0 + r) * kN)[lane] = hr[r];
  }
}

// the path's last three pre-conv rows into the ring, head += len
__global__ void draft_tree_ring_kernel(DraftTreeCommitArgs a) {
  __shared__ int s_len, s_head, rows3[3];
  const long long inst = blockIdx.x;
  const int seq = (int)(inst / a.L);
  const int conv_dim = a.H * kP + 2 * kN;
  if (threadIdx.x < 32) {
    const int len = tree_path_len(a, seq, false);
    if (threadIdx.x == 0) {
      s_len = len;
      s_head = a.ring_head[inst];
      for (int j = 0; j < 3; ++j) {
        const int jj = len - 3 + j;
        rows3[j] = jj >= 0 ? a.path[(size_t)seq * a.max_path + jj] : -1;
      }
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

size_t draft_tree_workspace_bytes(int n, int H, long long n_inst) {
  return (size_t)n_inst * ws_floats_per_inst(n, H) * sizeof(float);
}

cudaError_t launch_draft_tree_level(const DraftTreeArgs& a, void* workspace, cudaStream_t s) {
  const long long inst = (long long)a.n_seq * a.L;
  if (inst == 0) return cudaSuccess;
  float* ws = static_cast<float*>(workspace);
  // programmatic dependent launch: each grid may be scheduled while the one before it runs,
  // and waits for it before reading what it writes
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int bsmem = bc_layout(a.n).total;
  cudaError_t e = cudaFuncSetAttribute(draft_tree_bc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bsmem);
  if (e != cudaSuccess) return e;
  draft_tree_bc_kernel<<<(unsigned)inst, TTHREADS, bsmem, s>>>(a, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int n_blocks = (a.H + PG - 1) / PG;
  const int psmem = prep_layout(a.n).total;
  e = cudaFuncSetAttribute(draft_tree_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3((unsigned)(inst * n_blocks));
  pcfg.blockDim = dim3(TTHREADS);
  pcfg.dynamicSmemBytes = (size_t)psmem;
  pcfg.stream = s;
  pcfg.attrs = attr;
  pcfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&pcfg, draft_tree_prep_kernel, a, ws)) != cudaSuccess) return e;
  const int smem = level_smem_bytes();
  e = cudaFuncSetAttribute(draft_tree_level_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long items = inst * a.H;
  const long long grid = items < 2LL * sms ? items : 2LL * sms;  // persistent: two CTAs per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(MTHREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cfg.attrs = attr;  // may start while the prep runs
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, draft_tree_level_kernel, a, static_cast<const float*>(ws));
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
