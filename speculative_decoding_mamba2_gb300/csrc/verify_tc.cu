// Tree verification with the state contraction on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory).
//
// Method: SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践") §3.2 (FIFO tree
// verification: every node continues from its parent's state) and §3.1 (the target
// recomputes only the accepted path); the Mamba2 update (LightMamba page, "为什么 Mamba 难加速":
// Ā·h_{t-1} + B̄·X) is linear in h, so for node v with root-to-node path P(v)
//     y_v[p] = e^{S_v}·(C_v·h[p,:]) + Σ_{m ∈ P(v)} e^{S_v - S_m}·Δ_m·(C_v·B_m)·x_m[p] + D·x_v[p],
//     S_v = Σ_{m ∈ P(v)} Δ_m·A,
// and the commit of the previous step's accepted path m_0..m_{len-1} is the rank-len update
//     h' = E·h + Σ_j u_j ⊗ B_j,  E = Π_j a_j,  u_j = Δ_j·(Π_{i>j} a_i)·x_j,  a_j = exp(Δ_j·A).
// Per-node states are never formed; the state is read once (and, with the commit, written
// once) per call.
//
// The contraction runs on the state as it was read (before the commit), using
//     C_v·h'[p,:] = E·(C_v·h[p,:]) + Σ_j u_j[p]·(C_v·B_j),
// so it never waits for the commit's update; h' itself is formed only for the store.
//
// Two kernels.
//  * tc_prep_kernel, one CTA per (instance, block of 16 heads): the B | C conv + SiLU of the
//    tree, the ancestor table and the products C_v·B_m along every path (every block, they are
//    cheap); for its heads Δ, S, e^S, the path coefficients e^{S_v - S_m}·Δ_m·(C_v·B_m) (+ D on
//    the node's own term) and, with a folded commit, E and w_j.  Block 0 also writes C split
//    into bf16 hi + lo in the tensor cores' K-major layout and, with a folded commit, the path
//    check, the path's post-conv B rows (split, K-major), the products C_v·B_j, the conv ring's
//    B | C channels and the ring head.  Everything goes to a per-instance workspace record.
//  * tc_verify_kernel, persistent (two CTAs per SM when shared memory allows), walks a
//    contiguous run of (instance, head pair) items.  A head pair is 128 state rows, the
//    MMA's M and the TMEM lanes.  Warp roles:
//      - warps 0-3, thread = state row (and x channel): the x conv + SiLU of its channel (and
//        u_j), then per 16-column state chunk: the chunk split into bf16 hi + lo as the MMA's A
//        tile, and with a folded commit h' = E·h + (U·Bᵀ)[row, chunk] (U·Bᵀ from TMEM) stored
//        over h; at the end of the item y_v = e^{S_v}·(E·D[row, v] + Σ_j u_j·C_v·B_j) + path
//        terms, with D read from TMEM;
//      - warp 4 (one lane): bulk tensor copies (TMA, 64-byte swizzle) of the state chunks
//        into a ring of stages, the item's x rows and per-head rows, and the instance's tables;
//      - warp 5 (one lane): the MMAs.  Per item U·Bᵀ (128 x 128 x 16, three products) into
//        TMEM, and per chunk D[128 x NP] += A·Cᵀ (three products hi·hi + hi·lo + lo·hi of
//        bf16 splits, fp32 accumulation; each product to ~2^-17 relative).  NP = nodes
//        rounded up to 16 (<= 64), so the whole tree's C·h comes from one pass over the state.
// Every wait on an mbarrier is bounded (one second of global time); a role that gives up
// sets SSM_STATUS_TIMEOUT, the others see the abort flag or time out in turn, and copies
// in flight get a bounded chance to land before the CTA leaves.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

namespace ssmtree {

namespace {

constexpr int ROWS = 128;                 // state rows per item: a head pair
constexpr int KC = 16;                    // state columns per chunk (one bf16 k-step)
constexpr int NCH = kN / KC;              // chunks per item
constexpr int AS = 2;                     // A-tile slots
constexpr int EW = 4;                     // element warps
constexpr int THREADS = (EW + 2) * 32;    // + producer warp + MMA warp
constexpr int PRODUCER_WARP = EW, MMA_WARP = EW + 1;
constexpr int DMAX = SSM_MAX_DEPTH + 1;
constexpr int XW = 2 * kP;                // x channels staged per item
constexpr int PREP_THREADS = 256;
constexpr int BCW = 2 * kN;               // B | C channels
constexpr uint32_t A_LBO = 128, A_SBO = 256;          // [128 x 16] bf16 tiles
constexpr uint32_t C_LBO = 128, C_SBO = 128 * (kN / 8);  // [NP x 128] bf16 C table
constexpr int A_TILE = ROWS * KC * 2;     // 4 KB
constexpr int BT_TILE = kN * 16 * 2;      // [128 state columns x 16 path slots] bf16, 4 KB
constexpr int kMeta = 20;                 // [0] path length, [1] ring head before it, [4..19] path nodes
constexpr int SMEM_CAP = 232448;
constexpr int TWO_PER_SM = 113 * 1024;    // a plan at most this large fits twice on an SM
constexpr int MIN_TWO = 80 * 1024;        // ... and at least this large never three times (TMEM is split in two)

__host__ __device__ constexpr int np_of(int n) { return (n + 15) & ~15; }

// ---------------------------------------------------------------------------
// per-instance workspace record (byte offsets, each section 128-byte aligned)
// ---------------------------------------------------------------------------
constexpr int HB = 16;     // heads per prep block
constexpr int EWS = 20;    // per head: E, then w_j (j < 16), padded
__host__ __device__ inline int pp_of(int n, int max_depth) { return (n * (max_depth + 1) + 3) & ~3; }

struct TcWs {
  int PP;
  size_t Ct, Bt, Gp, pathn, poff, meta, eS, coef, EW, stride;
};
__host__ __device__ inline TcWs tc_ws(int n, int max_depth, int H, int LP) {
  TcWs w;
  w.PP = pp_of(n, max_depth);
  const int NP = np_of(n);
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t r = o;
    o += (b + 127) & ~size_t(127);
    return r;
  };
  w.Ct = take((size_t)2 * NP * kN * 2);           // C hi, then C lo: K-major [NP][128] bf16
  w.Bt = take(LP > 0 ? 2 * BT_TILE : 0);          // path B hi, then lo: K-major [128][16] bf16
  w.Gp = take(LP > 0 ? (size_t)16 * NP * 4 : 0);  // C_v·B_j  [16][NP]
  w.pathn = take((size_t)n * DMAX * 4);           // ancestor of v at depth j  [n][DMAX]
  w.poff = take((size_t)n * 4);                   // first path pair of node v [n]
  w.meta = take(LP > 0 ? kMeta * 4 : 0);
  w.eS = take((size_t)H * NP * 4);                // e^{S_v}  [H][NP]
  w.coef = take((size_t)H * w.PP * 4);            // path coefficients [H][PP], pair poff[v] + j
  w.EW = take(LP > 0 ? (size_t)H * EWS * 4 : 0);  // E, w_j  [H][EWS]
  w.stride = o;
  return w;
}

// Validated copy of a layout record (bad fields are clamped and reported).
__device__ ssm_node tc_checked_node(const ssm_node* lay, int v, int max_depth, int32_t* status) {
  ssm_node r = lay[v];
  bool bad = false;
  if (v == 0) {
    bad |= r.parent != -1 || r.depth != 0;
    r.parent = -1;
    r.depth = 0;
  } else if (r.parent < 0 || r.parent >= v) {
    bad = true;
    r.parent = 0;
  }
  if (r.depth < 0 || r.depth > max_depth) {
    bad = true;
    r.depth = r.depth < 0 ? 0 : max_depth;
  }
  for (int d = 0; d < 3; ++d)
    if (r.tap[d] >= v || r.tap[d] < -3) {
      bad = true;
      r.tap[d] = -1;
    }
  if (bad) flag(status, SSM_STATUS_BAD_LAYOUT);
  return r;
}

// ---------------------------------------------------------------------------
// prep: one CTA per (instance, block of HB heads)
// ---------------------------------------------------------------------------
struct PrepLayout {
  int nodes, pathn, poff, xin, Bs, Cs, Gm, Bj, dl, Sv, pp, total;
};
__host__ __device__ inline PrepLayout tc_prep_layout(int n, int PP) {
  PrepLayout s;
  int o = 0;
  auto take = [&](int b) {
    const int r = o;
    o += (b + 15) & ~15;
    return r;
  };
  s.nodes = take(n * (int)sizeof(ssm_node));
  s.pathn = take(n * DMAX * 4);
  s.poff = take(n * 4);
  s.xin = take((n + 3) * BCW * 2);
  s.Bs = take(n * kN * 4);
  s.Cs = take(n * kN * 4);
  s.Gm = take(PP * 4);
  s.Bj = take(16 * kN * 4);
  s.dl = take(n * HB * 4);
  s.Sv = take(n * HB * 4);
  s.pp = take(kMeta * 4);
  s.total = o;
  return s;
}

__global__ void __launch_bounds__(PREP_THREADS) tc_prep_kernel(VerifyArgs a, unsigned char* __restrict__ ws_base) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int n = a.n, H = a.H, NP = np_of(n);
  const bool fuse = a.LP > 0;
  const TcWs W = tc_ws(n, a.max_depth, H, a.LP);
  const PrepLayout L = tc_prep_layout(n, W.PP);
  ssm_node* nodes = reinterpret_cast<ssm_node*>(smem + L.nodes);
  int* pathn = reinterpret_cast<int*>(smem + L.pathn);
  int* poff = reinterpret_cast<int*>(smem + L.poff);
  uint16_t* xin = reinterpret_cast<uint16_t*>(smem + L.xin);
  float* Bs = reinterpret_cast<float*>(smem + L.Bs);
  float* Cs = reinterpret_cast<float*>(smem + L.Cs);
  float* Gm = reinterpret_cast<float*>(smem + L.Gm);
  float* Bj = reinterpret_cast<float*>(smem + L.Bj);
  float* dl = reinterpret_cast<float*>(smem + L.dl);
  float* Sv = reinterpret_cast<float*>(smem + L.Sv);
  int* pp = reinterpret_cast<int*>(smem + L.pp);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  launch_dependents();  // the main kernel may be scheduled; it waits for this grid before reading its output
  const int nhb = (H + HB - 1) / HB;
  const int inst = blockIdx.x / nhb, hb = blockIdx.x % nhb;
  const int seq = inst / a.L, layer = inst % a.L;
  const int h0 = hb * HB, nh = min(HB, H - h0);
  const bool lead = hb == 0;  // writes what every head shares
  const int d_inner = H * kP, conv_dim = d_inner + BCW, R = a.R;
  const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  const uint16_t* prev_xbc = fuse ? a.prev_xBC + (size_t)inst * a.prev_n * conv_dim : nullptr;
  unsigned char* ws = ws_base + (size_t)inst * W.stride;
  int32_t* status = lead ? a.status : nullptr;  // one block reports the instance's bad inputs

  for (int i = tid; i < n * (BCW / 8); i += PREP_THREADS) {  // the tree's B | C rows (staged rows 3..n+2)
    const int r = 3 + i / (BCW / 8), pc = i % (BCW / 8);
    cp_async16(xin + r * BCW + pc * 8, xbc + (size_t)(r - 3) * conv_dim + d_inner + pc * 8);
  }
  const ssm_node* lay = a.layout + (size_t)seq * n;
  const int t0 = fuse ? 32 : 0;
  if (tid >= t0)
    for (int v = tid - t0; v < n; v += PREP_THREADS - t0) nodes[v] = tc_checked_node(lay, v, a.max_depth, status);
  if (fuse && tid < 32) {
    // the committed path, checked as the stand-alone commit checks it: root first, then each node
    // a child of the one before; it ends at the first bad entry (a bad root commits node 0)
    const int32_t* pth = a.prev_path + (size_t)seq * a.LP;
    int len = a.prev_path_len[seq];
    const bool bad_len = len < 1 || len > a.LP;
    len = len < 1 ? 1 : (len > a.LP ? a.LP : len);
    const int v = lane < len ? pth[lane] : 0;
    const int before = __shfl_up_sync(0xffffffffu, v, 1);
    bool ok = true;
    if (lane < len)
      ok = lane == 0 ? v == 0
                     : (v > before && v >= 1 && v < a.prev_n && a.prev_layout[(size_t)seq * a.prev_n + v].parent == before);
    const unsigned badm = __ballot_sync(0xffffffffu, lane < len && !ok);
    const int good = badm ? __ffs(badm) - 1 : len;
    if (lane < 16) pp[4 + lane] = lane < good ? v : 0;
    if (lane == 0) {
      pp[0] = good < 1 ? 1 : good;
      pp[1] = a.ring_head[inst];
      pp[2] = pp[3] = 0;
      if (bad_len || badm) flag(status, SSM_STATUS_PATH_RANGE);
    }
  }
  __syncthreads();
  const int lenP = fuse ? pp[0] : 0;
  const int head_old = fuse ? pp[1] : a.ring_head[inst];
  // the three rows before the root: after the commit, the path's last rows, then the ring rows
  // that preceded the path
  for (int i = tid; i < 3 * (BCW / 8); i += PREP_THREADS) {
    const int r = i / (BCW / 8), pc = i % (BCW / 8);
    const int k = 3 - r;  // k-th row before the root
    const uint16_t* src = k <= lenP ? prev_xbc + (size_t)pp[4 + lenP - k] * conv_dim
                                    : ring + (size_t)ring_pos(head_old, lenP - k, R) * conv_dim;
    cp_async16(xin + r * BCW + pc * 8, src + d_inner + pc * 8);
  }
  cp_async_commit();
  for (int v = tid; v < n; v += PREP_THREADS) {  // ancestor of v at every depth; first pair of v
    int m = v;
    for (int j = nodes[v].depth; j >= 0; --j) {
      pathn[v * DMAX + j] = m;
      m = m > 0 ? nodes[m].parent : 0;
    }
    for (int j = nodes[v].depth + 1; j < DMAX; ++j) pathn[v * DMAX + j] = 0;
    int off = 0;
    for (int u = 0; u < v; ++u) off += nodes[u].depth + 1;
    poff[v] = off;
  }
  // this block's Δ per (node, head); with a folded commit the path's Δ_j, decays, E and w_j
  float* EWg = reinterpret_cast<float*>(ws + W.EW);
  for (int i = tid; i < n * nh; i += PREP_THREADS) {
    const int v = i / nh, hl = i - v * nh, h = h0 + hl;
    dl[v * HB + hl] = softplus_f(bf16f(a.dt[((size_t)inst * n + v) * H + h]) + a.dt_bias[(size_t)layer * H + h]);
  }
  if (fuse && tid < nh) {
    const int h = h0 + tid;
    const size_t ph = (size_t)layer * H + h;
    const float A = neg_exp(a.A_log[ph]), bias = a.dt_bias[ph];
    float dj[16], aj[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      dj[j] = 0.f;
      aj[j] = 1.f;
      if (j < lenP) {
        dj[j] = softplus_f(bf16f(a.prev_dt[((size_t)inst * a.prev_n + pp[4 + j]) * H + h]) + bias);
        aj[j] = decay_of(dj[j], A);
      }
    }
    float* ew = EWg + (size_t)h * EWS;
    float run = 1.f;
#pragma unroll
    for (int j = 15; j >= 0; --j) {
      ew[1 + j] = dj[j] * run;  // w_j = Δ_j·Π_{i>j} a_i (0 past the path)
      run *= aj[j];
    }
    ew[0] = run;  // E
  }
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float4 w = cw[d_inner + tid];
  const float bb = a.conv_b[(size_t)layer * conv_dim + d_inner + tid];
  cp_async_wait<0>();
  __syncthreads();
  {  // B and C conv + SiLU: thread = channel of B | C, four nodes at a time
    float* dst = tid < kN ? Bs + tid : Cs + (tid - kN);
    const uint16_t* xi = xin + tid;
    int v = 0;
    for (; v + 4 <= n; v += 4) {
      float r[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const ssm_node& nd = nodes[v + u];
        r[u][0] = bf16f(xi[(nd.tap[2] + 3) * BCW]);
        r[u][1] = bf16f(xi[(nd.tap[1] + 3) * BCW]);
        r[u][2] = bf16f(xi[(nd.tap[0] + 3) * BCW]);
        r[u][3] = bf16f(xi[(v + u + 3) * BCW]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) dst[(v + u) * kN] = silu_fast(conv4_acc(w, bb, r[u][0], r[u][1], r[u][2], r[u][3]));
    }
    for (; v < n; ++v) {
      const ssm_node& nd = nodes[v];
      dst[v * kN] = silu_fast(conv4_acc(w, bb, bf16f(xi[(nd.tap[2] + 3) * BCW]), bf16f(xi[(nd.tap[1] + 3) * BCW]),
                                        bf16f(xi[(nd.tap[0] + 3) * BCW]), bf16f(xi[(v + 3) * BCW])));
    }
  }
  // S_v of this block's heads (path sums of Δ·A, root first)
  for (int i = tid; i < n * nh; i += PREP_THREADS) {
    const int v = i / nh, hl = i - v * nh;
    const float A = neg_exp(a.A_log[(size_t)layer * H + h0 + hl]);
    float s = 0.f;
    for (int j = 0; j <= nodes[v].depth; ++j) s = fmaf(dl[pathn[v * DMAX + j] * HB + hl], A, s);
    Sv[v * HB + hl] = s;
    reinterpret_cast<float*>(ws + W.eS)[(size_t)(h0 + hl) * NP + v] = expf(s);
  }
  __syncthreads();
  // Gm[poff[v] + j] = C_v · B_{ancestor at depth j}: one warp per pair
  for (int v = 0; v < n; ++v)
    for (int j = warp; j <= nodes[v].depth; j += PREP_THREADS / 32) {
      const float4 c4 = reinterpret_cast<const float4*>(Cs + v * kN)[lane];
      const float4 b4 = reinterpret_cast<const float4*>(Bs + pathn[v * DMAX + j] * kN)[lane];
      float s = c4.x * b4.x;
      s = fmaf(c4.y, b4.y, s);
      s = fmaf(c4.z, b4.z, s);
      s = fmaf(c4.w, b4.w, s);
      s = warp_sum(s);
      if (lane == 0) Gm[poff[v] + j] = s;
    }
  __syncthreads();
  {  // coefficients of this block's heads: coef[h][poff[v] + j] = e^{S_v - S_m}·Δ_m·(C_v·B_m), m the
     // ancestor at depth j, + D on the node's own term; zero in the padding
    float* cg = reinterpret_cast<float*>(ws + W.coef);
    const int npair = poff[n - 1] + nodes[n - 1].depth + 1;
    for (int i = tid; i < W.PP * nh; i += PREP_THREADS) {
      const int hl = i / W.PP, k = i - hl * W.PP, h = h0 + hl;
      float c = 0.f;
      if (k < npair) {
        int v = 0;  // node of pair k
        while (v + 1 < n && poff[v + 1] <= k) ++v;
        const int j = k - poff[v], m = pathn[v * DMAX + j];
        c = expf(Sv[v * HB + hl] - Sv[m * HB + hl]) * dl[m * HB + hl] * Gm[k];
        if (j == nodes[v].depth) c += a.D[(size_t)layer * H + h];
      }
      cg[(size_t)h * W.PP + k] = c;
    }
  }
  if (!lead) return;

  {  // C as bf16 hi + lo in the K-major layout of the MMA's B operand: 16-byte pieces of 8 columns
    unsigned char* chi = ws + W.Ct;
    unsigned char* clo = chi + (size_t)NP * kN * 2;
    for (int i = tid; i < NP * (kN / 8); i += PREP_THREADS) {
      const int v = i / (kN / 8), k0 = (i % (kN / 8)) * 8;
      uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
      if (v < n)
        for (int e = 0; e < 4; ++e) split_bf16x2(Cs[v * kN + k0 + 2 * e], Cs[v * kN + k0 + 2 * e + 1], hi[e], lo[e]);
      const uint32_t off = kmajor_off(v, k0, C_LBO, C_SBO);
      *reinterpret_cast<uint4*>(chi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(clo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    int* dp = reinterpret_cast<int*>(ws + W.pathn);
    for (int i = tid; i < n * DMAX; i += PREP_THREADS) dp[i] = pathn[i];
    int* dq = reinterpret_cast<int*>(ws + W.poff);
    for (int i = tid; i < n; i += PREP_THREADS) dq[i] = poff[i];
  }
  if (!fuse) return;

  // ---- the committed path: post-conv B rows (window = ring rows before it ‖ path rows) ----
  {
    const float* cbias = a.conv_b + (size_t)layer * conv_dim;
    auto window_row = [&](int t) -> const uint16_t* {
      return t < 3 ? ring + (size_t)ring_pos(head_old, t - 3, R) * conv_dim : prev_xbc + (size_t)pp[4 + t - 3] * conv_dim;
    };
    if (tid < kN) {
      const int c = d_inner + tid;
      const float4 wk = cw[c];
      const float bk = cbias[c];
      float bj[16];
      float r0 = bf16f(window_row(0)[c]), r1 = bf16f(window_row(1)[c]), r2 = bf16f(window_row(2)[c]);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        bj[j] = 0.f;
        if (j < lenP) {
          const float r3 = bf16f(window_row(3 + j)[c]);
          bj[j] = silu_f(conv4_acc(wk, bk, r0, r1, r2, r3));
          r0 = r1;
          r1 = r2;
          r2 = r3;
        }
        Bj[j * kN + tid] = bj[j];
      }
      // B_j split into bf16 hi + lo, K-major [128 state columns][16 path slots]
      unsigned char* bhi = ws + W.Bt;
      unsigned char* blo = bhi + BT_TILE;
#pragma unroll
      for (int p8 = 0; p8 < 2; ++p8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16x2(bj[p8 * 8 + 2 * e], bj[p8 * 8 + 2 * e + 1], hi[e], lo[e]);
        const uint32_t off = kmajor_off(tid, p8 * 8, A_LBO, A_SBO);
        *reinterpret_cast<uint4*>(bhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(blo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  }
  __syncthreads();
  {  // Gp[j][v] = C_v · B_j: one warp per (j, v) pair of the path
    float* gp = reinterpret_cast<float*>(ws + W.Gp);
    for (int k = warp; k < 16 * NP; k += PREP_THREADS / 32) {
      const int j = k / NP, v = k % NP;
      float s = 0.f;
      if (j < lenP && v < n) {
        const float4 c4 = reinterpret_cast<const float4*>(Cs + v * kN)[lane];
        const float4 b4 = reinterpret_cast<const float4*>(Bj + j * kN)[lane];
        s = c4.x * b4.x;
        s = fmaf(c4.y, b4.y, s);
        s = fmaf(c4.z, b4.z, s);
        s = fmaf(c4.w, b4.w, s);
        s = warp_sum(s);
      }
      if (lane == 0) gp[k] = s;
    }
  }
  {  // conv ring, B | C channels: the path's last rows (staged rows 0..2 that are path rows) go to
     // ring positions head + j; the main kernel writes the x channels of the same rows
    uint16_t* rw = a.ring_w + (size_t)inst * R * conv_dim;
    for (int i = tid; i < 3 * (BCW / 8); i += PREP_THREADS) {
      const int r = i / (BCW / 8), pc = i % (BCW / 8);
      const int k = 3 - r;
      if (k > lenP) continue;
      *reinterpret_cast<uint4*>(rw + (size_t)ring_pos(head_old, lenP - k, R) * conv_dim + d_inner + pc * 8) =
          *reinterpret_cast<const uint4*>(xin + r * BCW + pc * 8);
    }
  }
  int* meta = reinterpret_cast<int*>(ws + W.meta);
  if (tid < kMeta) meta[tid] = pp[tid];
  // the ring head is advanced by the main kernel: other prep CTAs of the instance still read it
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
enum Bar { B_FULL = 0, B_EMPTY = 8, B_AFULL = 16, B_AEMPTY = 18, B_XFULL = 20, B_XFREE = 22, B_READY = 24, B_DU = 25,
           B_YFULL = 26, B_YFREE = 28, B_TAB = 30, B_ESYNC = 31, B_DONE = 32, B_COUNT = 33 };
constexpr int MAX_ST = 8;

struct Smem {
  int bars, stage, aslot, Ct, Bt, Gp, Au, Us, nodes, pathn, poff, meta, xin, srow, xs, total;
  int xrows, srow_floats;  // per buffer
};
__host__ __device__ inline Smem tc_smem(int n, int max_depth, int LP, int ST) {
  Smem s;
  int o = 0;
  auto take = [&](int b, int align) {
    o = (o + align - 1) & ~(align - 1);
    const int r = o;
    o += b;
    return r;
  };
  const int NP = np_of(n), PP = pp_of(n, max_depth);
  s.xrows = 3 + LP + n;
  s.srow_floats = 2 * NP + 2 * PP + (LP > 0 ? 2 * EWS : 0);  // eS [2][NP], coef [2][PP], EW [2][EWS]
  s.bars = take(B_COUNT * 8 + 16, 8);            // barriers, TMEM address, abort flag
  s.stage = take(ST * ROWS * KC * 4, 1024);      // state chunks (64-byte swizzle)
  s.aslot = take(AS * 2 * A_TILE, 128);          // A tiles: hi, lo per slot
  s.Ct = take(2 * NP * kN * 2, 128);             // instance: C hi, lo
  s.Bt = take(LP > 0 ? 2 * BT_TILE : 0, 128);    // instance: path B hi, lo
  s.Gp = take(LP > 0 ? 16 * NP * 4 : 0, 16);     // instance: C_v·B_j
  s.Au = take(LP > 0 ? 2 * A_TILE : 0, 128);     // item: U hi, lo
  s.Us = take(LP > 0 ? 16 * ROWS * 4 : 0, 16);   // item: u_j per row, fp32 [16][128]
  s.nodes = take(n * (int)sizeof(ssm_node), 16); // instance
  s.pathn = take(n * DMAX * 4, 16);              // instance
  s.poff = take(n * 4, 16);                      // instance
  s.meta = take(kMeta * 4, 16);                  // instance
  s.xin = take(2 * s.xrows * XW * 2, 16);        // item: staged x rows, two buffers
  s.srow = take(2 * s.srow_floats * 4, 16);      // item: the two heads' rows, two buffers
  s.xs = take(n * ROWS * 4, 16);                 // item: post-conv x of the tree nodes [n][128]
  s.total = o + 1024;                            // slack for aligning the dynamic base
  return s;
}

template <bool FUSE>
__global__ void __launch_bounds__(THREADS, 2)
    tc_verify_kernel(VerifyArgs a, const unsigned char* __restrict__ ws_base, const __grid_constant__ CUtensorMap tmap,
                     int ST, int tmem_cols) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int n = a.n, H = a.H, NP = np_of(n);
  const int LP = FUSE ? a.LP : 0;
  const TcWs W = tc_ws(n, a.max_depth, H, LP);
  const int PP = W.PP;
  const Smem S = tc_smem(n, a.max_depth, LP, ST);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NHP = (H + 1) / 2;
  const long long items = (long long)a.n_seq * a.L * NHP;
  const long long i0 = items * blockIdx.x / gridDim.x, i1 = items * (blockIdx.x + 1) / gridDim.x;
  const int n_items = (int)(i1 - i0);
  const int d_inner = H * kP, conv_dim = d_inner + BCW, R = a.R;
  const uint32_t bar0 = smem_u32(smem + S.bars);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S.bars + B_COUNT * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S.bars + B_COUNT * 8 + 4);
  float* stage = reinterpret_cast<float*>(smem + S.stage);
  ssm_node* nodes = reinterpret_cast<ssm_node*>(smem + S.nodes);
  const int* pathn = reinterpret_cast<const int*>(smem + S.pathn);
  const int* poff = reinterpret_cast<const int*>(smem + S.poff);
  const int* meta = reinterpret_cast<const int*>(smem + S.meta);
  const float* Gp = reinterpret_cast<const float*>(smem + S.Gp);
  float* Us = reinterpret_cast<float*>(smem + S.Us);
  float* xs = reinterpret_cast<float*>(smem + S.xs);

  auto item_inst = [&](int k) { return (int)((i0 + k) / NHP); };
  auto new_instance = [&](int k) { return k == 0 || item_inst(k) != item_inst(k - 1); };
  auto timeout = [&]() {
    flag(a.status, SSM_STATUS_TIMEOUT);
    *abort_flag = 1;
  };
  auto wait_bar = [&](uint32_t b, uint32_t parity) -> bool {  // bounded; false = give up
    if (*abort_flag) return false;
    if (!mbar_wait(b, parity)) {
      timeout();
      return false;
    }
    return true;
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), EW);
    }
    for (int s = 0; s < AS; ++s) {
      mbar_init(bar(B_AFULL + s), EW);
      mbar_init(bar(B_AEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_XFULL + b), 1);
      mbar_init(bar(B_XFREE + b), EW);
      mbar_init(bar(B_YFULL + b), 1);
      mbar_init(bar(B_YFREE + b), EW);
    }
    mbar_init(bar(B_READY), EW);
    mbar_init(bar(B_DU), 1);
    mbar_init(bar(B_TAB), 1);
    mbar_init(bar(B_ESYNC), EW);
    mbar_init(bar(B_DONE), 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc_warp(smem_u32(tslot), (uint32_t)tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t DU_COL = 0, DY0 = FUSE ? 128u : 0u;  // TMEM columns: U·Bᵀ, then the two accumulators
  auto dy_col = [&](int b) { return DY0 + (uint32_t)(b * NP); };

  if (warp == PRODUCER_WARP) {
    // ---------------- producer: one lane issues every copy ----------------
    if (lane == 0 && n_items > 0) {
      int q = 0;  // chunks issued
      int t = 0;  // instance tables loaded
      auto issue_chunks = [&](int k, int upto) {
        const long long it = i0 + k;
        const int row0 = (int)((it / NHP) * H + 2 * (it % NHP)) * kP;
        while (q < (k + 1) * NCH && q < upto) {
          const int s = q % ST, use = q / ST, kc = q % NCH;
          if (use > 0 && !wait_bar(bar(B_EMPTY + s), (use - 1) & 1)) return false;
          mbar_arrive_expect_tx(bar(B_FULL + s), ROWS * KC * 4);
          tma_load_2d(smem_u32(stage + s * ROWS * KC), &tmap, kc * KC, row0, bar(B_FULL + s));
          ++q;
        }
        return true;
      };
      bool ok = issue_chunks(0, ST);  // the state does not depend on the prep grid
      grid_dependency_wait();
      for (int k = 0; ok && k < n_items; ++k) {
        const long long it = i0 + k;
        const int inst = (int)(it / NHP), hp = (int)(it % NHP), seq = inst / a.L;
        const unsigned char* ws = ws_base + (size_t)inst * W.stride;
        if (new_instance(k)) {
          // the previous item's epilogue (and so its MMAs) are done with the tables
          if (k > 0 && !wait_bar(bar(B_YFREE + ((k - 1) & 1)), ((k - 1) >> 1) & 1)) break;
          const uint32_t bytes = (uint32_t)(2 * NP * kN * 2 + (FUSE ? 2 * BT_TILE + 16 * NP * 4 + kMeta * 4 : 0) +
                                            n * (int)sizeof(ssm_node) + n * DMAX * 4 + ((n * 4 + 15) & ~15));
          mbar_arrive_expect_tx(bar(B_TAB), bytes);
          bulk_load(smem_u32(smem + S.Ct), ws + W.Ct, 2 * NP * kN * 2, bar(B_TAB));
          if (FUSE) {
            bulk_load(smem_u32(smem + S.Bt), ws + W.Bt, 2 * BT_TILE, bar(B_TAB));
            bulk_load(smem_u32(smem + S.Gp), ws + W.Gp, 16 * NP * 4, bar(B_TAB));
            bulk_load(smem_u32(smem + S.meta), ws + W.meta, kMeta * 4, bar(B_TAB));
          }
          bulk_load(smem_u32(nodes), a.layout + (size_t)seq * n, n * (uint32_t)sizeof(ssm_node), bar(B_TAB));
          bulk_load(smem_u32(smem + S.pathn), ws + W.pathn, n * DMAX * 4, bar(B_TAB));
          bulk_load(smem_u32(smem + S.poff), ws + W.poff, (n * 4 + 15) & ~15, bar(B_TAB));
          if (!wait_bar(bar(B_TAB), t & 1)) break;  // the window rows below need the path record
          ++t;
        }
        // the item's x rows (two heads = 256 bytes per row: window, then the tree's nodes) and the
        // two heads' rows of e^S, the coefficients and E, w_j
        const int b = k & 1;
        if (k >= 2 && !wait_bar(bar(B_XFREE + b), ((k >> 1) - 1) & 1)) break;
        const int lenP = FUSE ? min(max(meta[0], 1), LP) : 0;
        const int head_old = FUSE ? meta[1] : a.ring_head[inst];
        if (FUSE && hp == 0) a.head_w[inst] = head_old + lenP;  // after the whole prep grid
        const int win = 3 + lenP;
        const int heads = min(2, H - 2 * hp);
        const uint32_t rb = (uint32_t)heads * kP * 2;
        float* sr = reinterpret_cast<float*>(smem + S.srow) + (size_t)b * S.srow_floats;
        mbar_arrive_expect_tx(bar(B_XFULL + b), rb * (uint32_t)(win + n) + (uint32_t)heads * (NP + PP + (FUSE ? EWS : 0)) * 4);
        bulk_load(smem_u32(sr), ws + W.eS + (size_t)(2 * hp) * NP * 4, heads * NP * 4, bar(B_XFULL + b));
        bulk_load(smem_u32(sr + 2 * NP), ws + W.coef + (size_t)(2 * hp) * PP * 4, heads * PP * 4, bar(B_XFULL + b));
        if (FUSE)
          bulk_load(smem_u32(sr + 2 * NP + 2 * PP), ws + W.EW + (size_t)(2 * hp) * EWS * 4, heads * EWS * 4,
                    bar(B_XFULL + b));
        uint16_t* xin = reinterpret_cast<uint16_t*>(smem + S.xin) + (size_t)b * S.xrows * XW;
        const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim + (size_t)(2 * hp) * kP;
        const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim + (size_t)(2 * hp) * kP;
        for (int r = 0; r < win + n; ++r) {
          const uint16_t* src;
          if (r < 3)
            src = ring + (size_t)ring_pos(head_old, r - 3, R) * conv_dim;
          else if (r < win)
            src = a.prev_xBC + ((size_t)inst * a.prev_n + meta[4 + r - 3]) * conv_dim + (size_t)(2 * hp) * kP;
          else
            src = xbc + (size_t)(r - win) * conv_dim;
          bulk_load(smem_u32(xin + r * XW), src, rb, bar(B_XFULL + b));
        }
        if (!issue_chunks(k, 1 << 30)) break;
        if (k + 1 < n_items && !issue_chunks(k + 1, q + ST)) break;  // the next item's first chunks
      }
      // copies still in flight get a bounded chance to land before the CTA's memory is released
      if (*abort_flag)
        for (int c = q > ST ? q - ST : 0; c < q; ++c) mbar_wait(bar(B_FULL + c % ST), (c / ST) & 1);
    }
  } else if (warp == MMA_WARP) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && n_items > 0) {
      const uint32_t id_y = idesc_bf16(ROWS, NP), id_u = idesc_bf16(ROWS, kN);
      const uint32_t ct = smem_u32(smem + S.Ct), ct_lo = ct + (uint32_t)(NP * kN * 2);
      int q = 0, t = 0;
      for (int k = 0; k < n_items; ++k) {
        const int b = k & 1;
        if (new_instance(k)) {
          if (!wait_bar(bar(B_TAB), t & 1)) break;
          ++t;
        }
        if (k >= 2 && !wait_bar(bar(B_YFREE + b), ((k >> 1) - 1) & 1)) break;  // D[b] has been read
        tc_fence_after();
        for (int kc = 0; kc < NCH; ++kc, ++q) {
          const int s = q % AS;
          if (!wait_bar(bar(B_AFULL + s), (q / AS) & 1)) break;
          tc_fence_after();
          const uint32_t as = smem_u32(smem + S.aslot) + (uint32_t)(s * 2 * A_TILE);
          const uint64_t ahi = desc_kmajor(as, A_LBO, A_SBO), alo = desc_kmajor(as + A_TILE, A_LBO, A_SBO);
          const uint64_t chi = desc_kmajor(ct + kc * 2 * C_LBO, C_LBO, C_SBO);
          const uint64_t clo = desc_kmajor(ct_lo + kc * 2 * C_LBO, C_LBO, C_SBO);
          const uint32_t d = tmem + dy_col(b);
          mma_bf16_tc(d, ahi, chi, id_y, kc > 0);
          mma_bf16_tc(d, ahi, clo, id_y, 1);
          mma_bf16_tc(d, alo, chi, id_y, 1);
          mma_commit(bar(B_AEMPTY + s));  // the A slot is free once these complete
          if (FUSE && kc == 0) {
            // U·Bᵀ for the whole item: 128 rows x 128 state columns x 16 path slots (the element warps
            // wrote the U tile before their first A tile)
            const uint32_t au = smem_u32(smem + S.Au), bt = smem_u32(smem + S.Bt);
            const uint64_t uhi = desc_kmajor(au, A_LBO, A_SBO), ulo = desc_kmajor(au + A_TILE, A_LBO, A_SBO);
            const uint64_t bhi = desc_kmajor(bt, A_LBO, A_SBO), blo = desc_kmajor(bt + BT_TILE, A_LBO, A_SBO);
            mma_bf16_tc(tmem + DU_COL, uhi, bhi, id_u, 0);
            mma_bf16_tc(tmem + DU_COL, uhi, blo, id_u, 1);
            mma_bf16_tc(tmem + DU_COL, ulo, bhi, id_u, 1);
            mma_commit(bar(B_DU));
          }
        }
        if (*abort_flag) break;
        mma_commit(bar(B_YFULL + b));  // the item's accumulator is complete
      }
      mma_commit(bar(B_DONE));  // arrives once every MMA issued above has completed
    }
  } else {
    // ---------------- element warps: thread = state row = x channel of the head pair ----------------
    const int hh = tid >> 6;  // head within the pair
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int q = 0, t = 0, ep = 0;
    // barrier of the element warps alone, bounded like every other wait (an mbarrier, so a warp
    // that gave up cannot leave the others waiting forever)
    auto esync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ESYNC));
      return wait_bar(bar(B_ESYNC), (ep++) & 1);
    };
    // the conv weights of this thread's x channel, fetched one item ahead
    auto conv_w_of = [&](int k, float4& w4, float& b4) {
      const long long it = i0 + k;
      const int layer = (int)((it / NHP) % a.L), c = 2 * (int)(it % NHP) * kP + tid;
      const int cc = c < d_inner ? c : 0;
      w4 = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW)[cc];
      b4 = a.conv_b[(size_t)layer * conv_dim + cc];
    };
    float4 wx;
    float bx;
    if (n_items > 0) conv_w_of(0, wx, bx);
    for (int k = 0; k < n_items; ++k) {
      const long long it = i0 + k;
      const int inst = (int)(it / NHP), hp = (int)(it % NHP);
      const int b = k & 1;
      const int h = 2 * hp + hh;
      const bool hv = h < H;
      if (new_instance(k)) {
        if (!wait_bar(bar(B_TAB), t & 1)) break;
        ++t;
        // the prep kernel checked and reported the layout; clamp the staged records the same way
        // so that no tap or depth leaves its table
        for (int v = tid; v < n; v += EW * 32) {
          ssm_node r = nodes[v];
          for (int d = 0; d < 3; ++d)
            if (r.tap[d] >= v || r.tap[d] < -3) r.tap[d] = -1;
          r.depth = v == 0 ? 0 : min(max(r.depth, 0), a.max_depth);
          nodes[v] = r;
        }
        if (!esync()) break;
      }
      const int lenP = FUSE ? min(max(meta[0], 1), LP) : 0;
      if (!wait_bar(bar(B_XFULL + b), (k >> 1) & 1)) break;
      const float* sr = reinterpret_cast<const float*>(smem + S.srow) + (size_t)b * S.srow_floats;
      const float* eh = sr + hh * NP;                       // e^{S_v} of this thread's head
      const float* ch = sr + 2 * NP + hh * PP;              // its path coefficients
      const float* ew = sr + 2 * NP + 2 * PP + hh * EWS;    // its E, w_j
      // ---- x conv + SiLU of this thread's channel; the committed path's u_j ----
      const uint16_t* xin = reinterpret_cast<const uint16_t*>(smem + S.xin) + (size_t)b * S.xrows * XW + tid;
      const int cg = 2 * hp * kP + tid;  // x channel
      const int win = 3 + lenP;
      {
        int v = 0;
        for (; v + 4 <= n; v += 4) {  // four nodes at a time: 16 loads in flight
          float r[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {  // staged row of a tap: win + node index, or win - j for ring position head - j
            const ssm_node& nd = nodes[v + u];
            r[u][0] = bf16f(xin[(win + nd.tap[2]) * XW]);
            r[u][1] = bf16f(xin[(win + nd.tap[1]) * XW]);
            r[u][2] = bf16f(xin[(win + nd.tap[0]) * XW]);
            r[u][3] = bf16f(xin[(win + v + u) * XW]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) xs[(v + u) * ROWS + tid] = silu_fma(conv4_acc(wx, bx, r[u][0], r[u][1], r[u][2], r[u][3]));
        }
        for (; v < n; ++v) {
          const ssm_node& nd = nodes[v];
          xs[v * ROWS + tid] =
              silu_fma(conv4_acc(wx, bx, bf16f(xin[(win + nd.tap[2]) * XW]), bf16f(xin[(win + nd.tap[1]) * XW]),
                                 bf16f(xin[(win + nd.tap[0]) * XW]), bf16f(xin[(win + v) * XW])));
        }
      }
      if (FUSE) {
        float u[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          u[j] = 0.f;
          if (j < lenP)
            u[j] = ew[1 + j] * silu_fma(conv4_acc(wx, bx, bf16f(xin[j * XW]), bf16f(xin[(j + 1) * XW]),
                                                   bf16f(xin[(j + 2) * XW]), bf16f(xin[(j + 3) * XW])));
          Us[j * ROWS + tid] = u[j];
        }
        unsigned char* au = smem + S.Au;
#pragma unroll
        for (int p8 = 0; p8 < 2; ++p8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(u[p8 * 8 + 2 * e], u[p8 * 8 + 2 * e + 1], hi[e], lo[e]);
          const uint32_t off = kmajor_off(tid, p8 * 8, A_LBO, A_SBO);
          *reinterpret_cast<uint4*>(au + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(au + A_TILE + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        // conv ring, this head pair's x channels: the path's last min(len, 3) rows (window rows
        // 3 + j) go to ring positions head + j (the prep writes their B | C channels)
        if (hv) {
          uint16_t* rw = a.ring_w + (size_t)inst * R * conv_dim + cg;
          for (int j = lenP > 3 ? lenP - 3 : 0; j < lenP; ++j) rw[(size_t)ring_pos(meta[1], j, R) * conv_dim] = xin[(3 + j) * XW];
        }
        fence_async_smem();  // the U tile is read by the tensor cores
      }
      if (k + 1 < n_items) conv_w_of(k + 1, wx, bx);  // in flight during the chunks
      // ---- the state chunks ----
      const size_t hrow = ((size_t)inst * H + 2 * hp) * kP + tid;  // this thread's state row
      const float E = FUSE ? ew[0] : 1.f;
      bool bad = false;
      for (int kc = 0; kc < NCH; ++kc, ++q) {
        const int s = q % ST;
        if (!wait_bar(bar(B_FULL + s), (q / ST) & 1)) {
          bad = true;
          break;
        }
        // row tid of the stage, 16 columns; the copy engine's 64-byte swizzle XORs the 16-byte
        // piece index with address bits 7..8
        const unsigned char* r0 = reinterpret_cast<const unsigned char*>(stage + s * ROWS * KC) + tid * KC * 4;
        const uint32_t sw = (smem_u32(r0) >> 7) & 3;
        float v[16];
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const float4 f = *reinterpret_cast<const float4*>(r0 + ((pc ^ sw) << 4));
          v[4 * pc] = f.x;
          v[4 * pc + 1] = f.y;
          v[4 * pc + 2] = f.z;
          v[4 * pc + 3] = f.w;
        }
        // the chunk as the MMA's A tile (bf16 hi + lo) -- the state as read, the commit's update
        // enters y through E and C_v·B_j
        const int as = q % AS;
        if (q >= AS && !wait_bar(bar(B_AEMPTY + as), ((q / AS) - 1) & 1)) {
          bad = true;
          break;
        }
        unsigned char* at = smem + S.aslot + as * 2 * A_TILE;
#pragma unroll
        for (int p8 = 0; p8 < 2; ++p8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(v[p8 * 8 + 2 * e], v[p8 * 8 + 2 * e + 1], hi[e], lo[e]);
          const uint32_t off = kmajor_off(tid, p8 * 8, A_LBO, A_SBO);
          *reinterpret_cast<uint4*>(at + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(at + A_TILE + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_AFULL + as));
        if (FUSE) {  // h' = E·h + (U·Bᵀ)[row, chunk], stored over h
          if (kc == 0 && !wait_bar(bar(B_DU), k & 1)) {
            bad = true;
            break;
          }
          tc_fence_after();
          float du[16];
          tmem_ld16(tmem + lane_base + DU_COL + (uint32_t)(kc * KC), du);
          if (hv) {
            float4* g = reinterpret_cast<float4*>(a.h_w + hrow * kN + kc * KC);
#pragma unroll
            for (int pc = 0; pc < 4; ++pc)
              g[pc] = make_float4(fmaf(E, v[4 * pc], du[4 * pc]), fmaf(E, v[4 * pc + 1], du[4 * pc + 1]),
                                  fmaf(E, v[4 * pc + 2], du[4 * pc + 2]), fmaf(E, v[4 * pc + 3], du[4 * pc + 3]));
          }
        }
        // the stage goes back only now that its values are consumed: handed back as soon as the
        // loads were issued, it could be refilled by the next copy before they returned
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EMPTY + s));
      }
      if (bad) break;
      // ---- epilogue: y_v = e^{S_v}·(E·C_v·h + Σ_j u_j·C_v·B_j) + Σ_j coef[v][j]·x_{ancestor j} ----
      if (!wait_bar(bar(B_YFULL + b), (k >> 1) & 1)) break;
      tc_fence_after();
      float* yrow = a.y + (size_t)inst * n * d_inner + cg;
      for (int g = 0; g < NP / 16; ++g) {
        float acc[16];
        tmem_ld16(tmem + lane_base + dy_col(b) + (uint32_t)(g * 16), acc);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int v = g * 16 + i;
          if (v < n && hv) {
            float cv = E * acc[i];
            if (FUSE)
              for (int j = 0; j < lenP; ++j) cv = fmaf(Us[j * ROWS + tid], Gp[j * NP + v], cv);
            float yv = eh[v] * cv;
            const int dv = nodes[v].depth, o = poff[v];
            for (int j = 0; j <= dv; ++j) yv = fmaf(ch[o + j], xs[pathn[v * DMAX + j] * ROWS + tid], yv);
            yrow[(size_t)v * d_inner] = yv;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_YFREE + b));
        mbar_arrive(bar(B_XFREE + b));  // the item's staged rows may be replaced
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    // every MMA has completed before the accumulators are released (bounded, as every wait)
    if (lane == 0 && n_items > 0) mbar_wait(bar(B_DONE), 0);
    __syncwarp();
    tc_fence_after();
    tmem_free_warp(tmem, (uint32_t)tmem_cols);
  }
}

int g_tc_sms[64] = {0};
int g_tc_smem_set[2][64] = {{0}};

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// stages of the state ring and CTAs per SM: two CTAs per SM with 4 stages when that plan fits,
// else one CTA with as many stages (<= 8) as fit
void tc_plan(int n, int max_depth, int LP, int& ST, int& per_sm) {
  if (tc_smem(n, max_depth, LP, 4).total <= TWO_PER_SM) {
    ST = 4;
    per_sm = 2;
    return;
  }
  per_sm = 1;
  ST = MAX_ST;
  while (ST > 2 && tc_smem(n, max_depth, LP, ST).total > SMEM_CAP) --ST;
}

template <bool FUSE>
cudaError_t launch_tc_main(const VerifyArgs& a, const unsigned char* ws, cudaStream_t s, int dev) {
  int ST = 4, per_sm = 2;
  const int LP = FUSE ? a.LP : 0;
  tc_plan(a.n, a.max_depth, LP, ST, per_sm);
  const Smem S = tc_smem(a.n, a.max_depth, LP, ST);
  const int smem_bytes = per_sm == 2 && S.total < MIN_TWO ? MIN_TWO : S.total;
  if (dev >= 64 || g_tc_smem_set[FUSE][dev] < smem_bytes) {
    cudaError_t e = cudaFuncSetAttribute(tc_verify_kernel<FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) g_tc_smem_set[FUSE][dev] = smem_bytes;
  }
  int sms = dev < 64 ? g_tc_sms[dev] : 0;
  if (sms == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) g_tc_sms[dev] = sms;
  }
  const long long items = (long long)a.n_seq * a.L * ((a.H + 1) / 2);
  long long grid = items < (long long)per_sm * sms ? items : (long long)per_sm * sms;
  const int o_ctas = tuning(TUNE_VERIFY_CTAS);  // tuning / test override: at most this many CTAs
  if (o_ctas > 0 && grid > o_ctas) grid = o_ctas;
  const int NP = np_of(a.n);
  int cols = 32;
  while (cols < (FUSE ? 128 : 0) + 2 * NP) cols *= 2;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tc_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const long long rows = (long long)a.n_seq * a.L * a.H * kP;
  const cuuint64_t gdim[2] = {(cuuint64_t)kN, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)kN * sizeof(float)};
  const cuuint32_t box[2] = {(cuuint32_t)KC, (cuuint32_t)ROWS};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.h0), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the prep runs
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_verify_kernel<FUSE>, a, ws, tmap, ST, cols);
}

}  // namespace

size_t verify_tc_workspace_bytes(int n, int max_depth, int H, int LP, long long n_inst) {
  return tc_ws(n, max_depth, H, LP).stride * (size_t)n_inst;
}

bool verify_tc_fits(int n, int max_depth, int LP) {
  int ST, per_sm;
  tc_plan(n, max_depth, LP, ST, per_sm);
  return n <= 64 && tc_smem(n, max_depth, LP, ST).total <= SMEM_CAP &&
         tc_prep_layout(n, pp_of(n, max_depth)).total <= SMEM_CAP;
}

cudaError_t launch_verify_tc(const VerifyArgs& a, void* workspace, cudaStream_t s, int which) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((long long)a.n_seq * a.L == 0) return cudaSuccess;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  if (which != 2) {
    const int pb = tc_prep_layout(a.n, pp_of(a.n, a.max_depth)).total;
    static int prep_set[64] = {0};
    if (dev >= 64 || prep_set[dev] < pb) {
      e = cudaFuncSetAttribute(tc_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pb);
      if (e != cudaSuccess) return e;
      if (dev < 64) prep_set[dev] = pb;
    }
    const long long blocks = (long long)a.n_seq * a.L * ((a.H + HB - 1) / HB);
    tc_prep_kernel<<<(unsigned)blocks, PREP_THREADS, pb, s>>>(a, ws);
    e = cudaGetLastError();
    if (e != cudaSuccess || which == 1) return e;
  }
  return a.LP > 0 ? launch_tc_main<true>(a, ws, s, dev) : launch_tc_main<false>(a, ws, s, dev);
}

}  // namespace ssmtree
