// Tree verification: every node of a breadth-first token tree through a Mamba2
// selective-SSM layer, from the committed state h0.
//
// Method: SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践") §3.2,
// FIFO-based tree verification: each child is updated from its parent's state,
// which is released once the children are done, so per-node states never have
// to be stored.  The Mamba2 update (LightMamba page, "为什么 Mamba 难加速":
// Ā·h_{t-1} + B̄·X) is linear in h, so the state after node v's root-to-node
// path is, exactly,
//     h_v = e^{S_v}·h0 + Σ_{m ∈ path(v)} e^{S_v - S_m}·Δ_m·(x_m ⊗ B_m),
//     S_v = Σ_{m ∈ path(v)} Δ_m·A,
// and y_v = C_v·h_v + D·x_v becomes
//     y_v[p] = e^{S_v}·(C_v·h0[p,:] + Σ_{m ∈ path(v)} coef[v,m]·x_m[p]),
//     coef[v,m] = e^{-S_m}·Δ_m·(C_v·B_m)  (+ D·e^{-S_v} for m = v, the D·x term).
// The per-node states are never formed (the extreme of "release after the
// children are done"); h0 is read from HBM exactly once.
//
// Two kernels per call:
//  * tree_prep_kernel, one CTA per (layer, sequence) instance, or per (instance,
//    block of heads) when the instances do not fill the SMs: B and C conv +
//    SiLU for every node, the path tables, C_v·B_m along every path, Δ, S,
//    e^S and coef[v,m] for every head, and C split into bf16 hi + lo, written
//    to a caller-provided workspace (tens of KB per instance, L2-sized).  Every
//    global load it makes goes out before its first barrier.  It lets the main
//    kernel be scheduled while its last CTAs run (programmatic dependent launch).
//  * tree_verify_kernel, one CTA (256 threads) per (instance, run of head
//    groups of G heads).  Warp 0 is the producer: it streams the group's h0
//    slice through a ring of 16-column chunks (4 stages, 3 with a folded commit;
//    2-D bulk tensor copies with 64-byte swizzle, full/empty mbarriers) -- the
//    first chunks go out before the kernel waits for the prep grid -- and brings
//    each group's inputs (x rows, e^S, coef) on a second barrier.  The x conv +
//    SiLU of group g+1 runs between group g's chunks.  Each node tile's
//    accumulator starts at the path terms, a (rows x nodes)·(nodes x nodes)
//    product on the tensor cores whose coefficients come through a per-node
//    bitmask of its path (k-steps no path reaches are skipped); trees of 2-4
//    tiles contract every chunk against all their tiles in one pass, with
//    accumulators sized to the tiles; each chunk is contracted against C on the
//    tensor cores (mma m16n8k16 on bf16 hi/lo splits of both operands, three
//    products hi·hi + hi·lo + lo·hi, fp32 accumulate: each product to ~2^-17
//    relative, far inside the 1e-3 output bound); the epilogue scales by
//    e^{S_v} and writes y.
//
// Commit folded into verify (LP > 0).  The selective recompute of the previous
// step's accepted path m_0..m_{len-1} (SpecMamba page §3.1) is, by the same
// linearity, a rank-len update of the state:
//     h' = E·h + Σ_j u_j ⊗ B_j,   E = Π_j a_j,   u_j = w_j·x_j,   w_j = Δ_j·Π_{i>j} a_i,
// with a_j = exp(Δ_j·A) and x_j, B_j the post-conv rows of path node j (conv over
// [the ring rows before the path ‖ the path rows]).  The prep kernel computes
// E, w_j and B_j and writes the path's last rows into the conv ring; the main
// kernel advances the ring head (after the whole prep grid: every prep CTA of an
// instance reads the old one), computes its heads' u_j next to the tree's x
// conv, rewrites every h chunk it streams in as h', stores it over h, and
// contracts C against h'.
// The state is read once and written once per speculative step, instead of
// read by verify and read + written again by a separate commit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace ssmtree {

namespace {

constexpr int NT = 16;           // nodes per tile
constexpr int KC = 16;           // d_state columns per pipeline stage
constexpr int KCH = kN / KC;     // stages per node tile
constexpr int STAGES_PLAIN = 4;  // h0 pipeline depth of the plain kernel
constexpr int STAGES_FUSED = 3;  // ... and of the commit-folding kernel (its extra tables need the room)
constexpr int STAGES_DEEP = 8;   // ... of either at one CTA per SM (few groups per SM: bytes in flight)
constexpr int SROW = KC;         // stage row: 64 B, 16-byte pieces swizzled by the copy engine
constexpr int THREADS = 256;
constexpr int DMAX = SSM_MAX_DEPTH + 1;
constexpr int XW = 256;          // channels per staged input row
constexpr int CSTR = kN + 16;    // padded row of the C tables: fp32 in the prep, bf16 hi/lo in the workspace
                                 // (288-byte bf16 rows: conflict-free 8-byte B-fragment loads)
constexpr int MAX_GPC = 64;      // head groups per CTA
constexpr int SMEM_LIMIT = 232448;
constexpr int kMetaInts = 20;    // folded-commit record: [0] path length, [1] ring head before it, [4..19] nodes
static_assert(2 * kN == THREADS, "one thread per B|C channel");

// ---------------------------------------------------------------------------
// per-instance workspace written by the prep kernel (byte offsets)
// ---------------------------------------------------------------------------
struct Ws {
  int NP;  // e^S row: n nodes (+ E_h at column n and w_{j,h} at n+1+j with a folded commit), padded to 4
  int PP;  // path pairs n*(max_depth+1) rounded up to 4
  size_t C, eS, coef, pathn, pairs, BP, meta, stride;
};

__host__ __device__ inline Ws ws_layout(int n, int max_depth, int H, int LP = 0) {
  Ws w;
  w.NP = (n + (LP > 0 ? 1 + LP : 0) + 3) & ~3;
  w.PP = (n * (max_depth + 1) + 3) & ~3;
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t r = o;
    o += (b + 15) & ~size_t(15);
    return r;
  };
  w.C = take((size_t)n * CSTR * 4);        // post-conv C as bf16 hi [n][CSTR], then bf16 lo [n][CSTR]
  w.eS = take((size_t)H * w.NP * 4);       // e^{S_v} [H][NP]
  w.coef = take((size_t)H * w.PP * 4);     // coef [H][PP] in pair order
  w.pathn = take((size_t)n * DMAX * 4);    // ancestor of v at depth j [n][DMAX]
  w.pairs = take((size_t)(w.PP + 4) * 4);  // [count, v*DMAX+j ...]
  w.BP = take((size_t)LP * kN * 4);           // committed path: post-conv B_j [LP][N]
  w.meta = take(LP > 0 ? kMetaInts * 4 : 0);  // committed path: length, old ring head, nodes
  w.stride = o;
  return w;
}

// Validated copy of a layout record (bad fields are clamped and reported).
__device__ ssm_node checked_node(const ssm_node* lay, int v, int max_depth, int32_t* status) {
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

// staged row of each conv tap (rows 0..2 = ring positions head-3..head-1, 3+v = node v), oldest first
__device__ __forceinline__ int4 tap_rows(const ssm_node& r, int v) {
  return make_int4(r.tap[2] + 3, r.tap[1] + 3, r.tap[0] + 3, v + 3);
}

// ---------------------------------------------------------------------------
// prep kernel: everything per instance that does not depend on the head group
// ---------------------------------------------------------------------------
struct PrepSmem {
  int nodes, rrow, pathn, pairs, xin, Bs, Cs, Gm, dl, S, pp, wP, aP, hp, total;
};

// per-head arrays sized by the heads one CTA computes (HR)
__host__ __device__ inline PrepSmem prep_layout(int n, int HR, int PP, int LP = 0) {
  PrepSmem s;
  int o = 0;
  auto take = [&](int b) {
    const int r = o;
    o += (b + 15) & ~15;
    return r;
  };
  const int HRP = HR | 1;  // odd row strides: a warp's reads across nodes hit distinct banks
  s.nodes = take(n * (int)sizeof(ssm_node));
  s.rrow = take(n * 16);  // staged rows of each node's four conv taps
  s.pathn = take(n * (DMAX + 1) * 4);
  s.pairs = take((PP + 4) * 4);
  s.xin = take((n + 3 + LP) * XW * 2);  // [window: 3 ring rows ‖ LP path rows][tree nodes]
  s.Bs = take(n * kN * 4);
  s.Cs = take(n * CSTR * 4);
  s.Gm = take(n * DMAX * 4);
  s.dl = take(n * HRP * 4);
  s.S = take(n * HRP * 4);
  s.pp = take(LP > 0 ? 20 * 4 : 0);  // committed path nodes [16], its length, -, a bad root's refetch
  s.wP = take(LP * HR * 4);          // Δ_j, then Δ_j·Π_{i>j} a_i  [LP][HR]
  s.aP = take(LP * HR * 4);          // a_j = exp(Δ_j·A)          [LP][HR]
  s.hp = take(3 * HR * 4);           // per head: A = -exp(A_log), dt_bias, D
  s.total = o;
  return s;
}

// (i / d, i % d) along i = i0, i0 + step, i0 + 2·step, ... with two divisions in all rather
// than two per element
struct DivWalk {
  int q, r, sq, sr, d;
  __device__ __forceinline__ DivWalk(int i0, int step, int d_) : d(d_) {
    q = i0 / d;
    r = i0 - q * d;
    sq = step / d;
    sr = step - sq * d;
  }
  __device__ __forceinline__ void next() {
    q += sq;
    r += sr;
    if (r >= d) {
      r -= d;
      ++q;
    }
  }
};

// The prep of instance `inst` for heads [h_lo, h_hi) (everything that does not depend on the head
// group), by the whole CTA into `smem`: the shared tables (lead), its heads' e^S and coefficients
// and, with a folded commit, E and w_j into the workspace record; the ring's B | C rows (lead).
// The ring head is left to the main kernel (other CTAs of the instance may still read it).
__device__ void prep_body(const VerifyArgs& a, unsigned char* __restrict__ ws_base, int inst, int h_lo, int h_hi,
                          bool lead, unsigned char* smem) {
  const int n = a.n, H = a.H;
  const bool fuse = a.LP > 0;
  const Ws W = ws_layout(n, a.max_depth, H, a.LP);
  const int HR = h_hi - h_lo, nh = HR;
  const int HRP = HR | 1;  // row stride of dl and e^{-S} (odd: conflict-free across nodes)
  constexpr int PNS = DMAX + 1;  // row stride of the path table in shared memory (odd)
  const PrepSmem L = prep_layout(n, HR, W.PP, a.LP);
  ssm_node* nodes = reinterpret_cast<ssm_node*>(smem + L.nodes);
  int* pathn = reinterpret_cast<int*>(smem + L.pathn);
  int* pairs = reinterpret_cast<int*>(smem + L.pairs);
  uint16_t* xin = reinterpret_cast<uint16_t*>(smem + L.xin);
  float* Bs = reinterpret_cast<float*>(smem + L.Bs);
  float* Cs = reinterpret_cast<float*>(smem + L.Cs);
  float* Gm = reinterpret_cast<float*>(smem + L.Gm);
  float* dl = reinterpret_cast<float*>(smem + L.dl);
  float* emS = reinterpret_cast<float*>(smem + L.S);  // e^{-S_v} [n][HRP]

  const int tid = threadIdx.x;
  int32_t* const status = lead ? a.status : nullptr;
  const int seq = inst / a.L, layer = inst % a.L;
  const int d_inner = H * kP, conv_dim = d_inner + 2 * kN, R = a.R;
  const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  unsigned char* ws = ws_base + (size_t)inst * W.stride;
  int* pp = reinterpret_cast<int*>(smem + L.pp);
  float* hA = reinterpret_cast<float*>(smem + L.hp);  // per head: A, then dt_bias, then D
  float* hBias = hA + HR;  // all per-head scratch indexed by h - h_lo
  float* hD = hA + 2 * HR;
  const uint16_t* prev_xbc = fuse ? a.prev_xBC + (size_t)inst * a.prev_n * conv_dim : nullptr;

  float* wP = reinterpret_cast<float*>(smem + L.wP);
  float* aP = reinterpret_cast<float*>(smem + L.aP);
  // Staged B|C rows: rows t < TB are the window (the three ring rows before the committed path,
  // then the path's rows), row TB + v is tree node v.  Without a folded commit the window is the
  // three ring rows before the root.
  const int TB = 3 + (fuse ? a.LP : 0);

  // ---- every global load of the prep is issued before the first barrier: what depends on the
  // committed path takes the path as given (clamped into the previous tree); warp 0 validates it
  // meanwhile, and rows fetched past a bad entry are never used ----
  for (int i = tid; i < n * 32; i += THREADS) {  // tree nodes' rows
    const int v = i >> 5, pc = i & 31;
    cp_async16(xin + (TB + v) * XW + pc * 8, xbc + (size_t)v * conv_dim + d_inner + pc * 8);
  }
  const int head_old = a.ring_head[inst];  // ring head before the committed path
  const int32_t* pth = fuse ? a.prev_path + (size_t)seq * a.LP : nullptr;
  int len_given = 0;  // path length as given, clamped to [1, LP]
  if (fuse) {
    const int len = a.prev_path_len[seq];
    len_given = len < 1 ? 1 : (len > a.LP ? a.LP : len);
  }
  auto given_node = [&](int j) {
    const int v = pth[j];
    return v < 0 ? 0 : (v >= a.prev_n ? a.prev_n - 1 : v);
  };
  for (int i = tid; i < (3 + len_given) * 32; i += THREADS) {  // window rows
    const int t = i >> 5, pc = i & 31;
    const uint16_t* src = t < 3 ? ring + (size_t)ring_pos(head_old, t - 3, R) * conv_dim
                                : prev_xbc + (size_t)given_node(t - 3) * conv_dim;
    cp_async16(xin + t * XW + pc * 8, src + d_inner + pc * 8);
  }
  cp_async_commit();
  for (int i = tid; i < len_given * nh; i += THREADS) {  // the path rows' dt of this CTA's heads
    const int j = i / nh, hr = i - j * nh;
    wP[j * HR + hr] = bf16f(a.prev_dt[((size_t)inst * a.prev_n + given_node(j)) * H + h_lo + hr]);
  }
  const ssm_node* lay = a.layout + (size_t)seq * n;
  const int t0 = fuse ? 32 : 0;
  for (int hr = tid; hr < HR; hr += THREADS) {
    const int h = h_lo + hr;
    hA[hr] = neg_exp(a.A_log[(size_t)layer * H + h]);
    hBias[hr] = a.dt_bias[(size_t)layer * H + h];
    hD[hr] = a.D[(size_t)layer * H + h];
  }
  if (tid >= t0) {
    for (int v = tid - t0; v < n; v += THREADS - t0) nodes[v] = checked_node(lay, v, a.max_depth, status);
    DivWalk w(tid - t0, THREADS - t0, nh);
    for (int i = tid - t0; i < n * nh; i += THREADS - t0, w.next()) {
      const int v = w.q, h = h_lo + w.r;
      dl[v * HRP + h - h_lo] = softplus_f(bf16f(a.dt[((size_t)inst * n + v) * H + h]) + a.dt_bias[(size_t)layer * H + h]);
    }
  }
  if (fuse && tid < 32) {
    // the committed path, checked as the stand-alone commit checks it: root first, then each
    // node a child of the one before; it ends at the first bad entry (a bad root commits node 0)
    const int lane = tid;
    const int len = a.prev_path_len[seq];
    const bool bad_len = len < 1 || len > a.LP;
    const int v = lane < len_given ? pth[lane] : 0;
    const int before = __shfl_up_sync(0xffffffffu, v, 1);
    bool ok = true;
    if (lane < len_given)
      ok = lane == 0 ? v == 0
                     : (v > before && v >= 1 && v < a.prev_n &&
                        a.prev_layout[(size_t)seq * a.prev_n + v].parent == before);
    const unsigned badm = __ballot_sync(0xffffffffu, lane < len_given && !ok);
    const int good = badm ? __ffs(badm) - 1 : len_given;
    if (lane < good) pp[lane] = v;
    if (lane == 0) {
      if (good == 0) pp[0] = 0;
      pp[16] = good < 1 ? 1 : good;
      pp[18] = good == 0 && given_node(0) != 0;  // node 0's row and dt still to fetch
      if (bad_len || badm) flag(status, SSM_STATUS_PATH_RANGE);
    }
  }
  // conv weights and bias of this thread's B|C channel
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float4 w = cw[d_inner + tid];
  const float bb = a.conv_b[(size_t)layer * conv_dim + d_inner + tid];
  cp_async_wait<0>();
  __syncthreads();
  const int lenP = fuse ? pp[16] : 0;
  if (fuse && pp[18]) {  // a bad root: node 0 of the previous tree is committed instead
    for (int i = tid; i < 32; i += THREADS) cp_async16(xin + 3 * XW + i * 8, prev_xbc + d_inner + i * 8);
    cp_async_commit();
    for (int hr = tid; hr < nh; hr += THREADS)
      wP[hr] = bf16f(a.prev_dt[(size_t)inst * a.prev_n * H + h_lo + hr]);
    cp_async_wait<0>();
    __syncthreads();
  }

  // ---- paths and pairs, the B|C conv, the committed path's Δ_j and a_j ----
  int4* rrow = reinterpret_cast<int4*>(smem + L.rrow);
  for (int v = tid; v < n; v += THREADS) {
    int m = v;
    const ssm_node nd = nodes[v];
    const int dv = nd.depth;
    for (int j = dv; j >= 0; --j) {
      pathn[v * PNS + j] = m;
      m = m > 0 ? nodes[m].parent : 0;
      if (m < 0) m = 0;
    }
    int off = 0;
    for (int u = 0; u < v; ++u) off += nodes[u].depth + 1;
    for (int j = 0; j <= dv; ++j) pairs[1 + off + j] = v * DMAX + j;
    if (v == n - 1) pairs[0] = off + dv + 1;
    // a tap before the root (-k) is the k-th row before it: window row 3 + lenP - k
    auto row = [&](int tap) { return tap < 0 ? 3 + lenP + tap : TB + tap; };
    rrow[v] = make_int4(row(nd.tap[2]), row(nd.tap[1]), row(nd.tap[0]), TB + v);
  }
  __syncthreads();
  {  // B and C conv + SiLU (thread = channel of B|C), four nodes at a time for ILP
    float* __restrict__ dst = tid < kN ? Bs + tid : Cs + (tid - kN);
    const int dstr = tid < kN ? kN : CSTR;
    const uint16_t* __restrict__ xi = xin + tid;
    int v = 0;
    for (; v + 4 <= n; v += 4) {
      float r[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int4 t = rrow[v + u];
        r[u][0] = bf16f(xi[t.x * XW]);
        r[u][1] = bf16f(xi[t.y * XW]);
        r[u][2] = bf16f(xi[t.z * XW]);
        r[u][3] = bf16f(xi[t.w * XW]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) dst[(v + u) * dstr] = silu_fast(conv4_acc(w, bb, r[u][0], r[u][1], r[u][2], r[u][3]));
    }
    for (; v < n; ++v) {
      const int4 t = rrow[v];
      dst[v * dstr] = silu_fast(conv4_acc(w, bb, bf16f(xi[t.x * XW]), bf16f(xi[t.y * XW]), bf16f(xi[t.z * XW]),
                                          bf16f(xi[t.w * XW])));
    }
  }
  for (int i = tid; i < lenP * nh; i += THREADS) {
    const int j = i / nh, hr = i - j * nh;
    const float d = softplus_f(wP[j * HR + hr] + hBias[hr]);
    wP[j * HR + hr] = d;
    aP[j * HR + hr] = decay_of(d, hA[hr]);
  }
  __syncthreads();

  // ---- S_v, C·B products, the shared tables, E and w_j, the path's B conv, the ring rows ----
  // S_v per head: Σ over the path of Δ·A, root first; e^{S_v} to the workspace (v fastest:
  // contiguous stores), Δ_v·e^{-S_v} kept for the coefficients
  DivWalk ws_(tid, THREADS, n);
  for (int i = tid; i < n * nh; i += THREADS, ws_.next()) {
    const int h = h_lo + ws_.q, v = ws_.r;
    const int hr = h - h_lo;
    const float A = hA[hr];
    float s = 0.f;
    const int dv = nodes[v].depth;
    for (int j = 0; j <= dv; ++j) s = fmaf(dl[pathn[v * PNS + j] * HRP + hr], A, s);
    const float em = expf(-s);
    emS[v * HRP + hr] = em;
    reinterpret_cast<float*>(ws + W.eS)[h * W.NP + v] = expf(s);
  }
  const int n_pairs = pairs[0];
  {  // Gm[v][j] = C_v · B_{path_j(v)}: one warp per pair
    const int warp = tid >> 5, lane = tid & 31;
    for (int k = warp; k < n_pairs; k += THREADS / 32) {
      const int pr = pairs[1 + k];
      const int v = pr / DMAX, m = pathn[v * PNS + pr - v * DMAX];
      const float4 c4 = reinterpret_cast<const float4*>(Cs + v * CSTR)[lane];
      const float4 b4 = reinterpret_cast<const float4*>(Bs + m * kN)[lane];
      float s = c4.x * b4.x;
      s = fmaf(c4.y, b4.y, s);
      s = fmaf(c4.z, b4.z, s);
      s = fmaf(c4.w, b4.w, s);
      s = warp_sum(s);
      if (lane == 0) Gm[pr] = s;
    }
  }
  if (lead) {  // workspace: C table, path tables
    // C split once for the tensor cores: C = hi + lo (bf16 pairs, 2^-18 relative)
    uint32_t* dhi = reinterpret_cast<uint32_t*>(ws + W.C);
    uint32_t* dlo = dhi + n * CSTR / 2;
    for (int i = tid; i < n * CSTR / 2; i += THREADS) {
      const int v = i / (CSTR / 2), k = 2 * (i - v * (CSTR / 2));
      uint32_t hi = 0, lo = 0;
      if (k < kN) split_bf16x2(Cs[v * CSTR + k], Cs[v * CSTR + k + 1], hi, lo);
      dhi[i] = hi;
      dlo[i] = lo;
    }
    int* dp = reinterpret_cast<int*>(ws + W.pathn);
    for (int i = tid; i < n * DMAX; i += THREADS) dp[i] = pathn[(i / DMAX) * PNS + i % DMAX];
    int* dq = reinterpret_cast<int*>(ws + W.pairs);
    for (int i = tid; i < W.PP + 4; i += THREADS) dq[i] = i <= n_pairs ? pairs[i] : 0;
  }
  if (fuse) {
    // w_j = Δ_j·Π_{i>j} a_i and E = Π_j a_j per head
    for (int h = h_lo + tid; h < h_hi; h += THREADS) {
      float* eh = reinterpret_cast<float*>(ws + W.eS) + h * W.NP;
      float run = 1.f;
      for (int j = lenP - 1; j >= 0; --j) {
        eh[n + 1 + j] = wP[j * HR + h - h_lo] * run;  // w_{j,h}
        run *= aP[j * HR + h - h_lo];
      }
      eh[n] = run;  // E_h
    }
  }
  if (fuse && lead) {
    // conv + SiLU of the path's B channels over the window (thread = B channel; the x channels
    // are done per head group by the main kernel): path row j from window rows j .. j+3
    if (tid < kN) {
      float* BP = reinterpret_cast<float*>(ws + W.BP);
      const uint16_t* __restrict__ xi = xin + tid;
      for (int j = 0; j < lenP; ++j)
        BP[j * kN + tid] = silu_f(conv4_acc(w, bb, bf16f(xi[j * XW]), bf16f(xi[(j + 1) * XW]), bf16f(xi[(j + 2) * XW]),
                                            bf16f(xi[(j + 3) * XW])));
    }
    // conv ring, B | C channels: the three rows before the new root that are path rows (window
    // rows 3 + lenP - k) go to their ring positions head+lenP-k (the main kernel writes the x
    // channels of the same rows from its staged window); rows of the old ring stay where they are
    uint16_t* rw = a.ring_w + (size_t)inst * R * conv_dim;
    for (int i = tid; i < 3 * 32; i += THREADS) {
      const int k = 3 - (i >> 5), pc = i & 31;
      if (k > lenP) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(xin + (3 + lenP - k) * XW + pc * 8);
      *reinterpret_cast<uint4*>(rw + (size_t)ring_pos(head_old, lenP - k, R) * conv_dim + d_inner + pc * 8) = v;
    }
    int* meta = reinterpret_cast<int*>(ws + W.meta);
    if (tid < 16) meta[4 + tid] = tid < lenP ? pp[tid] : 0;
    if (tid == 0) {
      meta[0] = lenP;
      meta[1] = head_old;
    }
  }
  __syncthreads();
  // coef[h][k] = e^{-S_m}·Δ_m·(C_v·B_m) for pair k = (v, depth-j ancestor m), plus D·e^{-S_v}
  // on the node's own pair: the path terms and D·x of y_v, divided by e^{S_v} (k fastest:
  // contiguous stores)
  float* wc = reinterpret_cast<float*>(ws + W.coef);
  DivWalk wk(tid, THREADS, max(n_pairs, 1));
  for (int i = tid; i < n_pairs * nh; i += THREADS, wk.next()) {
    const int h = h_lo + wk.q, k = wk.r;
    const int pr = pairs[1 + k];
    const int v = pr / DMAX, m = pathn[v * PNS + pr - v * DMAX];
    const int hr = h - h_lo;
    float c = emS[m * HRP + hr] * dl[m * HRP + hr] * Gm[pr];
    if (m == v) c = fmaf(hD[hr], emS[v * HRP + hr], c);
    wc[h * W.PP + k] = c;
  }
}

__global__ void __launch_bounds__(THREADS, 4) tree_prep_kernel(VerifyArgs a, unsigned char* __restrict__ ws_base) {
  extern __shared__ __align__(128) unsigned char smem[];
  // the main kernel may be scheduled once every prep CTA is running; it waits for this grid's
  // completion before it reads anything written here
  launch_dependents();
  // the instance's heads may be split over several CTAs (few instances): each redoes the shared
  // part (cheap) and computes its own heads; block 0 alone writes the shared tables, the ring
  // rows and the head, and reports bad inputs
  const int nhb = a.prep_hb > 1 ? a.prep_hb : 1;
  const int inst = blockIdx.x / nhb, hblk = blockIdx.x % nhb;
  const int hper = (a.H + nhb - 1) / nhb, h_lo = hblk * hper, h_hi = min(a.H, h_lo + hper);
  prep_body(a, ws_base, inst, h_lo, h_hi, hblk == 0, smem);
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
struct Smem {
  int bars, stage, nodes, rowidx, poff, pmask, dep, tkm, pathn, pairs, Cs, xs, xinX, eSg, coefg, BPs, uPs, meta, total;
};

// x rows of a group: node v at xs[v * xs_stride<G>()], rows padded by 4 floats so that the
// path-term A fragments (8 rows x 4 node pairs per load) hit 32 different banks; nodes
// padded to 16 (one k-step of the path-term product)
template <int G>
__host__ __device__ constexpr int xs_stride() { return G * kP + 4; }

template <int G, bool FUSE, bool DEEP = false>
__host__ __device__ inline Smem smem_layout(int n, int PP, int NP, int LP) {
  constexpr int ROWS = G * kP;
  constexpr int ST = DEEP ? STAGES_DEEP : FUSE ? STAGES_FUSED : STAGES_PLAIN;
  Smem s;
  int o = 0;
  auto take = [&](int bytes) {
    const int r = o;
    o += (bytes + 15) & ~15;
    return r;
  };
  s.bars = take((2 * ST + 2) * 8 + 16);  // full[], empty[], prologue, group inputs; abort flag
  o = (o + 127) & ~127;                  // swizzled copies need 128-byte alignment
  s.stage = take(ST * ROWS * SROW * 4);
  s.nodes = take(n * (int)sizeof(ssm_node));
  s.rowidx = take(n * 16);
  s.poff = take(n * 4);
  s.pmask = take(((n + 15) & ~15) * 8);  // per node: which nodes lie on its path (bit m)
  s.dep = take((n + 15) & ~15);           // per node: its depth
  s.tkm = take(4 * 4);                    // per node tile: the k-steps its path terms touch (bit k)
  s.pathn = take(n * DMAX * 4);
  s.pairs = take((PP + 4) * 4);
  s.Cs = take(n * CSTR * 4);
  s.xs = take(((n + 15) & ~15) * xs_stride<G>() * 4);
  s.xinX = take((n + 3 + LP) * G * kP * 2);  // [window: 3 ring rows before the path ‖ path rows][tree rows]
  s.eSg = take(2 * G * NP * 4);    // two groups in flight: the next group's inputs land
  s.coefg = take(2 * G * PP * 4);  // before the current group's epilogue
  s.BPs = take(FUSE ? LP * kN * 4 : 0);        // committed path B_j
  s.uPs = take(FUSE ? 2 * LP * ROWS * 4 : 0);  // committed path u_j of a group's rows (two groups)
  s.meta = take(FUSE ? kMetaInts * 4 : 0);
  s.total = o;
  return s;
}

// NTL: node tiles contracted per pass over a chunk.  With NTL = 1 a tree of several 16-node
// tiles streams each state chunk once per tile; with NTL > 1 (up to NTL tiles) every chunk is
// read, committed and split once and contracted against all tiles, their accumulators held
// side by side.
// DEEP: one CTA per SM with STAGES_DEEP chunks in flight instead of two with 3-4 each, for
// batches with no more head groups than SMs: each CTA has its SM to itself either way, and its
// stream is bound by the bytes it keeps in flight.  (With more groups two CTAs per SM stream
// faster: a CTA's warps alone do not hide their own latencies.)
template <int G, bool FUSE, int NTL, bool DEEP>
__global__ void __launch_bounds__(THREADS, DEEP ? 1 : 2)
    tree_verify_kernel(VerifyArgs a, const unsigned char* __restrict__ ws_base, const __grid_constant__ CUtensorMap tmap) {
  constexpr int ROWS = G * kP;
  constexpr int XWG = G * kP;  // channels per staged x row: this group's
  constexpr int STAGES = DEEP ? STAGES_DEEP : FUSE ? STAGES_FUSED : STAGES_PLAIN;
  extern __shared__ __align__(128) unsigned char smem[];
  const int n = a.n;
  const int LP = FUSE ? a.LP : 0;
  const Ws W = ws_layout(n, a.max_depth, a.H, LP);
  const Smem L = smem_layout<G, FUSE, DEEP>(n, W.PP, W.NP, LP);
  float* stage = reinterpret_cast<float*>(smem + L.stage);
  ssm_node* nodes = reinterpret_cast<ssm_node*>(smem + L.nodes);
  int4* rowidx = reinterpret_cast<int4*>(smem + L.rowidx);
  int* poff = reinterpret_cast<int*>(smem + L.poff);
  unsigned long long* pmask = reinterpret_cast<unsigned long long*>(smem + L.pmask);
  uint8_t* dep = reinterpret_cast<uint8_t*>(smem + L.dep);
  unsigned* tkm = reinterpret_cast<unsigned*>(smem + L.tkm);
  int* pathn = reinterpret_cast<int*>(smem + L.pathn);
  int* pairs = reinterpret_cast<int*>(smem + L.pairs);
  const uint16_t* Chi = reinterpret_cast<const uint16_t*>(smem + L.Cs);  // bf16 [n][CSTR]
  const uint16_t* Clo = Chi + n * CSTR;                                   // bf16 [n][CSTR]
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  uint16_t* xinX = reinterpret_cast<uint16_t*>(smem + L.xinX);
  float* eSg = reinterpret_cast<float*>(smem + L.eSg);
  float* coefg = reinterpret_cast<float*>(smem + L.coefg);
  float* BPs = reinterpret_cast<float*>(smem + L.BPs);
  float* uPs = reinterpret_cast<float*>(smem + L.uPs);
  int* s_meta = reinterpret_cast<int*>(smem + L.meta);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NG = (a.H + G - 1) / G;
  const int parts = (NG + a.gpc - 1) / a.gpc;
  const int part = blockIdx.x % parts;
  const int inst = blockIdx.x / parts;
  const int g_first = part * a.gpc;
  const int g_count = min(a.gpc, NG - g_first);
  const int hc_begin = g_first * G;
  const int seq = inst / a.L;
  const int layer = inst % a.L;
  const int d_inner = a.H * kP;
  const int conv_dim = d_inner + 2 * kN;
  const int R = a.R;
  const int n_tiles = (n + NT - 1) / NT;
  const int n_tb = (n_tiles + NTL - 1) / NTL;  // passes over the state per group
  const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  const unsigned char* ws = ws_base + (size_t)inst * W.stride;

  const uint32_t bar0 = smem_u32(smem + L.bars);
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (STAGES + s); };
  const uint32_t pro_bar = bar0 + 8 * (2 * STAGES);
  const uint32_t x_bar = bar0 + 8 * (2 * STAGES + 1);
  volatile int& s_abort = *reinterpret_cast<int*>(smem + L.bars + (2 * STAGES + 2) * 8);
  const int total = g_count * n_tb * KCH;  // h0 chunks this CTA consumes

  // swizzled tensor copies need a 128-byte aligned destination; refuse rather than copy
  if (smem_u32(stage) & 127) {
    if (tid == 0) flag(a.status, SSM_STATUS_TIMEOUT);
    return;
  }

  // Producer = warp 0.  Chunk c goes to stage c % STAGES.  A group's inputs (x rows for the
  // conv, e^S and coef of its heads) come on x_bar: group 0's once the prologue tables are in
  // (the folded commit's record names the rows), group g+1's at the start of group g, after
  // the barrier that follows every thread's conv of group g -- so every thread has waited on
  // x_bar's phase g, and the x rows and the e^S / coef buffer (g+1) & 1 are free.
  // x rows, oldest first: the window (the three ring rows before the committed path, then
  // the path's rows; without a folded commit, the three ring rows before the root), then the
  // tree's nodes.
  int pf_g = 0, pf_t = 0, pf_k = 0, pf_n = 0;
  int win = 3, head_old = 0;  // window rows, ring head before the window's path (warp 0)
  auto issue_inputs = [&](int g) {  // warp 0, all lanes
    const int hb = hc_begin + g * G;
    const int heads = min(G, a.H - hb);
    const uint32_t xb = (uint32_t)heads * kP * 2;
    const int buf = g & 1;
    if (lane == 0) mbar_arrive_expect_tx(x_bar, xb * (win + n) + (uint32_t)heads * (W.NP + W.PP) * 4);
    __syncwarp();
    for (int r = lane; r < win + n; r += 32) {
      const uint16_t* src;
      if (r < 3)
        src = ring + (size_t)ring_pos(head_old, r - 3, R) * conv_dim;
      else if (r < win)
        src = a.prev_xBC + ((size_t)inst * a.prev_n + s_meta[4 + r - 3]) * conv_dim;
      else
        src = xbc + (size_t)(r - win) * conv_dim;
      bulk_load(smem_u32(xinX + r * XWG), src + hb * kP, xb, x_bar);
    }
    if (lane == 0)
      bulk_load(smem_u32(eSg + buf * G * W.NP), ws + W.eS + (size_t)hb * W.NP * 4, heads * W.NP * 4, x_bar);
    if (lane == 1)
      bulk_load(smem_u32(coefg + buf * G * W.PP), ws + W.coef + (size_t)hb * W.PP * 4, heads * W.PP * 4, x_bar);
  };
  auto produce = [&](int upto) {  // warp 0, all lanes
    while (pf_n < upto && pf_n < total) {
      const int slot = pf_n % STAGES;
      if (pf_n >= STAGES && !mbar_wait(empty_bar(slot), ((pf_n / STAGES) - 1) & 1)) {
        flag(a.status, SSM_STATUS_TIMEOUT);
        s_abort = 1;
        return;
      }
      const int hb = hc_begin + pf_g * G;
      if (lane == 0) {
        mbar_arrive_expect_tx(full_bar(slot), ROWS * SROW * 4);
        tma_load_2d(smem_u32(stage + slot * ROWS * SROW), &tmap, pf_k * KC, (inst * a.H + hb) * kP, full_bar(slot));
      }
      if (++pf_k == KCH) {
        pf_k = 0;
        if (++pf_t == n_tb) {
          pf_t = 0;
          ++pf_g;
        }
      }
      ++pf_n;
    }
  };
  auto wait_or_abort = [&](uint32_t bar, uint32_t parity) {
    if (s_abort) return;
    if (!mbar_wait(bar, parity)) {
      flag(a.status, SSM_STATUS_TIMEOUT);
      s_abort = 1;
    }
  };

  // ---- prologue: barriers, the first h chunks (h is not written by the prep kernel), then --
  // once the prep kernel has finished (programmatic dependent launch) -- its tables ----
  if (warp == 0) {
    if (lane == 0) {
      s_abort = 0;
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(full_bar(i), 1);
        mbar_init(empty_bar(i), THREADS / 32);
      }
      mbar_init(pro_bar, 1);
      mbar_init(x_bar, 1);
      fence_barrier_init();
    }
    __syncwarp();
    produce(STAGES);
  }
  if (warp == 0) {
    grid_dependency_wait();
    if (lane == 0) {
      mbar_arrive_expect_tx(pro_bar, n * (uint32_t)sizeof(ssm_node) + n * CSTR * 4 + n * DMAX * 4 + (W.PP + 4) * 4 +
                                         (FUSE ? (uint32_t)LP * kN * 4 + kMetaInts * 4 : 0u));
      bulk_load(smem_u32(nodes), a.layout + (size_t)seq * n, n * (uint32_t)sizeof(ssm_node), pro_bar);
      bulk_load(smem_u32(smem + L.Cs), ws + W.C, n * CSTR * 4, pro_bar);
      bulk_load(smem_u32(pathn), ws + W.pathn, n * DMAX * 4, pro_bar);
      bulk_load(smem_u32(pairs), ws + W.pairs, (W.PP + 4) * 4, pro_bar);
      if (FUSE) {
        bulk_load(smem_u32(BPs), ws + W.BP, LP * kN * 4, pro_bar);
        bulk_load(smem_u32(s_meta), ws + W.meta, kMetaInts * 4, pro_bar);
      }
    }
    __syncwarp();
    if (FUSE) {
      if (!mbar_wait(pro_bar, 0)) {
        flag(a.status, SSM_STATUS_TIMEOUT);
        s_abort = 1;
      } else {
        win = 3 + min(max(s_meta[0], 1), LP);
        head_old = s_meta[1];
        // the ring head advances here, not in the prep grid: every prep CTA of an instance reads
        // the old head, and a grid larger than the SMs hold starts some of them late
        if (lane == 0 && g_first == 0) a.head_w[inst] = head_old + s_meta[0];
      }
    } else {
      head_old = a.ring_head[inst];
    }
    if (!s_abort) issue_inputs(0);
  }
  // x conv: two channels per thread (2*cp, 2*cp+1), the nodes split between PARTS threads
  constexpr int XSTR = xs_stride<G>();
  constexpr int PAIRS = ROWS / 2;
  constexpr int PARTS = THREADS / PAIRS;
  const int NX = (n + 15) & ~15;
  {  // padding nodes (trees of several tiles: whole node pairs past the tree, a half pair is
     // written by the conv)
    const int x0 = NTL > 1 ? ((n + 1) & ~1) * XSTR : n * XSTR;
    for (int i = x0 + tid; i < NX * XSTR; i += THREADS) xs[i] = 0.f;
  }
  const int cp = tid % PAIRS, cpart = tid / PAIRS;
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float* cb = a.conv_b + (size_t)layer * conv_dim;
  // the x conv weights of the group whose conv runs next (NTL = 1: carried through the previous
  // group's chunks in registers, fetched early; NTL > 1: loaded by the conv itself, which keeps
  // them out of the registers the several tiles' accumulators need)
  float4 wx0 = make_float4(0.f, 0.f, 0.f, 0.f), wx1 = wx0;
  float bx0 = 0.f, bx1 = 0.f;
  auto load_xw = [&](int hb) {
    if (2 * cp < min(G, a.H - hb) * kP) {
      const int c = hb * kP + 2 * cp;
      wx0 = cw[c];
      wx1 = cw[c + 1];
      bx0 = cb[c];
      bx1 = cb[c + 1];
    }
  };
  if (NTL == 1) load_xw(hc_begin);
  grid_dependency_wait();  // nothing below reads the prep kernel's output before it is complete
  __syncthreads();                  // barriers initialised
  wait_or_abort(pro_bar, 0);
  const int lenP = FUSE ? min(max(s_meta[0], 1), LP) : 0;
  for (int v = tid; v < n; v += THREADS) {
    // the prep kernel checked and reported the layout; clamp again so no index leaves its table
    ssm_node r = nodes[v];
    for (int d = 0; d < 3; ++d)
      if (r.tap[d] >= v || r.tap[d] < -3) r.tap[d] = -1;
    r.depth = v == 0 ? 0 : min(max(r.depth, 0), a.max_depth);
    nodes[v] = r;
    const int4 t = tap_rows(r, v);  // rows counted from the last three window rows
    rowidx[v] = make_int4(t.x + lenP, t.y + lenP, t.z + lenP, t.w + lenP);
  }
  if (tid < 4) tkm[tid] = 0u;
  __syncthreads();
  for (int v = tid; v < n; v += THREADS) {
    int off = 0;
    for (int u = 0; u < v; ++u) off += nodes[u].depth + 1;
    poff[v] = off;
  }
  {  // m lies on v's path when v's ancestor at m's depth is m (a ballot per node and 32 m's)
    const int NXN = (n + 15) & ~15;
    for (int v = warp; v < NXN; v += THREADS / 32) {
      unsigned long long mk = 0ull;
      if (v < n) {
        const int dv = nodes[v].depth;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int m = lane + 32 * half;
          bool on = false;
          if (m <= v) {
            const int dm = nodes[m].depth;
            on = dm <= dv && pathn[v * DMAX + dm] == m;
          }
          mk |= (unsigned long long)__ballot_sync(0xffffffffu, on) << (32 * half);
        }
      }
      if (lane == 0) {
        pmask[v] = mk;
        unsigned ks = 0u;  // the 16-node blocks of m this node's path touches
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if ((mk >> (16 * k)) & 0xffffull) ks |= 1u << k;
        if (ks) atomicOr(&tkm[v >> 4], ks);
      }
    }
    for (int m = tid; m < NXN; m += THREADS) dep[m] = m < n ? (uint8_t)nodes[m].depth : 0;
  }

  // coef[v,m] of the tree (this warp's head) for node v (path mask pm, first pair po) and node m:
  // zero unless m is on v's path
  auto path_coef = [&](const float* chd, unsigned long long pm, int po, int m, int dm) -> float {
    return (pm >> m) & 1ull ? chd[po + dm] : 0.f;
  };

  // x conv + SiLU of group g's channels for every tree node (xs), and the committed path's
  // u_j (uPs buffer g & 1).  All threads.
  // the conv's SiLU: on the FMA pipe for one-tile trees (it runs beside tensor and memory work,
  // and measured faster there); with the special-function unit for trees of several tiles, whose
  // conv is 2.5x the work per state byte and issue-bound
  auto silu_x = [](float v) { return NTL > 1 ? silu_fast(v) : silu_fma(v); };
  // u_j = w_{j,h}·x_j of the committed path (window rows j .. j+3), this thread's channels
  auto conv_u = [&](int g, const uint32_t* __restrict__ xi) {
    if (!FUSE) return;
    const float* wj = eSg + ((g & 1) * G + (2 * cp) / kP) * W.NP + n + 1;
    float* ub = uPs + (g & 1) * LP * ROWS;
    for (int j = cpart; j < lenP; j += PARTS) {
      const uint32_t r0 = xi[j * (XWG / 2)], r1 = xi[(j + 1) * (XWG / 2)], r2 = xi[(j + 2) * (XWG / 2)],
                     r3 = xi[(j + 3) * (XWG / 2)];
      *reinterpret_cast<float2*>(ub + j * ROWS + 2 * cp) = make_float2(
          wj[j] * silu_x(conv4_acc(wx0, bx0, bf16_lo(r0), bf16_lo(r1), bf16_lo(r2), bf16_lo(r3))),
          wj[j] * silu_x(conv4_acc(wx1, bx1, bf16_hi(r0), bf16_hi(r1), bf16_hi(r2), bf16_hi(r3))));
    }
  };
  auto xconv = [&](int g) {
    const int hb = hc_begin + g * G, heads = min(G, a.H - hb);
    if (NTL > 1) load_xw(hb);  // in flight during the wait for the rows
    wait_or_abort(x_bar, g & 1);
    if (FUSE) {
      // conv ring, this group's x channels: the committed path's last min(len, 3) rows (window
      // rows 3 + j) go to ring positions head + j; the prep kernel writes their B | C channels
      const int j0 = lenP > 3 ? lenP - 3 : 0, per_row = heads * kP / 8;
      uint16_t* rw = a.ring_w + (size_t)inst * R * conv_dim + (size_t)hb * kP;
      for (int i = tid; i < (lenP - j0) * per_row; i += THREADS) {
        const int j = j0 + i / per_row, pc = i - (i / per_row) * per_row;
        *reinterpret_cast<uint4*>(rw + (size_t)ring_pos(s_meta[1], j, R) * conv_dim + pc * 8) =
            *reinterpret_cast<const uint4*>(xinX + (3 + j) * XWG + pc * 8);
      }
    }
    if (NTL > 1 && 2 * cp < heads * kP) {
      // trees of several tiles: x stored as the path-term A operand, node pairs (v, v + 1) of a
      // row split into bf16 hi and lo once here instead of once per node tile that reads them;
      // pair p of row r at xp[p * XSTR + r] = {hi, lo} (the bytes of the fp32 rows)
      const uint32_t* __restrict__ xi = reinterpret_cast<const uint32_t*>(xinX) + cp;  // row r: xi[r * XWG/2]
      uint4* __restrict__ xp = reinterpret_cast<uint4*>(xs) + cp;                       // pair p: xp[p * XSTR/2]
      const int per = ((n + PARTS - 1) / PARTS + 1) & ~1;  // even: a thread's nodes are whole pairs
      const int v1 = min(n, (cpart + 1) * per);
      auto load4 = [&](int v, uint32_t (&r)[4]) {  // the four conv taps' rows of node v
        const int4 t = rowidx[v];
        r[0] = xi[t.x * (XWG / 2)];
        r[1] = xi[t.y * (XWG / 2)];
        r[2] = xi[t.z * (XWG / 2)];
        r[3] = xi[t.w * (XWG / 2)];
      };
      // nodes v and v + 1 (taps ra, rb): conv + SiLU, split, stored as pair v / 2
      auto store_pair = [&](int v, const uint32_t (&ra)[4], const uint32_t (&rb)[4], bool has_b) {
        const float a0 = silu_x(conv4_acc(wx0, bx0, bf16_lo(ra[0]), bf16_lo(ra[1]), bf16_lo(ra[2]), bf16_lo(ra[3])));
        const float a1 = silu_x(conv4_acc(wx1, bx1, bf16_hi(ra[0]), bf16_hi(ra[1]), bf16_hi(ra[2]), bf16_hi(ra[3])));
        float b0 = 0.f, b1 = 0.f;
        if (has_b) {
          b0 = silu_x(conv4_acc(wx0, bx0, bf16_lo(rb[0]), bf16_lo(rb[1]), bf16_lo(rb[2]), bf16_lo(rb[3])));
          b1 = silu_x(conv4_acc(wx1, bx1, bf16_hi(rb[0]), bf16_hi(rb[1]), bf16_hi(rb[2]), bf16_hi(rb[3])));
        }
        uint4 o;
        split_bf16x2(a0, b0, o.x, o.y);
        split_bf16x2(a1, b1, o.z, o.w);
        xp[(v >> 1) * (XSTR / 2)] = o;
      };
      int v = cpart * per;
      for (; v + 4 <= v1; v += 4) {  // two pairs at a time: 16 loads in flight
        uint32_t r[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) load4(v + u, r[u]);
        store_pair(v, r[0], r[1], true);
        store_pair(v + 2, r[2], r[3], true);
      }
      for (; v < v1; v += 2) {  // a last pair; past the tree's end its second node is zero
        uint32_t r[2][4] = {};
        load4(v, r[0]);
        const bool has_b = v + 1 < n;
        if (has_b) load4(v + 1, r[1]);
        store_pair(v, r[0], r[1], has_b);
      }
      conv_u(g, xi);
    }
    if (NTL == 1 && 2 * cp < heads * kP) {
      const uint32_t* __restrict__ xi = reinterpret_cast<const uint32_t*>(xinX) + cp;  // row r: xi[r * XWG/2]
      float2* __restrict__ xo = reinterpret_cast<float2*>(xs) + cp;                     // node v: xo[v * XSTR/2]
      const int per = (n + PARTS - 1) / PARTS;
      const int v1 = min(n, (cpart + 1) * per);
      int v = cpart * per;
      for (; v + 4 <= v1; v += 4) {  // four nodes at a time: 16 loads in flight
        uint32_t r[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int4 t = rowidx[v + u];
          r[u][0] = xi[t.x * (XWG / 2)];
          r[u][1] = xi[t.y * (XWG / 2)];
          r[u][2] = xi[t.z * (XWG / 2)];
          r[u][3] = xi[t.w * (XWG / 2)];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          xo[(v + u) * (XSTR / 2)] =
              make_float2(silu_x(conv4_acc(wx0, bx0, bf16_lo(r[u][0]), bf16_lo(r[u][1]), bf16_lo(r[u][2]),
                                              bf16_lo(r[u][3]))),
                          silu_x(conv4_acc(wx1, bx1, bf16_hi(r[u][0]), bf16_hi(r[u][1]), bf16_hi(r[u][2]),
                                              bf16_hi(r[u][3]))));
      }
      for (; v < v1; ++v) {
        const int4 t = rowidx[v];
        const uint32_t r0 = xi[t.x * (XWG / 2)], r1 = xi[t.y * (XWG / 2)], r2 = xi[t.z * (XWG / 2)],
                       r3 = xi[t.w * (XWG / 2)];
        xo[v * (XSTR / 2)] =
            make_float2(silu_x(conv4_acc(wx0, bx0, bf16_lo(r0), bf16_lo(r1), bf16_lo(r2), bf16_lo(r3))),
                        silu_x(conv4_acc(wx1, bx1, bf16_hi(r0), bf16_hi(r1), bf16_hi(r2), bf16_hi(r3))));
      }
      conv_u(g, xi);
    }
    if (NTL == 1 && g + 1 < g_count) load_xw(hb + G);  // the next group's, early
  };
  xconv(0);

  // Z tile of a group: 8 warps x (MT m16 tiles) rows x 16 nodes, mma m16n8k16 (bf16 hi/lo, 3 products)
  constexpr int MT = G / 2;
  const int fg = lane >> 2, ft = lane & 3;  // fragment row group / thread-in-group
  const int wrow = warp * 16 * MT;          // first state row of this warp within the group
  const int whead = wrow / kP;              // every row of a warp belongs to one head
  float acc[NTL][MT][2][4];
  float Ew = 1.f;  // decay of the whole committed path for this warp's head
  int q = 0;       // chunk index
  for (int gi = 0; gi < g_count; ++gi) {
    const int hb = hc_begin + gi * G, heads = min(G, a.H - hb);
    // every thread's part of this group's x conv is in shared memory, every warp is past the
    // previous group's epilogue; the next group's inputs can replace this group's x rows
    __syncthreads();
    if (warp == 0 && gi + 1 < g_count && !s_abort) issue_inputs(gi + 1);
    if (FUSE) Ew = eSg[((gi & 1) * G + min(whead, heads - 1)) * W.NP + n];
    for (int tb = 0; tb < n_tb; ++tb) {
      const bool last_tb = tb == n_tb - 1;
      int brow[NTL][2];
#pragma unroll
      for (int i = 0; i < NTL; ++i)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) brow[i][nt] = min((tb * NTL + i) * NT + nt * 8 + fg, n - 1) * CSTR;
      for (int kc = 0; kc < KCH; ++kc, ++q) {
        if (kc == 0) {
          // each tile's accumulator starts at Σ_m coef[v,m]·x_m[p] (path terms and D·x over e^{S_v}):
          // A = x rows of the nodes m (K), B = coef of node v (N; zero off v's path)
          const float* chd = coefg + ((gi & 1) * G + min(whead, heads - 1)) * W.PP;
#pragma unroll
          for (int i = 0; i < NTL; ++i) {
            const int tile = tb * NTL + i;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][mt][nt][e] = 0.f;
            if (tile >= n_tiles) continue;
            // the k-steps (16 nodes m each) where some node of the tile has an ancestor or itself:
            // ancestors precede their nodes, so never past the tile (the same for the whole CTA)
            const unsigned kset = tkm[tile];
            for (int k16 = 0; k16 <= tile; ++k16) {
              if (!((kset >> k16) & 1u)) continue;
              // k = node m: lane (fg, ft) holds m = 2ft, 2ft+1 and 2ft+8, 2ft+9 of the k-step
              const int m0 = k16 * 16 + 2 * ft;
              const unsigned d01 = *reinterpret_cast<const uint16_t*>(dep + m0);  // depths of m0, m0 + 1
              const unsigned d89 = *reinterpret_cast<const uint16_t*>(dep + m0 + 8);
              uint32_t bhi[2][2], blo[2][2];
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                const int v = tile * NT + nt * 8 + fg;  // < NX: the masks are zero past the tree
                const unsigned long long pm = pmask[v];
                const int po = v < n ? poff[v] : 0;
                split_bf16x2(path_coef(chd, pm, po, m0, d01 & 0xff), path_coef(chd, pm, po, m0 + 1, d01 >> 8),
                             bhi[nt][0], blo[nt][0]);
                split_bf16x2(path_coef(chd, pm, po, m0 + 8, d89 & 0xff), path_coef(chd, pm, po, m0 + 9, d89 >> 8),
                             bhi[nt][1], blo[nt][1]);
              }
              const float* xa = xs + m0 * XSTR + wrow + fg;
              // several tiles: the pairs (m0, m0 + 1) and (m0 + 8, m0 + 9) already split by the conv
              const uint2* xq = reinterpret_cast<const uint2*>(xs) + (m0 >> 1) * XSTR + wrow + fg;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                uint32_t ahi[4], alo[4];
                if (NTL > 1) {
                  const uint2* q0 = xq + mt * 16;
                  const uint2 p0 = q0[0], p1 = q0[8], p2 = q0[4 * XSTR], p3 = q0[4 * XSTR + 8];
                  ahi[0] = p0.x, alo[0] = p0.y, ahi[1] = p1.x, alo[1] = p1.y;
                  ahi[2] = p2.x, alo[2] = p2.y, ahi[3] = p3.x, alo[3] = p3.y;
                } else {
                  const float* x0 = xa + mt * 16;
                  split_bf16x2(x0[0], x0[XSTR], ahi[0], alo[0]);
                  split_bf16x2(x0[8], x0[XSTR + 8], ahi[1], alo[1]);
                  split_bf16x2(x0[8 * XSTR], x0[9 * XSTR], ahi[2], alo[2]);
                  split_bf16x2(x0[8 * XSTR + 8], x0[9 * XSTR + 8], ahi[3], alo[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                  mma_bf16(acc[i][mt][nt], alo, bhi[nt]);
                  mma_bf16(acc[i][mt][nt], ahi, blo[nt]);
                  mma_bf16(acc[i][mt][nt], ahi, bhi[nt]);
                }
              }
            }
          }
        }
        const int slot = q % STAGES;
        wait_or_abort(full_bar(slot), (q / STAGES) & 1);
        // Contraction order within the 16-column chunk (one m16n8k16 k-step): k = 2t, 2t+1,
        // 2t+8, 2t+9 take columns 4t .. 4t+3, t = 0..3, so lane (fg, ft) needs exactly the
        // 16-byte piece ft of each of its rows wrow + 16*mt + fg (+8), and of each C row.
        // The copy engine's 64-byte swizzle XORs the piece index with address bits 7..8.
        const unsigned char* st = reinterpret_cast<const unsigned char*>(stage + slot * ROWS * SROW);
        float4 ra[MT], rb[MT];  // rows fg and fg+8 of each m-tile, columns 4*ft .. 4*ft+3
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const unsigned char* r0 = st + (wrow + mt * 16 + fg) * (SROW * 4);
          const int off = (ft ^ ((smem_u32(r0) >> 7) & 3)) << 4;  // rows r0 and r0+8 (512 B apart) share it
          ra[mt] = *reinterpret_cast<const float4*>(r0 + off);
          rb[mt] = *reinterpret_cast<const float4*>(r0 + 8 * SROW * 4 + off);
        }
        // the chunk's rows are in registers: the stage is free once every warp has them, and
        // warp 0 refills it with chunk q + STAGES before this chunk's arithmetic, so STAGES
        // chunks stay in flight while it runs
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(slot));
        if (warp == 0) produce(q + STAGES + 1);
        if (FUSE) {
          // h' = E·h + Σ_j u_j[row]·B_j[col] on this lane's 4 x 2*MT elements, then h' over h
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            ra[mt].x *= Ew; ra[mt].y *= Ew; ra[mt].z *= Ew; ra[mt].w *= Ew;
            rb[mt].x *= Ew; rb[mt].y *= Ew; rb[mt].z *= Ew; rb[mt].w *= Ew;
          }
          const float* ur = uPs + (gi & 1) * LP * ROWS + wrow + fg;
          const float* br = BPs + kc * KC + 4 * ft;
          for (int j = 0; j < lenP; ++j) {
            const float4 bj = *reinterpret_cast<const float4*>(br + j * kN);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const float u0 = ur[j * ROWS + mt * 16], u1 = ur[j * ROWS + mt * 16 + 8];
              ra[mt].x = fmaf(u0, bj.x, ra[mt].x);
              ra[mt].y = fmaf(u0, bj.y, ra[mt].y);
              ra[mt].z = fmaf(u0, bj.z, ra[mt].z);
              ra[mt].w = fmaf(u0, bj.w, ra[mt].w);
              rb[mt].x = fmaf(u1, bj.x, rb[mt].x);
              rb[mt].y = fmaf(u1, bj.y, rb[mt].y);
              rb[mt].z = fmaf(u1, bj.z, rb[mt].z);
              rb[mt].w = fmaf(u1, bj.w, rb[mt].w);
            }
          }
          // with several passes every pass rebuilds h' in registers; only the last one stores
          // it, so no pass can read back a chunk that is already committed
          if (whead < heads && last_tb) {
            float* g0 = a.h_w + ((size_t)(inst * a.H + hb) * kP + wrow + fg) * kN + kc * KC + 4 * ft;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              *reinterpret_cast<float4*>(g0 + (size_t)(mt * 16) * kN) = ra[mt];
              *reinterpret_cast<float4*>(g0 + (size_t)(mt * 16 + 8) * kN) = rb[mt];
            }
          }
        }
        // C of this lane's two B-fragment nodes (columns 4*ft .. 4*ft+3) of tile i
        auto c_frags = [&](int i, uint32_t (&bhi)[2][2], uint32_t (&blo)[2][2]) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint2 h2 = *reinterpret_cast<const uint2*>(Chi + brow[i][nt] + kc * KC + 4 * ft);
            const uint2 l2 = *reinterpret_cast<const uint2*>(Clo + brow[i][nt] + kc * KC + 4 * ft);
            bhi[nt][0] = h2.x;
            bhi[nt][1] = h2.y;
            blo[nt][0] = l2.x;
            blo[nt][1] = l2.y;
          }
        };
        uint32_t bhi0[2][2], blo0[2][2];
        if (NTL == 1) c_frags(0, bhi0, blo0);  // one tile: its fragments serve every m-tile
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t ahi[4], alo[4];
          split_bf16x2(ra[mt].x, ra[mt].y, ahi[0], alo[0]);
          split_bf16x2(rb[mt].x, rb[mt].y, ahi[1], alo[1]);
          split_bf16x2(ra[mt].z, ra[mt].w, ahi[2], alo[2]);
          split_bf16x2(rb[mt].z, rb[mt].w, ahi[3], alo[3]);
#pragma unroll
          for (int i = 0; i < NTL; ++i) {
            if (NTL > 1 && tb * NTL + i >= n_tiles) continue;
            uint32_t bhi[2][2], blo[2][2];
            if (NTL == 1) {
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {
                  bhi[nt][w2] = bhi0[nt][w2];
                  blo[nt][w2] = blo0[nt][w2];
                }
            } else {
              c_frags(i, bhi, blo);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              mma_bf16(acc[i][mt][nt], alo, bhi[nt]);
              mma_bf16(acc[i][mt][nt], ahi, blo[nt]);
              mma_bf16(acc[i][mt][nt], ahi, bhi[nt]);
            }
          }
        }
        if (kc == 1 && last_tb && gi + 1 < g_count) {
          // the next group's x conv (special-function heavy) runs between this group's chunks,
          // next to other warps' tensor and memory work; every warp must be past this group's
          // last path-term product (its x rows) first
          __syncthreads();
          xconv(gi + 1);
        }
        if (kc == KCH - 1 && whead < heads) {
          // ---- epilogue: y = e^{S_v}·acc ----
          const float* eh = eSg + ((gi & 1) * G + whead) * W.NP;
#pragma unroll
          for (int i = 0; i < NTL; ++i) {
            const int tile = tb * NTL + i;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int v = tile * NT + nt * 8 + 2 * ft + c;
                if (v >= n) continue;
                const float es = eh[v];
                float* yrow = a.y + ((size_t)inst * n + v) * d_inner + hb * kP + wrow + fg;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                  yrow[mt * 16] = es * acc[i][mt][nt][c];
                  yrow[mt * 16 + 8] = es * acc[i][mt][nt][2 + c];
                }
              }
          }
        }
      }
    }
  }
  if (warp == 0 && s_abort) {  // give copies still in flight a bounded chance to land
    for (int c = pf_n - STAGES > 0 ? pf_n - STAGES : 0; c < pf_n; ++c) mbar_wait(full_bar(c % STAGES), (c / STAGES) & 1);
    mbar_wait(x_bar, (g_count - 1) & 1);
  }
}

int g_sms[64] = {0};
int g_configured[32][64] = {{0}};  // [kernel variant][device]: the dynamic shared memory set so far

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

template <typename K>
cudaError_t ensure_smem(K kernel, int idx, int dev, int bytes) {
  if (dev >= 64 || g_configured[idx][dev] < bytes) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (dev < 64) g_configured[idx][dev] = bytes;
  }
  return cudaSuccess;
}

template <int G, bool FUSE, int NTL, bool DEEP = false>
cudaError_t launch_main(const VerifyArgs& a0, const unsigned char* ws, cudaStream_t s, int dev) {
  VerifyArgs a = a0;
  const int LP = FUSE ? a.LP : 0;
  const Ws W = ws_layout(a.n, a.max_depth, a.H, LP);
  const Smem L = smem_layout<G, FUSE, DEEP>(a.n, W.PP, W.NP, LP);
  if (L.total > SMEM_LIMIT) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(tree_verify_kernel<G, FUSE, NTL, DEEP>,
                              (G == 4 ? 0 : 1) + 2 * FUSE + 4 * (NTL - 1) + 16 * DEEP, dev, L.total);
  if (e != cudaSuccess) return e;
  int sms = dev < 64 ? g_sms[dev] : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) g_sms[dev] = sms;
  }
  const long long inst = (long long)a.n_seq * a.L;
  const int NG = (a.H + G - 1) / G;
  // groups per CTA: time ~ waves of CTAs x (a fixed part per CTA + one unit per group), the fixed
  // part (prologue, the wait for the prep grid, the first inputs) measured at about 1.5 groups;
  // so few instances get fewer, longer CTAs (batch 1 of the 2.7B shape: 256 CTAs of 5 groups
  // in one wave instead of 1280 of one in five)
  const long long slots = (DEEP ? 1LL : 2LL) * sms;
  int gpc = 1;
  double best = 1e300;
  for (int g = 1; g <= MAX_GPC && g <= NG; ++g) {
    const long long ctas = inst * ((NG + g - 1) / g);
    const double est = (double)((ctas + slots - 1) / slots) * (1.5 + g);
    if (est < best - 1e-9) {
      best = est;
      gpc = g;
    }
  }
  const int o_gpc = tuning(TUNE_VERIFY_GPC);  // tuning / test override
  if (o_gpc >= 1 && o_gpc <= MAX_GPC) gpc = o_gpc;
  a.gpc = gpc;
  const long long blocks = inst * ((NG + gpc - 1) / gpc);
  // h0 as a 2-D tensor: rows (instance, head, p), 128 fp32 columns; one box = G*64 rows x 16 columns
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)kN, (cuuint64_t)(inst * a.H * kP)};
  const cuuint64_t gstride[1] = {(cuuint64_t)kN * sizeof(float)};
  const cuuint32_t box[2] = {(cuuint32_t)KC, (cuuint32_t)(G * kP)};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.h0), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the prep runs
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_verify_kernel<G, FUSE, NTL, DEEP>, a, ws, tmap);
}

}  // namespace

// one workspace serves both kernel sets (the larger of their per-instance records)
size_t verify_workspace_bytes(int n, int max_depth, int H, long long n_inst, int LP) {
  const size_t a = ws_layout(n, max_depth, H, LP).stride * (size_t)n_inst;
  const size_t b = verify_tc_workspace_bytes(n, max_depth, H, LP, n_inst);
  return a > b ? a : b;
}

// heads per group used for n nodes (4 while the shared-memory plan fits, else 2; 0 if neither fits)
int verify_heads_per_group(int n, int max_depth, int H, int LP) {
  const Ws W = ws_layout(n, max_depth, H, LP);
  if (LP > 0) {
    if (smem_layout<4, true>(n, W.PP, W.NP, LP).total <= SMEM_LIMIT) return 4;
    if (smem_layout<2, true>(n, W.PP, W.NP, LP).total <= SMEM_LIMIT) return 2;
    return 0;
  }
  if (smem_layout<4, false>(n, W.PP, W.NP, 0).total <= SMEM_LIMIT) return 4;
  if (smem_layout<2, false>(n, W.PP, W.NP, 0).total <= SMEM_LIMIT) return 2;
  return 0;
}

int verify_prep_smem_bytes(int n, int max_depth, int H, int LP) {
  const Ws W = ws_layout(n, max_depth, H, LP);
  return prep_layout(n, H, W.PP, LP).total;
}

cudaError_t launch_verify(const VerifyArgs& a, void* workspace, cudaStream_t s, int which) {
  // the warp-level kernels below; the override 2 selects the tensor-memory kernels (verify_tc.cu),
  // which measured slower on every workload of this library (the per-chunk copies of 128 rows
  // keep too few bytes in flight and the per-item work runs on four warps)
  if (tuning(TUNE_VERIFY_KERNEL) == 2 && verify_tc_fits(a.n, a.max_depth, a.LP))
    return launch_verify_tc(a, workspace, s, which);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const long long inst = (long long)a.n_seq * a.L;
  if (inst == 0) return cudaSuccess;
  int G = verify_heads_per_group(a.n, a.max_depth, a.H, a.LP);
  if (G == 0) return cudaErrorInvalidValue;
  if (G == 4) {  // few instances: groups of 2 heads when they finish sooner (see the estimate below)
    int sms = dev < 64 ? g_sms[dev] : 0;
    if (sms == 0) {
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      if (dev < 64) g_sms[dev] = sms;
    }
    const long long slots = 2LL * sms, c4 = inst * ((a.H + 3) / 4), c2 = inst * ((a.H + 1) / 2);
    const Ws W2 = ws_layout(a.n, a.max_depth, a.H, a.LP);
    const bool fits2 = a.LP > 0 ? smem_layout<2, true>(a.n, W2.PP, W2.NP, a.LP).total <= SMEM_LIMIT
                                : smem_layout<2, false>(a.n, W2.PP, W2.NP, 0).total <= SMEM_LIMIT;
    // time ~ rounds of CTAs x (fixed cost per CTA + G heads): the fixed part (prologue, the wait
    // for the prep grid, the group's inputs) measured at about 6 heads' worth at the 2.7B shape,
    // so 2-head groups win only when they need no more rounds than 4-head groups
    const long long est4 = (c4 + slots - 1) / slots * (6 + 4), est2 = (c2 + slots - 1) / slots * (6 + 2);
    if (fits2 && est2 < est4) G = 2;
    const int o_g = tuning(TUNE_VERIFY_G);  // tuning / test override (2 or 4)
    if (o_g == 4 || (o_g == 2 && fits2)) G = o_g;
  }
  const int prep_bytes = verify_prep_smem_bytes(a.n, a.max_depth, a.H, a.LP);
  e = ensure_smem(tree_prep_kernel, 4, dev, prep_bytes);
  if (e != cudaSuccess) return e;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int sms = dev < 64 ? g_sms[dev] : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) g_sms[dev] = sms;
  }
  const int n_tiles = (a.n + NT - 1) / NT;
  if (which != 2) {
    // few instances: split each instance's heads over enough CTAs to cover the SMs (at most 16
    // heads per CTA); one CTA per instance once the instances fill them
    VerifyArgs ap = a;
    const long long want = (2LL * sms + inst - 1) / inst;
    const int max_hb = (a.H + 15) / 16;
    ap.prep_hb = (int)(want < 1 ? 1 : (want > max_hb ? max_hb : want));
    tree_prep_kernel<<<(unsigned)(inst * ap.prep_hb), THREADS, prep_bytes, s>>>(ap, ws);
    e = cudaGetLastError();
    if (e != cudaSuccess || which == 1) return e;
  }
  // trees of 2..4 node tiles: 2-head groups contract every tile per pass over the state
  if (n_tiles > 1 && n_tiles <= 4) {
    const Ws W2 = ws_layout(a.n, a.max_depth, a.H, a.LP);
    const bool fits = a.LP > 0 ? smem_layout<2, true>(a.n, W2.PP, W2.NP, a.LP).total <= SMEM_LIMIT
                               : smem_layout<2, false>(a.n, W2.PP, W2.NP, 0).total <= SMEM_LIMIT;
    // accumulators sized to the tree's tiles: registers the unused ones held spilled others (a
    // 40-node tree's folded call took 6.75 ms with four, 5.46 ms with three)
    if (fits && n_tiles == 2)
      return a.LP > 0 ? launch_main<2, true, 2>(a, ws, s, dev) : launch_main<2, false, 2>(a, ws, s, dev);
    if (fits && n_tiles == 3)
      return a.LP > 0 ? launch_main<2, true, 3>(a, ws, s, dev) : launch_main<2, false, 3>(a, ws, s, dev);
    if (fits) return a.LP > 0 ? launch_main<2, true, 4>(a, ws, s, dev) : launch_main<2, false, 4>(a, ws, s, dev);
  }
  // no more head groups than SMs (every CTA alone on its SM anyway): one CTA per group with the
  // deep pipeline, where its memory fits
  const Ws Wd = ws_layout(a.n, a.max_depth, a.H, a.LP);
  const bool deep_fits = a.LP > 0 ? (G == 4 ? smem_layout<4, true, true>(a.n, Wd.PP, Wd.NP, a.LP).total
                                            : smem_layout<2, true, true>(a.n, Wd.PP, Wd.NP, a.LP).total) <= SMEM_LIMIT
                                  : (G == 4 ? smem_layout<4, false, true>(a.n, Wd.PP, Wd.NP, 0).total
                                            : smem_layout<2, false, true>(a.n, Wd.PP, Wd.NP, 0).total) <= SMEM_LIMIT;
  const long long groups = inst * ((a.H + G - 1) / G);
  const int o_deep = tuning(TUNE_VERIFY_DEEP);  // tuning / test override: 1 = never, 2 = where it fits
  const bool deep = deep_fits && (o_deep == 2 || (o_deep != 1 && groups <= sms));
  if (deep) {
    if (a.LP > 0)
      return G == 4 ? launch_main<4, true, 1, true>(a, ws, s, dev) : launch_main<2, true, 1, true>(a, ws, s, dev);
    return G == 4 ? launch_main<4, false, 1, true>(a, ws, s, dev) : launch_main<2, false, 1, true>(a, ws, s, dev);
  }
  if (a.LP > 0) return G == 4 ? launch_main<4, true, 1>(a, ws, s, dev) : launch_main<2, true, 1>(a, ws, s, dev);
  return G == 4 ? launch_main<4, false, 1>(a, ws, s, dev) : launch_main<2, false, 1>(a, ws, s, dev);
}

}  // namespace ssmtree
