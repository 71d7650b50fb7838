// Tree verification kernel: every node of a breadth-first token tree through a
// Mamba2 selective-SSM layer, from the committed state h0.
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
//     y_v[p] = e^{S_v}·(C_v·h0[p,:]) + Σ_{m ∈ path(v)} coef[v,m]·x_m[p] + D·x_v[p],
//     coef[v,m] = e^{S_v - S_m}·Δ_m·(C_v·B_m).
// The only O(P·N) work per node is the dot product C_v·h0[p,:]; the per-node
// states are never formed at all (the extreme of "release after the children
// are done").  h0 is read from HBM exactly once; everything else stays in
// shared memory and registers.
//
// Work split: one CTA (256 threads) per (instance, run of `gpc` head groups of
// G heads).  h0 of the CTA's heads streams through one continuous 4-stage ring
// of 16-column chunks, each one 2-D bulk tensor copy (TMA, 64-byte swizzle)
// issued by a single thread and tracked by full/empty mbarriers, so warps only
// wait for their own data and for the stage they refill; the pre-conv input
// rows (nodes plus the three ring rows above the root) arrive by 1-D bulk
// copies, the B|C rows once per CTA and each group's x rows together with that
// group's first h0 chunk.  Per CTA, once: B and C conv + SiLU for every node and the C_v·B_m
// products along every path.  Per head group: x conv + SiLU, Δ, S, e^S and the
// path coefficients; then the main loop accumulates Z = C_v·h0[row,:] for a
// tile of 16 nodes with a G rows x 4 nodes register tile per thread, using
// packed fp32 FMAs (fma.rn.f32x2) on (even k, odd k) partial sums, and the
// epilogue writes y.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace ssmtree {

int verify_smem_bytes(int n, int* heads_per_group);

namespace {

typedef unsigned long long u64;

constexpr int NT = 16;           // nodes per tile
constexpr int KC = 16;           // d_state columns per pipeline stage
constexpr int KCH = kN / KC;     // stages per node tile
constexpr int STAGES = 4;
constexpr int SROW = KC;         // stage row: 64 B, 16-byte pieces swizzled by the copy engine
constexpr int THREADS = 256;
constexpr int DMAX = SSM_MAX_DEPTH + 1;
constexpr int XW = 256;          // channels per staged input row
constexpr int MAX_GPC = 8;       // head groups per CTA
constexpr int SMEM_LIMIT = 232448;
static_assert(2 * kN == THREADS, "one thread per B|C channel");

struct Smem {
  int bars, stage, nodes, rowidx, pathn, pairs, Cs, Bcoef, xsin, dl, S, eS, Gm, xinX, dts, prm, total;
};

template <int G>
__host__ __device__ inline Smem smem_layout(int n) {
  constexpr int ROWS = G * kP;
  Smem s;
  int o = 0;
  auto take = [&](int bytes) {
    const int r = o;
    o += (bytes + 15) & ~15;
    return r;
  };
  const int a = n * kN * 4, b = n * DMAX * G * 4, c = n * ROWS * 4, d = (n + 3) * XW * 2;
  s.bars = take((2 * STAGES + 2) * 8 + 16);  // full[], empty[], B|C rows, x rows; abort flag
  o = (o + 127) & ~127;                 // swizzled copies need 128-byte alignment
  s.stage = take(STAGES * ROWS * SROW * 4);
  s.nodes = take(n * (int)sizeof(ssm_node));
  s.rowidx = take(n * 16);
  s.pathn = take(n * DMAX * 4);
  s.pairs = take((n * DMAX + 1) * 4);
  s.Cs = take(n * kN * 4);
  s.Bcoef = take(a > b ? a : b);  // B (prologue) | path coefficients (per group)
  s.xsin = take(c > d ? c : d);   // staged B|C input rows (prologue) | post-conv x (per group)
  s.dl = take(n * G * 4);
  s.S = take(n * G * 4);
  s.eS = take(n * G * 4);
  s.Gm = take(n * DMAX * 4);
  s.xinX = take(d);
  s.dts = take(n * MAX_GPC * G * 4);
  s.prm = take(3 * MAX_GPC * G * 4);
  s.total = o;
  return s;
}

template <int G>
struct CoefVec;
template <>
struct CoefVec<4> {
  typedef float4 T;
  __device__ static float at(const float4& c, int i) { return i == 0 ? c.x : i == 1 ? c.y : i == 2 ? c.z : c.w; }
};
template <>
struct CoefVec<2> {
  typedef float2 T;
  __device__ static float at(const float2& c, int i) { return i == 0 ? c.x : c.y; }
};

template <int G>
__global__ void __launch_bounds__(THREADS, 2) tree_verify_kernel(VerifyArgs a, const __grid_constant__ CUtensorMap tmap) {
  constexpr int ROWS = G * kP;
  extern __shared__ __align__(128) unsigned char smem[];
  const int n = a.n;
  const Smem L = smem_layout<G>(n);
  float* stage = reinterpret_cast<float*>(smem + L.stage);
  ssm_node* nodes = reinterpret_cast<ssm_node*>(smem + L.nodes);
  int4* rowidx = reinterpret_cast<int4*>(smem + L.rowidx);
  int* pathn = reinterpret_cast<int*>(smem + L.pathn);
  int* pairs = reinterpret_cast<int*>(smem + L.pairs);  // [0] = count, then v*DMAX+j
  float* Cs = reinterpret_cast<float*>(smem + L.Cs);
  float* Bs = reinterpret_cast<float*>(smem + L.Bcoef);
  float* coef = reinterpret_cast<float*>(smem + L.Bcoef);
  uint16_t* xinBC = reinterpret_cast<uint16_t*>(smem + L.xsin);
  float* xs = reinterpret_cast<float*>(smem + L.xsin);
  float* dl = reinterpret_cast<float*>(smem + L.dl);
  float* Sv = reinterpret_cast<float*>(smem + L.S);
  float* eS = reinterpret_cast<float*>(smem + L.eS);
  float* Gm = reinterpret_cast<float*>(smem + L.Gm);
  uint16_t* xinX = reinterpret_cast<uint16_t*>(smem + L.xinX);
  float* dts = reinterpret_cast<float*>(smem + L.dts);
  float* pbias = reinterpret_cast<float*>(smem + L.prm);
  float* pA = pbias + MAX_GPC * G;
  float* pD = pA + MAX_GPC * G;

  const int tid = threadIdx.x;
  const int NG = (a.H + G - 1) / G;
  const int parts = (NG + a.gpc - 1) / a.gpc;
  const int part = blockIdx.x % parts;
  const int inst = blockIdx.x / parts;
  const int g_first = part * a.gpc;
  const int g_count = min(a.gpc, NG - g_first);
  const int hc_begin = g_first * G;
  const int hc_count = min(g_count * G, a.H - hc_begin);
  const int seq = inst / a.L;
  const int layer = inst % a.L;
  const int d_inner = a.H * kP;
  const int conv_dim = d_inner + 2 * kN;
  const int R = a.R;
  const int n_tiles = (n + NT - 1) / NT;
  const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  const int head = a.ring_head[inst];

  const uint32_t bar0 = smem_u32(smem + L.bars);
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (STAGES + s); };
  const uint32_t bc_bar = bar0 + 8 * (2 * STAGES);
  const uint32_t x_bar = bar0 + 8 * (2 * STAGES + 1);
  volatile int& s_abort = *reinterpret_cast<int*>(smem + L.bars + (2 * STAGES + 2) * 8);
  const int total = g_count * n_tiles * KCH;  // h0 chunks this CTA consumes

  // staged input row r: rows 0..2 are ring positions head-3 .. head-1, row 3+v is node v
  auto issue_inputs = [&](uint16_t* dst, int ch0, int nch, uint32_t bar) {  // one thread
    const uint32_t bytes = (uint32_t)nch * 2;
    mbar_arrive_expect_tx(bar, bytes * (n + 3));
    for (int r = 0; r < n + 3; ++r) {
      const uint16_t* src = r < 3 ? ring + (size_t)ring_pos(head, r - 3, R) * conv_dim : xbc + (size_t)(r - 3) * conv_dim;
      bulk_load(smem_u32(dst + r * XW), src + ch0, bytes, bar);
    }
  };
  // producer (thread 0): cursor over (group, tile, k-chunk); chunk c goes to stage c % STAGES
  int pf_g = 0, pf_t = 0, pf_k = 0, pf_n = 0;
  auto produce = [&](int upto) {
    while (pf_n < upto && pf_n < total) {
      const int slot = pf_n % STAGES;
      if (pf_n >= STAGES && !mbar_wait(empty_bar(slot), ((pf_n / STAGES) - 1) & 1)) {
        flag(a.status, SSM_STATUS_TIMEOUT);
        s_abort = 1;
        return;
      }
      const int hb = hc_begin + pf_g * G;
      if (pf_t == 0 && pf_k == 0) issue_inputs(xinX, hb * kP, min(G, a.H - hb) * kP, x_bar);  // group's x rows
      mbar_arrive_expect_tx(full_bar(slot), ROWS * SROW * 4);
      tma_load_2d(smem_u32(stage + slot * ROWS * SROW), &tmap, pf_k * KC, (inst * a.H + hb) * kP, full_bar(slot));
      if (++pf_k == KCH) {
        pf_k = 0;
        if (++pf_t == n_tiles) {
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

  // swizzled tensor copies need a 128-byte aligned destination; refuse rather than copy
  if (smem_u32(stage) & 127) {
    if (tid == 0) flag(a.status, SSM_STATUS_TIMEOUT);
    return;
  }
  // ---- prologue: barriers, then every input copy in flight first ----
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), THREADS / 32);
    }
    mbar_init(bc_bar, 1);
    mbar_init(x_bar, 1);
    fence_barrier_init();
    issue_inputs(xinBC, d_inner, 2 * kN, bc_bar);
    produce(STAGES);
  }

  const ssm_node* lay = a.layout + (size_t)seq * n;
  for (int v = tid; v < n; v += THREADS) {
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
    if (r.depth < 0 || r.depth > a.max_depth) {
      bad = true;
      r.depth = r.depth < 0 ? 0 : a.max_depth;
    }
    for (int d = 0; d < 3; ++d)
      if (r.tap[d] >= v || r.tap[d] < -3) {
        bad = true;
        r.tap[d] = -1;
      }
    if (bad) flag(a.status, SSM_STATUS_BAD_LAYOUT);
    nodes[v] = r;
    // staged row of each conv tap, oldest first, then the node's own row
    rowidx[v] = make_int4(r.tap[2] + 3, r.tap[1] + 3, r.tap[0] + 3, v + 3);
  }
  for (int i = tid; i < n * hc_count; i += THREADS) {
    const int v = i / hc_count, hh = i - v * hc_count;
    dts[v * (MAX_GPC * G) + hh] = bf16f(a.dt[((size_t)inst * n + v) * a.H + hc_begin + hh]);
  }
  if (tid < hc_count) {
    const size_t pi = (size_t)layer * a.H + hc_begin + tid;
    pbias[tid] = a.dt_bias[pi];
    pA[tid] = neg_exp(a.A_log[pi]);
    pD[tid] = a.D[pi];
  }
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float* cb = a.conv_b + (size_t)layer * conv_dim;
  const float4 wbc = cw[d_inner + tid];  // B|C channel tid
  const float bbc = cb[d_inner + tid];
  float4 wx = make_float4(0.f, 0.f, 0.f, 0.f);  // x conv weights of the next group
  float bx = 0.f;
  if (tid < min(G, a.H - hc_begin) * kP) {
    wx = cw[hc_begin * kP + tid];
    bx = cb[hc_begin * kP + tid];
  }
  __syncthreads();
  for (int v = tid; v < n; v += THREADS) {
    int m = v;  // pathn[v][j] = ancestor of v at depth j
    const int dv = nodes[v].depth;
    for (int j = dv; j >= 0; --j) {
      pathn[v * DMAX + j] = m;
      m = m > 0 ? nodes[m].parent : 0;
      if (m < 0) m = 0;
    }
    int off = 0;  // compact (v, j) pair list: prefix over earlier nodes' path lengths
    for (int u = 0; u < v; ++u) off += nodes[u].depth + 1;
    for (int j = 0; j <= dv; ++j) pairs[1 + off + j] = v * DMAX + j;
    if (v == n - 1) pairs[0] = off + dv + 1;
  }
  wait_or_abort(bc_bar, 0);  // B|C input rows have landed
  __syncthreads();
  {  // B and C conv + SiLU for every node (thread = channel of B|C)
    float* dst = tid < kN ? Bs + tid : Cs + (tid - kN);
    for (int v = 0; v < n; ++v) {
      const int4 r = rowidx[v];
      float s = fmaf(wbc.x, bf16f(xinBC[r.x * XW + tid]), bbc);
      s = fmaf(wbc.y, bf16f(xinBC[r.y * XW + tid]), s);
      s = fmaf(wbc.z, bf16f(xinBC[r.z * XW + tid]), s);
      s = fmaf(wbc.w, bf16f(xinBC[r.w * XW + tid]), s);
      dst[v * kN] = silu_fast(s);
    }
  }
  __syncthreads();
  const int n_pairs = pairs[0];
  {  // Gm[v][j] = C_v · B_{path_j(v)}, one warp per pair
    const int warp = tid >> 5, lane = tid & 31;
    for (int k = warp; k < n_pairs; k += THREADS / 32) {
      const int pr = pairs[1 + k];
      const int v = pr / DMAX;
      const int m = pathn[pr];
      const float4 c4 = reinterpret_cast<const float4*>(Cs + v * kN)[lane];
      const float4 b4 = reinterpret_cast<const float4*>(Bs + m * kN)[lane];
      float s = c4.x * b4.x;
      s = fmaf(c4.y, b4.y, s);
      s = fmaf(c4.z, b4.z, s);
      s = fmaf(c4.w, b4.w, s);
      s = warp_sum(s);
      if (lane == 0) Gm[pr] = s;
    }
  }
  // (B is dead from here on; its space holds the path coefficients)

  const int t_row = tid & 63;  // p
  const int t_nd = tid >> 6;   // node quad within the tile
  u64 acc[G][4];
  int q = 0;  // chunk index
  for (int gi = 0; gi < g_count; ++gi) {
    const int hb = hc_begin + gi * G, heads = min(G, a.H - hb);
    const int hl = gi * G;  // first head of the group within the CTA's head arrays
    for (int tile = 0; tile < n_tiles; ++tile) {
      int vrow[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) vrow[j] = min(tile * NT + t_nd * 4 + j, n - 1) * kN;
      for (int kc = 0; kc < KCH; ++kc, ++q) {
        if (tid == 0) produce(q + STAGES);  // refill the stage chunk q-1 used
        if (tile == 0 && kc == 0) {
          // ---- group set-up: x conv + SiLU, Δ, S, e^S, path coefficients ----
          __syncthreads();  // every warp is past the previous group's epilogue
          wait_or_abort(x_bar, gi & 1);
          if (tid < heads * kP) {
            for (int v = 0; v < n; ++v) {
              const int4 r = rowidx[v];
              float s = fmaf(wx.x, bf16f(xinX[r.x * XW + tid]), bx);
              s = fmaf(wx.y, bf16f(xinX[r.y * XW + tid]), s);
              s = fmaf(wx.z, bf16f(xinX[r.z * XW + tid]), s);
              s = fmaf(wx.w, bf16f(xinX[r.w * XW + tid]), s);
              xs[v * ROWS + tid] = silu_fast(s);
            }
          }
          if (gi + 1 < g_count) {  // prefetch the next group's x conv weights
            const int hn = hb + G;
            if (tid < min(G, a.H - hn) * kP) {
              wx = cw[hn * kP + tid];
              bx = cb[hn * kP + tid];
            }
          }
          for (int i = tid; i < n * G; i += THREADS) {
            const int v = i / G, g = i % G;
            dl[i] = g < heads ? softplus_f(dts[v * (MAX_GPC * G) + hl + g] + pbias[hl + g]) : 0.f;
          }
          __syncthreads();
          for (int i = tid; i < n * G; i += THREADS) {
            const int v = i / G, g = i % G;
            const float A = g < heads ? pA[hl + g] : 0.f;
            float s = 0.f;
            const int dv = nodes[v].depth;
            for (int j = 0; j <= dv; ++j) s = fmaf(dl[pathn[v * DMAX + j] * G + g], A, s);
            Sv[i] = s;
            eS[i] = expf(s);
          }
          __syncthreads();
          for (int i = tid; i < n_pairs * G; i += THREADS) {
            const int pr = pairs[1 + i / G], g = i % G;
            const int v = pr / DMAX, m = pathn[pr];
            coef[pr * G + g] = expf(Sv[v * G + g] - Sv[m * G + g]) * dl[m * G + g] * Gm[pr];
          }
          __syncthreads();
        }
        if (kc == 0) {
#pragma unroll
          for (int i = 0; i < G; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0ull;
        }
        const int slot = q % STAGES;
        wait_or_abort(full_bar(slot), (q / STAGES) & 1);
        const float* st = stage + slot * ROWS * SROW + t_row * SROW;
        const float* cs = Cs + kc * KC;
        // 64-byte swizzle: the 16-byte piece index is XORed with address bits 7..8
        // (rows i*64 + t_row, 4 KB apart, share them)
        const int swz = (smem_u32(st) >> 7) & 3;
#pragma unroll
        for (int k4 = 0; k4 < KC / 4; ++k4) {
          ulonglong2 hv[G], cv[4];
#pragma unroll
          for (int i = 0; i < G; ++i)
            hv[i] = *reinterpret_cast<const ulonglong2*>(st + i * kP * SROW + ((k4 ^ swz) * 4));
#pragma unroll
          for (int j = 0; j < 4; ++j) cv[j] = *reinterpret_cast<const ulonglong2*>(cs + vrow[j] + k4 * 4);
#pragma unroll
          for (int i = 0; i < G; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[i][j] = ffma2(hv[i].x, cv[j].x, acc[i][j]);
              acc[i][j] = ffma2(hv[i].y, cv[j].y, acc[i][j]);
            }
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(empty_bar(slot));  // this warp is done with the stage
        if (kc == KCH - 1) {
          // ---- epilogue: y = e^{S_v}·Z + Σ_path coef·x_m + D·x_v ----
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int v = tile * NT + t_nd * 4 + j;
            if (v >= n) continue;
            float yv[G];
#pragma unroll
            for (int i = 0; i < G; ++i) yv[i] = eS[v * G + i] * pair_sum(acc[i][j]);
            const int dv = nodes[v].depth;
            for (int jj = 0; jj <= dv; ++jj) {
              const int pr = v * DMAX + jj;
              const float* xm = xs + pathn[pr] * ROWS + t_row;
              const typename CoefVec<G>::T cf = *reinterpret_cast<const typename CoefVec<G>::T*>(coef + pr * G);
#pragma unroll
              for (int i = 0; i < G; ++i) yv[i] = fmaf(CoefVec<G>::at(cf, i), xm[i * kP], yv[i]);
            }
            float* yrow = a.y + ((size_t)inst * n + v) * d_inner + hb * kP + t_row;
            const float* xv = xs + v * ROWS + t_row;
#pragma unroll
            for (int i = 0; i < G; ++i)
              if (i < heads) yrow[i * kP] = fmaf(pD[hl + i], xv[i * kP], yv[i]);
          }
        }
      }
    }
  }
  if (tid == 0 && s_abort) {  // give copies still in flight a bounded chance to land
    for (int c = pf_n - STAGES > 0 ? pf_n - STAGES : 0; c < pf_n; ++c) mbar_wait(full_bar(c % STAGES), (c / STAGES) & 1);
  }
}

int g_sms[64] = {0};
int g_configured[2][64] = {{0}};

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

template <int G>
cudaError_t launch_g(const VerifyArgs& a0, cudaStream_t s, int dev) {
  VerifyArgs a = a0;
  const Smem L = smem_layout<G>(a.n);
  const int gi = G == 4 ? 0 : 1;
  if (dev >= 64 || g_configured[gi][dev] < L.total) {
    cudaError_t e = cudaFuncSetAttribute(tree_verify_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tree_verify_kernel<G>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (dev < 64) g_configured[gi][dev] = L.total;
  }
  int sms = dev < 64 ? g_sms[dev] : 0;
  if (sms == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) g_sms[dev] = sms;
  }
  const long long inst = (long long)a.n_seq * a.L;
  const int NG = (a.H + G - 1) / G;
  // enough CTAs for ~4 waves of two CTAs per SM; groups per CTA a divisor of NG when possible
  long long want = (inst * NG) / (8LL * sms);
  int target = (int)(want < 1 ? 1 : (want > MAX_GPC ? MAX_GPC : want));
  int gpc = 1;
  for (int d = 1; d <= target && d <= NG; ++d)
    if (NG % d == 0) gpc = d;
  if (2 * gpc < target) {
    const int parts = (NG + target - 1) / target;
    gpc = (NG + parts - 1) / parts;
  }
  a.gpc = gpc;
  const long long blocks = inst * ((NG + gpc - 1) / gpc);
  if (blocks == 0) return cudaSuccess;
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
  tree_verify_kernel<G><<<(unsigned)blocks, THREADS, L.total, s>>>(a, tmap);
  return cudaGetLastError();
}

}  // namespace

// heads per group used for n nodes (4 while the shared-memory plan fits, else 2)
int verify_smem_bytes(int n, int* heads_per_group) {
  const int t4 = smem_layout<4>(n).total;
  if (t4 <= SMEM_LIMIT) {
    if (heads_per_group) *heads_per_group = 4;
    return t4;
  }
  if (heads_per_group) *heads_per_group = 2;
  return smem_layout<2>(n).total;
}

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int G = 4;
  verify_smem_bytes(a.n, &G);
  return G == 4 ? launch_g<4>(a, s, dev) : launch_g<2>(a, s, dev);
}

}  // namespace ssmtree
