// Verification of a chain-shaped draft tree (parent[v] = v - 1), of any length.
//
// SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践") §3.2: the tree
// is walked in order, each node updated from its parent's state.  For a chain
// the walk is a plain scan, cut here into chunks of Q = 16 nodes.  With h the
// state before a chunk (h0 for the first), S_v = Σ_{m ≤ v in the chunk} Δ_m·A
// and the update linear in h (LightMamba page, "为什么 Mamba 难加速"), every
// node of the chunk and the state after it are, exactly,
//     y_v[p] = e^{S_v}·(C_v·h[p,:] + Σ_{m ≤ v} coef[v,m]·x_m[p]),
//     coef[v,m] = e^{-S_m}·Δ_m·(C_v·B_m)  (+ D·e^{-S_v} for m = v),
//     h'[p,:] = E·h[p,:] + Σ_m u_m[p]·B_m,   E = e^{S_last},  u_m = Δ_m·e^{S_last - S_m}·x_m,
// i.e. a 16-node tree verify from h followed by the commit of all 16 nodes
// (the same dual form as the tree kernels), and all three sums are small
// dense products on the tensor cores.
//
// Two kernels.  chain_prep_kernel, one CTA per (instance, chunk), does the work
// that does not depend on the state: the B | C conv + SiLU of the chunk's nodes,
// the Gram C_v·B_m and, for every head, Δ, the scan S and the per-node factors.
// It writes one workspace record per chunk, with B and C already split into
// bf16 hi/lo pairs in the order the mma fragments read them (one 16-byte load
// per lane and fragment).  chain_verify_kernel, one CTA (8 warps) per
// (instance, pair of heads), walks the chunks: warp w owns 16 state rows of
// head w / 4, kept in registers in the mma accumulator layout for the whole
// chain (that layout is also the A-operand layout of the C·h product over the
// state columns, so the state never goes through shared memory; h0 is read
// once, y is the only output).  Per chunk, warp 0 issues bulk copies (TMA) of
// the next chunk's record and pre-conv x rows; the CTA convolves x (+ SiLU)
// into the x and u = w·x pair tables, forms the coefficients, and runs the
// three products.  Every product uses bf16 hi/lo splits of both operands and
// three mma (hi·hi + hi·lo + lo·hi).
#include "common.cuh"

namespace ssmtree {
namespace {

constexpr int Q = 16;                    // chain nodes per chunk (one mma k-step)
constexpr int CHG = 2;                   // heads per CTA
constexpr int CROWS = CHG * kP;          // 128 state rows (and x channels) per CTA
constexpr int CTHREADS = 256;            // 8 warps, 16 rows each
constexpr int RAWR = Q + 3;              // pre-conv rows of a chunk (3 before it)
constexpr int PS = 12;                   // row stride (u32) of the node-pair tables: conflict-free
constexpr int KS = kN / 16;              // k-steps over the state columns (8)
constexpr int JT = kN / 8;               // 8-column tiles of the state (16)

// workspace record of one (instance, chunk), bytes: the part every head reads, then one
// scan block per head
constexpr int REC_C = 0;                         // uint4 [KS][2][32]: C pairs, B operand of C·h
constexpr int REC_B = REC_C + KS * 2 * 32 * 16;  // uint4 [JT][32]: B pairs along the nodes, B operand of the update
constexpr int REC_G = REC_B + JT * 32 * 16;      // float [Q][Q]: Gram C_v·B_m
constexpr int REC_S = REC_G + Q * Q * 4;         // 17408: start of the scan blocks
// scan block of a head (floats): e^{-S_m}·Δ_m, D·e^{-S_v}, e^{S_v}, w_v = Δ_v·e^{S_last - S_v}, E, pad
constexpr int SC_ED = 0, SC_DE = Q, SC_ES = 2 * Q, SC_W = 3 * Q, SC_E = 4 * Q, SCW = 4 * Q + 4;
constexpr int SCB = SCW * 4;                     // 272 bytes
__host__ __device__ constexpr size_t rec_bytes(int H) { return (size_t)REC_S + (size_t)H * SCB; }

static_assert(CHG * Q * (Q / 2) == CTHREADS, "one coefficient pair per thread");
static_assert(2 * kN == CTHREADS, "one B | C channel per prep thread");
static_assert(2 * CROWS == CTHREADS, "two threads per x channel");
static_assert(CHG * Q == 32, "one warp for Δ and S of the head pair");
static_assert(REC_S % 16 == 0 && SCB % 16 == 0, "records are bulk-copied in 16-byte multiples");

// ------------------------------------------------------------------------------------------
// prep: B | C conv + SiLU of one chunk, its fragment-ordered pair tables and the Gram
// ------------------------------------------------------------------------------------------
struct PrepSmem {
  uint16_t raw[RAWR][2 * kN];   // pre-conv B | C rows: chain positions c0 - 3 .. c0 + 15
  uint32_t cf[KS][2][32][4];    // C pairs {hi lo-k, hi hi-k, lo lo-k, lo hi-k} per (k-step, node tile, lane)
  uint32_t bcf[KS][2][32][4];   // the same for B (B operand of the Gram)
};

__global__ void __launch_bounds__(CTHREADS) chain_prep_kernel(VerifyArgs a, unsigned char* __restrict__ ws) {
  __shared__ __align__(16) PrepSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = a.n, R = a.R;
  const int n_chunks = (n + Q - 1) / Q;
  const int inst = blockIdx.x / n_chunks, ci = blockIdx.x - inst * n_chunks;
  const int layer = inst % a.L;
  const int c0 = ci * Q, cnt = min(Q, n - c0);
  const int d_inner = a.H * kP, conv_dim = d_inner + 2 * kN;
  const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  const int head = a.ring_head[inst];
  unsigned char* rec = ws + ((size_t)inst * n_chunks + ci) * rec_bytes(a.H);

  constexpr int PIECES = 2 * kN / 8;  // 16-byte pieces of a B | C row
  for (int i = tid; i < RAWR * PIECES; i += CTHREADS) {
    const int r = i / PIECES, pc = i - r * PIECES;
    const int pos = c0 - 3 + r;
    uint16_t* dst = &sm.raw[r][pc * 8];
    if (pos >= n) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint16_t* row = pos >= 0 ? xbc + (size_t)pos * conv_dim : ring + (size_t)ring_pos(head, pos, R) * conv_dim;
    cp_async16(dst, row + d_inner + pc * 8);
  }
  cp_async_commit();

  // every head's scan block (warp = a pair of heads at a time; lane = head * Q + node)
  {
    const int hx = lane / Q, v = lane - hx * Q;
    for (int hp = warp; 2 * hp < a.H; hp += CTHREADS / 32) {
      const int h = 2 * hp + hx;
      const bool hv = h < a.H;
      float d = 0.f, A = 0.f, Dh = 0.f;
      if (hv) {
        const size_t ph = (size_t)layer * a.H + h;
        A = neg_exp(a.A_log[ph]);
        Dh = a.D[ph];
        if (v < cnt) d = softplus_f(bf16f(a.dt[((size_t)inst * n + c0 + v) * a.H + h]) + a.dt_bias[ph]);
      }
      float sv = d * A;  // Δ = 0 past the chain: no decay, no input
#pragma unroll
      for (int off = 1; off < Q; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, sv, off, Q);
        if (v >= off) sv += o;
      }
      const float s_last = __shfl_sync(0xffffffffu, sv, Q - 1, Q);
      if (hv) {
        float* sc = reinterpret_cast<float*>(rec + REC_S + (size_t)h * SCB);
        const float em = expf(-sv);
        sc[SC_ED + v] = em * d;
        sc[SC_DE + v] = Dh * em;
        sc[SC_ES + v] = expf(sv);
        sc[SC_W + v] = d * expf(s_last - sv);
        if (v < 4) sc[SC_E + v] = v == 0 ? expf(s_last) : 0.f;
      }
    }
  }

  const int c = tid;  // B | C channel
  const float4 wk = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW)[d_inner + c];
  const float bk = a.conv_b[(size_t)layer * conv_dim + d_inner + c];
  cp_async_wait<0>();
  __syncthreads();

  float val[Q];
  {
    float r0 = bf16f(sm.raw[0][c]), r1 = bf16f(sm.raw[1][c]), r2 = bf16f(sm.raw[2][c]);
#pragma unroll
    for (int v = 0; v < Q; ++v) {
      const float r3 = bf16f(sm.raw[v + 3][c]);
      val[v] = v < cnt ? silu_fast(conv4_acc(wk, bk, r0, r1, r2, r3)) : 0.f;
      r0 = r1;
      r1 = r2;
      r2 = r3;
    }
  }
  const int col = c & (kN - 1), odd = c & 1;
  if (c < kN) {  // B along the nodes (update B operand): lane (g = col % 8, t) of tile col / 8
    uint4* dst = reinterpret_cast<uint4*>(rec + REC_B) + (col >> 3) * 32 + (col & 7) * 4;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint4 f;
      split_bf16x2(val[2 * t], val[2 * t + 1], f.x, f.z);
      split_bf16x2(val[2 * t + 8], val[2 * t + 9], f.y, f.w);
      dst[t] = f;
    }
  }
  {  // pairs along the columns: even lanes nodes 0..7, odd lanes nodes 8..15, pair = (even, odd column)
    uint32_t(*tab)[2][32][4] = c < kN ? sm.bcf : sm.cf;
    const int cp = col >> 1, ks = cp >> 3, t = cp & 3, slot = (cp >> 2) & 1;
#pragma unroll
    for (int v = 0; v < Q; ++v) {
      const float nb = __shfl_xor_sync(0xffffffffu, val[v], 1);
      if ((v < Q / 2) != (odd != 0)) {
        const float e0 = odd ? nb : val[v], e1 = odd ? val[v] : nb;
        uint32_t* f = tab[ks][v >> 3][(v & 7) * 4 + t];
        split_bf16x2(e0, e1, f[slot], f[slot + 2]);
      }
    }
  }
  __syncthreads();
  {  // C pairs out (coalesced 16-byte stores)
    const uint4* src = reinterpret_cast<const uint4*>(&sm.cf[0][0][0][0]);
    uint4* dst = reinterpret_cast<uint4*>(rec + REC_C);
    for (int i = tid; i < KS * 2 * 32; i += CTHREADS) dst[i] = src[i];
  }
  if (warp < 2) {
    // Gram[v][m] = C_v·B_m: M = the 16 nodes v, N = the 8 nodes m of node tile `warp`, K = the columns
    float g4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint4 c0f = *reinterpret_cast<const uint4*>(sm.cf[ks][0][lane]);
      const uint4 c1f = *reinterpret_cast<const uint4*>(sm.cf[ks][1][lane]);
      const uint4 bf = *reinterpret_cast<const uint4*>(sm.bcf[ks][warp][lane]);
      const uint32_t ahi[4] = {c0f.x, c1f.x, c0f.y, c1f.y}, alo[4] = {c0f.z, c1f.z, c0f.w, c1f.w};
      const uint32_t bh[2] = {bf.x, bf.y}, bl[2] = {bf.z, bf.w};
      mma_bf16(g4, alo, bh);
      mma_bf16(g4, ahi, bl);
      mma_bf16(g4, ahi, bh);
    }
    float* gram = reinterpret_cast<float*>(rec + REC_G);
    const int g = lane >> 2, m = warp * 8 + 2 * (lane & 3);
    *reinterpret_cast<float2*>(gram + g * Q + m) = make_float2(g4[0], g4[1]);
    *reinterpret_cast<float2*>(gram + (g + 8) * Q + m) = make_float2(g4[2], g4[3]);
  }
}

// ------------------------------------------------------------------------------------------
// main: the walk over the chunks, two heads per CTA
// ------------------------------------------------------------------------------------------
struct ChainSmem {
  unsigned char rec[2][REC_S];               // the chunk's shared record part (double-buffered across chunks)
  float sc[2][CHG][SCW];                     // the pair's scan blocks (likewise)
  uint16_t raw[2][RAWR][CROWS];              // pre-conv x rows of the pair's channels (likewise)
  uint32_t xhi[CROWS][PS], xlo[CROWS][PS];   // x as bf16 pairs along the nodes (A of the path terms)
  uint32_t uhi[CROWS][PS], ulo[CROWS][PS];   // u = w·x likewise (A of the update)
  uint32_t khi[CHG][Q][PS], klo[CHG][Q][PS]; // coef[v][m] pairs along m (B of the path terms)
  float4 cw[CROWS];                          // conv weights and bias of the pair's x channels
  float cb[CROWS];
  unsigned long long full[2];                // bulk-copy barriers of the two buffers
  int abort;                                 // a bounded wait gave up
};

__global__ void __launch_bounds__(CTHREADS, 2)
    chain_verify_kernel(VerifyArgs a, const unsigned char* __restrict__ ws) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChainSmem& sm = *reinterpret_cast<ChainSmem*>(smem_raw);
  volatile int& s_abort = sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int fg = lane >> 2, ft = lane & 3;
  const int n_pairs = (a.H + CHG - 1) / CHG;
  const int hp = blockIdx.x % n_pairs;
  const int inst = blockIdx.x / n_pairs;
  const int layer = inst % a.L;
  const int h_begin = hp * CHG;
  const int heads = min(CHG, a.H - h_begin);
  const int n = a.n;
  const int n_chunks = (n + Q - 1) / Q;
  const int d_inner = a.H * kP, conv_dim = d_inner + 2 * kN;
  const int hh = warp / 4;                      // this warp's head within the pair
  const int rbase = hh * kP + (warp % 4) * 16;  // its first state row within the pair
  const bool live = hh < heads;

  // warp 0: bulk copies of chunk ci's record part, the pair's scan blocks and its pre-conv x
  // rows (row r = chain position c0 - 3 + r; negative: the conv ring) into buffer `buf`, all
  // counted on full[buf]; rows past the chain are zero-filled instead.  Addresses are
  // recomputed from the kernel parameters: nothing of this stays live across the walk.
  auto stage = [&](int ci, int buf) {
    const int np = (a.H + CHG - 1) / CHG, in = blockIdx.x / np, hb = (blockIdx.x - in * np) * CHG;
    const int hd = min(CHG, a.H - hb), nn = a.n, nc = (nn + Q - 1) / Q, cd = a.H * kP + 2 * kN;
    const int c0 = ci * Q, rows = min(RAWR, nn - c0 + 3);
    const uint32_t xbytes = hd * kP * 2, bar = smem_u32(&sm.full[buf]);
    const unsigned char* rec = ws + ((size_t)in * nc + ci) * rec_bytes(a.H);
    if (lane == 0) mbar_arrive_expect_tx(bar, REC_S + hd * SCB + rows * xbytes);
    __syncwarp();
    if (lane == 0) bulk_load(smem_u32(sm.rec[buf]), rec, REC_S, bar);
    if (lane == 1) bulk_load(smem_u32(sm.sc[buf]), rec + REC_S + (size_t)hb * SCB, hd * SCB, bar);
    if (lane < RAWR) {
      const int pos = c0 - 3 + lane;
      if (lane < rows) {
        const uint16_t* row = pos >= 0 ? a.xBC + ((size_t)in * nn + pos) * cd
                                       : a.ring + ((size_t)in * a.R + ring_pos(a.ring_head[in], pos, a.R)) * cd;
        bulk_load(smem_u32(sm.raw[buf][lane]), row + hb * kP, xbytes, bar);
      } else {
        uint4* z = reinterpret_cast<uint4*>(sm.raw[buf][lane]);
#pragma unroll
        for (int i = 0; i < CROWS / 8; ++i) z[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  auto wait_or_abort = [&](int buf, int parity) {
    if (s_abort) return;
    if (!mbar_wait(smem_u32(&sm.full[buf]), parity)) {
      flag(a.status, SSM_STATUS_TIMEOUT);
      s_abort = 1;
    }
  };

  // ---- prologue: barriers, zero columns of a missing second head, the first chunk's copies ----
  if (tid == 0) {
    s_abort = 0;
    mbar_init(smem_u32(&sm.full[0]), 1);
    mbar_init(smem_u32(&sm.full[1]), 1);
    fence_barrier_init();
  }
  if (heads < CHG) {  // never bulk-written: the second head's x columns and scan blocks stay zero
    for (int i = tid; i < 2 * RAWR * kP; i += CTHREADS) {
      const int b = i / (RAWR * kP), rest = i - b * (RAWR * kP), r = rest / kP, c = rest - r * kP;
      sm.raw[b][r][kP + c] = 0;
    }
    for (int i = tid; i < 2 * SCW; i += CTHREADS) sm.sc[i / SCW][1][i % SCW] = 0.f;
  }
  if (tid < CROWS) {
    const int hx = tid / kP;
    float4 wk = make_float4(0.f, 0.f, 0.f, 0.f);
    float bk = 0.f;
    if (hx < heads) {
      const int ch = (h_begin + hx) * kP + (tid - hx * kP);
      wk = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW)[ch];
      bk = a.conv_b[(size_t)layer * conv_dim + ch];
    }
    sm.cw[tid] = wk;
    sm.cb[tid] = bk;
  }
  __syncthreads();
  if (warp == 0) stage(0, 0);

  // this warp's state rows rbase + fg (+8), columns 8j + 2ft (+1): the accumulator layout
  float st[JT][4];
  {
    const float* h0 = a.h0 + ((size_t)inst * a.H + h_begin) * kP * kN;
#pragma unroll
    for (int j = 0; j < JT; ++j) {
      float2 lo = make_float2(0.f, 0.f), hi = lo;
      if (live) {
        lo = *reinterpret_cast<const float2*>(h0 + (size_t)(rbase + fg) * kN + 8 * j + 2 * ft);
        hi = *reinterpret_cast<const float2*>(h0 + (size_t)(rbase + fg + 8) * kN + 8 * j + 2 * ft);
      }
      st[j][0] = lo.x;
      st[j][1] = lo.y;
      st[j][2] = hi.x;
      st[j][3] = hi.y;
    }
  }

  float* const yb = a.y + (size_t)inst * n * d_inner + (size_t)(h_begin * kP + rbase + fg);  // y[.][this thread's row]
  int last_issued = 0;  // warp 0: the last chunk whose copies were issued
  for (int ci = 0; ci < n_chunks; ++ci) {
    const int c0 = ci * Q, cnt = min(Q, n - c0), buf = ci & 1;
    __syncthreads();  // chunk ci-1's tables and buffer buf ^ 1 are no longer read
    wait_or_abort(buf, (ci >> 1) & 1);
    if (warp == 0 && ci + 1 < n_chunks && !s_abort) {  // in flight during this chunk
      stage(ci + 1, buf ^ 1);
      last_issued = ci + 1;
    }

    // ---- x conv + SiLU into the x and u = w·x pairs (thread = channel, half of the nodes) ----
    {
      const int ch = tid & (CROWS - 1), half = tid / CROWS, hx = ch / kP;
      const float4 wk = sm.cw[ch];
      const float bk = sm.cb[ch];
      const int v0 = half * (Q / 2);
      float val[Q / 2];
      float r0 = bf16f(sm.raw[buf][v0][ch]), r1 = bf16f(sm.raw[buf][v0 + 1][ch]), r2 = bf16f(sm.raw[buf][v0 + 2][ch]);
#pragma unroll
      for (int i = 0; i < Q / 2; ++i) {
        const float r3 = bf16f(sm.raw[buf][v0 + i + 3][ch]);
        val[i] = v0 + i < cnt ? silu_fast(conv4_acc(wk, bk, r0, r1, r2, r3)) : 0.f;
        r0 = r1;
        r1 = r2;
        r2 = r3;
      }
      const float* wv = sm.sc[buf][hx] + SC_W + v0;
#pragma unroll
      for (int k = 0; k < Q / 4; ++k) {
        const int kp = half * (Q / 4) + k;
        split_bf16x2(val[2 * k], val[2 * k + 1], sm.xhi[ch][kp], sm.xlo[ch][kp]);
        split_bf16x2(wv[2 * k] * val[2 * k], wv[2 * k + 1] * val[2 * k + 1], sm.uhi[ch][kp], sm.ulo[ch][kp]);
      }
    }
    // ---- coef pairs along m (thread = head, node v, pair k) ----
    {
      const int hx = tid / (Q * (Q / 2)), rest = tid - hx * (Q * (Q / 2)), v = rest / (Q / 2), k = rest - v * (Q / 2);
      const float* gram = reinterpret_cast<const float*>(sm.rec[buf] + REC_G) + v * Q;
      const float* sc = sm.sc[buf][hx];
      float cm[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int m = 2 * k + e;
        float cf = m <= v ? sc[SC_ED + m] * gram[m] : 0.f;
        if (m == v) cf += sc[SC_DE + v];
        cm[e] = cf;
      }
      split_bf16x2(cm[0], cm[1], sm.khi[hx][v][k], sm.klo[hx][v][k]);
    }
    __syncthreads();

    // ---- this warp: the chunk's y and the state after it ----
    if (live) {
      float acc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
      {  // path terms: A = x (rows x nodes m), B = coef (nodes m x nodes v)
        uint32_t ahi[4], alo[4];
        ahi[0] = sm.xhi[rbase + fg][ft];
        alo[0] = sm.xlo[rbase + fg][ft];
        ahi[1] = sm.xhi[rbase + fg + 8][ft];
        alo[1] = sm.xlo[rbase + fg + 8][ft];
        ahi[2] = sm.xhi[rbase + fg][ft + 4];
        alo[2] = sm.xlo[rbase + fg][ft + 4];
        ahi[3] = sm.xhi[rbase + fg + 8][ft + 4];
        alo[3] = sm.xlo[rbase + fg + 8][ft + 4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int v = nt * 8 + fg;
          const uint32_t bh[2] = {sm.khi[hh][v][ft], sm.khi[hh][v][ft + 4]};
          const uint32_t bl[2] = {sm.klo[hh][v][ft], sm.klo[hh][v][ft + 4]};
          mma_bf16(acc[nt], alo, bh);
          mma_bf16(acc[nt], ahi, bl);
          mma_bf16(acc[nt], ahi, bh);
        }
      }
      // C·h: A = the state in registers (rows x state columns), B = C (columns x nodes)
      const uint4* cfr = reinterpret_cast<const uint4*>(sm.rec[buf] + REC_C) + lane;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t ahi[4], alo[4];
        split_bf16x2(st[2 * ks][0], st[2 * ks][1], ahi[0], alo[0]);
        split_bf16x2(st[2 * ks][2], st[2 * ks][3], ahi[1], alo[1]);
        split_bf16x2(st[2 * ks + 1][0], st[2 * ks + 1][1], ahi[2], alo[2]);
        split_bf16x2(st[2 * ks + 1][2], st[2 * ks + 1][3], ahi[3], alo[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint4 f = cfr[(ks * 2 + nt) * 32];
          const uint32_t bh[2] = {f.x, f.y}, bl[2] = {f.z, f.w};
          mma_bf16(acc[nt], alo, bh);
          mma_bf16(acc[nt], ahi, bl);
          mma_bf16(acc[nt], ahi, bh);
        }
      }
      // y_v[p] = e^{S_v}·acc
      const float* eS = sm.sc[buf][hh] + SC_ES;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int v = nt * 8 + 2 * ft + c;
          if (v < cnt) {
            const float es = eS[v];
            float* yr = yb + (size_t)(c0 + v) * d_inner;
            yr[0] = es * acc[nt][c];
            yr[8] = es * acc[nt][2 + c];
          }
        }
      // h' = E·h + u·B: A = u (rows x nodes), B = B (nodes x state columns), accumulator = the state
      uint32_t uhi[4], ulo[4];
      uhi[0] = sm.uhi[rbase + fg][ft];
      ulo[0] = sm.ulo[rbase + fg][ft];
      uhi[1] = sm.uhi[rbase + fg + 8][ft];
      ulo[1] = sm.ulo[rbase + fg + 8][ft];
      uhi[2] = sm.uhi[rbase + fg][ft + 4];
      ulo[2] = sm.ulo[rbase + fg][ft + 4];
      uhi[3] = sm.uhi[rbase + fg + 8][ft + 4];
      ulo[3] = sm.ulo[rbase + fg + 8][ft + 4];
      const float E = sm.sc[buf][hh][SC_E];
      const uint4* bfr = reinterpret_cast<const uint4*>(sm.rec[buf] + REC_B) + lane;
#pragma unroll
      for (int j = 0; j < JT; ++j) {
        const uint4 f = bfr[j * 32];
        const uint32_t bh[2] = {f.x, f.y}, bl[2] = {f.z, f.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) st[j][e] *= E;
        mma_bf16(st[j], ulo, bh);
        mma_bf16(st[j], uhi, bl);
        mma_bf16(st[j], uhi, bh);
      }
    }
  }
  __syncthreads();
  if (warp == 0 && s_abort)  // give copies still in flight a bounded chance to land
    mbar_wait(smem_u32(&sm.full[last_issued & 1]), (last_issued >> 1) & 1);
}

}  // namespace

size_t chain_workspace_bytes(int n, int H, long long n_inst) {
  return (size_t)n_inst * ((n + Q - 1) / Q) * rec_bytes(H);
}

cudaError_t launch_chain_verify(const VerifyArgs& a, void* workspace, cudaStream_t s) {
  const long long n_inst = (long long)a.n_seq * a.L;
  const long long blocks = n_inst * ((a.H + CHG - 1) / CHG);
  if (blocks == 0) return cudaSuccess;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  chain_prep_kernel<<<(unsigned)(n_inst * ((a.n + Q - 1) / Q)), CTHREADS, 0, s>>>(a, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int bytes = (int)sizeof(ChainSmem);
  static int configured[64] = {0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(chain_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = 1;
  }
  chain_verify_kernel<<<(unsigned)blocks, CTHREADS, bytes, s>>>(a, ws);
  return cudaGetLastError();
}

}  // namespace ssmtree
