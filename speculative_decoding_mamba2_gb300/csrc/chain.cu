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
// One CTA (8 warps) per (instance, pair of heads); warp w owns 16 state rows of
// head w / 4, kept in registers in the mma accumulator layout for the whole
// chain: that layout is also the A-operand layout of the C·h product over the
// state columns, so the state never goes through shared memory; h0 is read
// once, y is the only output.  Per chunk: the pre-conv rows (prefetched with
// cp.async one chunk ahead, dt in registers) are convolved + SiLU'd straight into
// the bf16 hi/lo pair tables the mma fragments read (x and u = w·x of both heads,
// B and C); Δ, S, E (a shuffle scan), the Gram C_v·B_m (mma) and the coefficients
// follow.  Every product uses bf16 hi/lo splits of both operands and three mma
// (hi·hi + hi·lo + lo·hi).
#include "common.cuh"

namespace ssmtree {
namespace {

constexpr int Q = 16;                    // chain nodes per chunk (one mma k-step)
constexpr int CHG = 2;                   // heads per CTA
constexpr int CROWS = CHG * kP;          // 128 state rows
constexpr int CTHREADS = 256;            // 8 warps, 16 rows each
constexpr int RAWR = Q + 3;              // pre-conv rows of a chunk (3 before it)
constexpr int RAWC = CHG * kP + 2 * kN;  // staged channels: the pair's x, then B | C (384)
constexpr int PS = 12;                   // row stride (u32) of the node-pair tables: conflict-free
constexpr int CPS = kN / 2 + 4;          // row stride (u32) of the C pair table: conflict-free

static_assert(CHG * Q * (Q / 2) == CTHREADS, "one coefficient pair per thread");
static_assert(2 * kN == CTHREADS, "one B | C channel per thread");
static_assert(CHG * Q == 32, "one warp for Δ and S of the head pair");

struct ChainSmem {
  uint16_t raw[2][RAWR][RAWC];               // pre-conv rows, double-buffered across chunks
  uint32_t chi[Q][CPS], clo[Q][CPS];         // C as bf16 pairs along the state columns (B of C·h, A of the Gram)
  uint32_t bchi[Q][CPS], bclo[Q][CPS];       // B as bf16 pairs along the state columns (B of the Gram)
  uint32_t bhi[kN][PS], blo[kN][PS];         // B as bf16 pairs along the nodes (B of the update)
  uint32_t xhi[CROWS][PS], xlo[CROWS][PS];   // x as bf16 pairs along the nodes (A of the path terms)
  uint32_t uhi[CROWS][PS], ulo[CROWS][PS];   // u = w·x likewise (A of the update)
  uint32_t khi[CHG][Q][PS], klo[CHG][Q][PS]; // coef[v][m] pairs along m (B of the path terms)
  float gram[Q][Q];                          // C_v·B_m
  float dl[CHG][Q], S[CHG][Q], eS[CHG][Q], emS[CHG][Q], w[CHG][Q];
  float E[CHG];
};

__global__ void __launch_bounds__(CTHREADS, 2) chain_verify_kernel(VerifyArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChainSmem& sm = *reinterpret_cast<ChainSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int fg = lane >> 2, ft = lane & 3;
  const int n_pairs = (a.H + CHG - 1) / CHG;
  const int hp = blockIdx.x % n_pairs;
  const int inst = blockIdx.x / n_pairs;
  const int layer = inst % a.L;
  const int h_begin = hp * CHG;
  const int heads = min(CHG, a.H - h_begin);
  const int n = a.n, R = a.R;
  const int d_inner = a.H * kP, conv_dim = d_inner + 2 * kN;
  const uint16_t* xbc = a.xBC + (size_t)inst * n * conv_dim;
  const uint16_t* ring = a.ring + (size_t)inst * R * conv_dim;
  const int head = a.ring_head[inst];
  const int hh = warp / 4;                      // this warp's head within the pair
  const int rbase = hh * kP + (warp % 4) * 16;  // its first state row within the pair
  const bool live = hh < heads;
  const float4* cw = reinterpret_cast<const float4*>(a.conv_w + (size_t)layer * conv_dim * kW);
  const float* cb = a.conv_b + (size_t)layer * conv_dim;

  // pre-conv rows of the chunk starting at c0 into raw buffer `buf`: row r = chain position
  // c0 - 3 + r (negative: the conv ring), channels [the pair's x | B | C]; rows past the
  // chain and channels past the last head are zero
  auto stage = [&](int c0, int buf) {
    constexpr int XP = (CHG * kP) / 8;  // 16-byte pieces of x per row
    constexpr int PIECES = RAWC / 8;
    for (int i = tid; i < RAWR * PIECES; i += CTHREADS) {
      const int r = i / PIECES, pc = i - r * PIECES;
      const int pos = c0 - 3 + r;
      uint16_t* dst = &sm.raw[buf][r][pc * 8];
      const int ch = pc < XP ? h_begin * kP + pc * 8 : d_inner + (pc - XP) * 8;
      if (pos >= n || (pc < XP && ch >= d_inner)) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      const uint16_t* row = pos >= 0 ? xbc + (size_t)pos * conv_dim : ring + (size_t)ring_pos(head, pos, R) * conv_dim;
      cp_async16(dst, row + ch);
    }
    cp_async_commit();
  };

  // this warp's state rows rbase + fg (+8), columns 8j + 2ft (+1): the accumulator layout
  float st[kN / 8][4];
  {
    const float* h0 = a.h0 + ((size_t)inst * a.H + h_begin) * kP * kN;
#pragma unroll
    for (int j = 0; j < kN / 8; ++j) {
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

  // dt of a chunk for warp 0's lanes (lane = head * Q + node), one chunk ahead
  auto load_dt = [&](int c0) -> float {
    const int hx = lane / Q, v = lane - hx * Q;
    if (warp != 0 || hx >= heads || c0 + v >= n) return 0.f;
    return bf16f(a.dt[((size_t)inst * n + c0 + v) * a.H + h_begin + hx]);
  };
  stage(0, 0);
  float dt_next = load_dt(0);
  const int n_chunks = (n + Q - 1) / Q;
  for (int ci = 0; ci < n_chunks; ++ci) {
    const int c0 = ci * Q, cnt = min(Q, n - c0), buf = ci & 1;
    const float dt_cur = dt_next;
    __syncthreads();  // the previous chunk's tables and the other raw buffer are no longer read
    if (ci + 1 < n_chunks) {
      stage(c0 + Q, buf ^ 1);  // the next chunk's rows stay in flight during this chunk
      dt_next = load_dt(c0 + Q);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // ---- phase 1: Δ, S, e^{±S}, E, w (warp 0, shuffle scan); B | C conv + SiLU into pairs ----
    if (warp == 0) {
      const int hx = lane / Q, v = lane - hx * Q;
      float d = 0.f, A = 0.f;
      if (hx < heads) {
        A = neg_exp(a.A_log[(size_t)layer * a.H + h_begin + hx]);
        if (v < cnt) d = softplus_f(dt_cur + a.dt_bias[(size_t)layer * a.H + h_begin + hx]);
      }
      float s = d * A;  // Δ = 0 past the chain: no decay, no input
#pragma unroll
      for (int off = 1; off < Q; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, s, off, Q);
        if (v >= off) s += o;
      }
      const float s_last = __shfl_sync(0xffffffffu, s, Q - 1, Q);
      sm.dl[hx][v] = d;
      sm.S[hx][v] = s;
      sm.eS[hx][v] = expf(s);
      sm.emS[hx][v] = expf(-s);
      sm.w[hx][v] = d * expf(s_last - s);
      if (v == Q - 1) sm.E[hx] = expf(s_last);
    }
    {  // thread = B | C channel: 16 nodes, then the pair tables (neighbour column by shuffle)
      const int c = tid;
      const float4 wk = cw[d_inner + c];
      const float bk = cb[d_inner + c];
      float val[Q];
      float r0 = bf16f(sm.raw[buf][0][CROWS + c]), r1 = bf16f(sm.raw[buf][1][CROWS + c]),
            r2 = bf16f(sm.raw[buf][2][CROWS + c]);
#pragma unroll
      for (int v = 0; v < Q; ++v) {
        const float r3 = bf16f(sm.raw[buf][v + 3][CROWS + c]);
        val[v] = v < cnt ? silu_fast(conv4_acc(wk, bk, r0, r1, r2, r3)) : 0.f;
        r0 = r1;
        r1 = r2;
        r2 = r3;
      }
      const int col = c & (kN - 1), odd = c & 1;
      if (c < kN) {  // B: pairs along the nodes for the update
#pragma unroll
        for (int k = 0; k < Q / 2; ++k) split_bf16x2(val[2 * k], val[2 * k + 1], sm.bhi[col][k], sm.blo[col][k]);
      }
      // pairs along the columns (B for the Gram, C for C·h and the Gram): even lanes nodes 0..7,
      // odd lanes nodes 8..15, each pair = (even column, odd column)
      uint32_t(*phi)[CPS] = c < kN ? sm.bchi : sm.chi;
      uint32_t(*plo)[CPS] = c < kN ? sm.bclo : sm.clo;
#pragma unroll
      for (int v = 0; v < Q; ++v) {
        const float nb = __shfl_xor_sync(0xffffffffu, val[v], 1);
        if ((v < Q / 2) != (odd != 0)) {
          const float e0 = odd ? nb : val[v], e1 = odd ? val[v] : nb;
          split_bf16x2(e0, e1, phi[v][col >> 1], plo[v][col >> 1]);
        }
      }
    }
    __syncthreads();

    // ---- phase 2: x conv + SiLU into x and u = w·x pairs (threads 0..127); the Gram (warps 4, 5) ----
    if (tid < CROWS) {
      const int hx = tid / kP;
      float4 wk = make_float4(0.f, 0.f, 0.f, 0.f);
      float bk = 0.f;
      if (hx < heads) {
        const int c = (h_begin + hx) * kP + (tid - hx * kP);
        wk = cw[c];
        bk = cb[c];
      }
      float val[Q];
      float r0 = bf16f(sm.raw[buf][0][tid]), r1 = bf16f(sm.raw[buf][1][tid]), r2 = bf16f(sm.raw[buf][2][tid]);
#pragma unroll
      for (int v = 0; v < Q; ++v) {
        const float r3 = bf16f(sm.raw[buf][v + 3][tid]);
        val[v] = (v < cnt && hx < heads) ? silu_fast(conv4_acc(wk, bk, r0, r1, r2, r3)) : 0.f;
        r0 = r1;
        r1 = r2;
        r2 = r3;
      }
#pragma unroll
      for (int k = 0; k < Q / 2; ++k) {
        split_bf16x2(val[2 * k], val[2 * k + 1], sm.xhi[tid][k], sm.xlo[tid][k]);
        split_bf16x2(sm.w[hx][2 * k] * val[2 * k], sm.w[hx][2 * k + 1] * val[2 * k + 1], sm.uhi[tid][k],
                     sm.ulo[tid][k]);
      }
    } else if (warp == 4 || warp == 5) {
      // Gram[v][m] = C_v·B_m: M = 16 nodes v, N = 8 nodes m of this warp, K = the 128 columns
      const int nt = warp - 4;
      float g4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < kN / 16; ++ks) {
        const int kk = 8 * ks + ft;
        const uint32_t ahi[4] = {sm.chi[fg][kk], sm.chi[fg + 8][kk], sm.chi[fg][kk + 4], sm.chi[fg + 8][kk + 4]};
        const uint32_t alo[4] = {sm.clo[fg][kk], sm.clo[fg + 8][kk], sm.clo[fg][kk + 4], sm.clo[fg + 8][kk + 4]};
        const int m = nt * 8 + fg;
        const uint32_t bh[2] = {sm.bchi[m][kk], sm.bchi[m][kk + 4]};
        const uint32_t bl[2] = {sm.bclo[m][kk], sm.bclo[m][kk + 4]};
        mma_bf16(g4, alo, bh);
        mma_bf16(g4, ahi, bl);
        mma_bf16(g4, ahi, bh);
      }
      const int m = nt * 8 + 2 * ft;
      sm.gram[fg][m] = g4[0];
      sm.gram[fg][m + 1] = g4[1];
      sm.gram[fg + 8][m] = g4[2];
      sm.gram[fg + 8][m + 1] = g4[3];
    }
    __syncthreads();

    // ---- phase 3: coef pairs along m (thread = head, node v, pair k) ----
    {
      const int hx = tid / (Q * (Q / 2)), rest = tid - hx * (Q * (Q / 2)), v = rest / (Q / 2), k = rest - v * (Q / 2);
      const float Dh = hx < heads ? a.D[(size_t)layer * a.H + h_begin + hx] : 0.f;
      float cm[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int m = 2 * k + e;
        float c = m <= v ? sm.emS[hx][m] * sm.dl[hx][m] * sm.gram[v][m] : 0.f;
        if (m == v) c = fmaf(Dh, sm.emS[hx][v], c);
        cm[e] = c;
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
#pragma unroll
      for (int ks = 0; ks < kN / 16; ++ks) {
        uint32_t ahi[4], alo[4];
        split_bf16x2(st[2 * ks][0], st[2 * ks][1], ahi[0], alo[0]);
        split_bf16x2(st[2 * ks][2], st[2 * ks][3], ahi[1], alo[1]);
        split_bf16x2(st[2 * ks + 1][0], st[2 * ks + 1][1], ahi[2], alo[2]);
        split_bf16x2(st[2 * ks + 1][2], st[2 * ks + 1][3], ahi[3], alo[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int v = nt * 8 + fg;
          const uint32_t bh[2] = {sm.chi[v][8 * ks + ft], sm.chi[v][8 * ks + ft + 4]};
          const uint32_t bl[2] = {sm.clo[v][8 * ks + ft], sm.clo[v][8 * ks + ft + 4]};
          mma_bf16(acc[nt], alo, bh);
          mma_bf16(acc[nt], ahi, bl);
          mma_bf16(acc[nt], ahi, bh);
        }
      }
      // y_v[p] = e^{S_v}·acc
      float* yb = a.y + (size_t)inst * n * d_inner + (size_t)(h_begin * kP + rbase + fg);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int v = nt * 8 + 2 * ft + c;
          if (v < cnt) {
            const float es = sm.eS[hh][v];
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
      const float E = sm.E[hh];
#pragma unroll
      for (int j = 0; j < kN / 8; ++j) {
        const int col = 8 * j + fg;
        const uint32_t bh[2] = {sm.bhi[col][ft], sm.bhi[col][ft + 4]};
        const uint32_t bl[2] = {sm.blo[col][ft], sm.blo[col][ft + 4]};
#pragma unroll
        for (int e = 0; e < 4; ++e) st[j][e] *= E;
        mma_bf16(st[j], ulo, bh);
        mma_bf16(st[j], uhi, bl);
        mma_bf16(st[j], uhi, bh);
      }
    }
  }
}

}  // namespace

cudaError_t launch_chain_verify(const VerifyArgs& a, cudaStream_t s) {
  const long long blocks = (long long)a.n_seq * a.L * ((a.H + CHG - 1) / CHG);
  if (blocks == 0) return cudaSuccess;
  const int bytes = (int)sizeof(ChainSmem);
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(chain_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = 1;
  }
  chain_verify_kernel<<<(unsigned)blocks, CTHREADS, bytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ssmtree
