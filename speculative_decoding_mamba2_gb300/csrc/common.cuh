// Device helpers shared by the libssmtree kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_tree.h"

namespace ssmtree {

// Shape constants of this library: Mamba2 head_dim 64, d_state 128, conv width 4.
constexpr int kP = 64;
constexpr int kN = 128;
constexpr int kW = 4;

// bf16 bit pattern -> fp32 (exact).
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// The two bf16 values of a 32-bit word (low half = lower channel) -> fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

// SiLU with the fast exp/divide intrinsics (relative error ~1e-6 on the
// conv outputs' range); below -80 the result is below 1e-33 and returned as 0.
__device__ __forceinline__ float silu_fast(float v) {
  return v < -80.0f ? 0.0f : __fdividef(v, 1.0f + __expf(-v));
}

// SiLU on the FMA pipe only (no special-function unit), for conv work that runs next to
// tensor-core work: v / (1 + 2^t), t = -v·log2(e), with v first raised to -87 (below it the
// exact result is under 2e-36 in magnitude, and silu(-87) is returned, about -1.4e-36).
//  * 2^t: t <= 125.5 after that, and t is raised to -126 (large v give v); Cody-Waite range
//    reduction -- n = round(t) by adding and subtracting 1.5·2^23, f = t - n in [-1/2, 1/2] --
//    then the degree-6 Taylor series of 2^f = e^{f·ln 2} (coefficients (ln 2)^k / k!,
//    remainder about 1e-7 on that interval), scaled by 2^n through the exponent field.
//  * 1 / d: Newton-Raphson r <- r·(2 - d·r), three steps from the linear bit-pattern guess
//    0x7F000000 - bits(d) (relative error below 1/8, then 2^-6, 2^-12, 2^-24).
// Relative error of the result about 4e-6, like the special-function version above.
__device__ __forceinline__ float exp2_poly(float t) {  // t in [-126, 126]
  const float m = t + 12582912.0f;  // 1.5·2^23: m's low mantissa bits hold round(t)
  const float f = t - (m - 12582912.0f);
  float p = 1.5403530393381608e-4f;
  p = fmaf(p, f, 1.3333558146428443e-3f);
  p = fmaf(p, f, 9.618129107628477e-3f);
  p = fmaf(p, f, 5.550410866482158e-2f);
  p = fmaf(p, f, 2.402265069591007e-1f);
  p = fmaf(p, f, 6.931471805599453e-1f);
  p = fmaf(p, f, 1.0f);
  return __int_as_float(__float_as_int(p) + (__float_as_int(m) - 0x4B400000) * (1 << 23));
}
__device__ __forceinline__ float recip_nr(float d) {
  float r = __int_as_float(0x7F000000 - __float_as_int(d));
#pragma unroll
  for (int i = 0; i < 3; ++i) r = fmaf(r, fmaf(-d, r, 1.0f), r);
  return r;
}
__device__ __forceinline__ float silu_fma(float v) {
  const float vc = fmaxf(v, -87.0f);
  return vc * recip_nr(1.0f + exp2_poly(fmaxf(-1.4426950408889634f * vc, -126.0f)));
}

// softplus(v) = log(1 + e^v); above 20 it equals v to fp32 precision.
__device__ __forceinline__ float softplus_f(float v) { return v > 20.0f ? v : log1pf(expf(v)); }

// A = -exp(A_log) and the per-head decay exp(Δ·A).  Written with explicit
// round-to-nearest operations so the draft step and the replay (which must
// agree bit for bit) cannot be contracted differently by the compiler.
__device__ __forceinline__ float neg_exp(float a_log) { return -expf(a_log); }
__device__ __forceinline__ float decay_of(float delta, float A) { return expf(__fmul_rn(delta, A)); }

// One element of the state update h' = a·h + (Δ·x)·B with u = Δ·x precomputed.
__device__ __forceinline__ float ssm_update(float a, float h, float u, float b) {
  return __fmaf_rn(a, h, __fmul_rn(u, b));
}

__device__ __forceinline__ int ring_pos(int head, int offset, int R) {
  int p = (head + offset) % R;
  return p < 0 ? p + R : p;
}

// Causal width-4 conv + SiLU for one channel given the four pre-conv values,
// oldest first: SiLU(b + w0·r0 + w1·r1 + w2·r2 + w3·r3).
__device__ __forceinline__ float conv4_silu(float4 w, float b, float r0, float r1, float r2, float r3) {
  float acc = b;
  acc = fmaf(w.x, r0, acc);
  acc = fmaf(w.y, r1, acc);
  acc = fmaf(w.z, r2, acc);
  acc = fmaf(w.w, r3, acc);
  return silu_f(acc);
}

// b + w0·r0 + w1·r1 + w2·r2 + w3·r3 (the conv before its SiLU), taps oldest first.
__device__ __forceinline__ float conv4_acc(float4 w, float b, float r0, float r1, float r2, float r3) {
  float acc = fmaf(w.x, r0, b);
  acc = fmaf(w.y, r1, acc);
  acc = fmaf(w.z, r2, acc);
  return fmaf(w.w, r3, acc);
}

// Pre-conv value of channel c for tap source `src` of a tree node: a node row
// of this instance's xBC (src >= 0) or a ring row (src = -j: position head - j).
__device__ __forceinline__ float tap_value(const uint16_t* __restrict__ xbc, const uint16_t* __restrict__ ring,
                                           int head, int R, int conv_dim, int src, int c) {
  if (src >= 0) return bf16f(xbc[(size_t)src * conv_dim + c]);
  return bf16f(ring[(size_t)ring_pos(head, src, R) * conv_dim + c]);
}

// Post-conv value of channel c at tree node v (taps from its layout record).
__device__ __forceinline__ float node_conv(const uint16_t* __restrict__ xbc, const uint16_t* __restrict__ ring,
                                           int head, int R, int conv_dim, const int* tap /*[3]: d=1,2,3*/, int v,
                                           int c, float4 w, float b) {
  float r0 = tap_value(xbc, ring, head, R, conv_dim, tap[2], c);
  float r1 = tap_value(xbc, ring, head, R, conv_dim, tap[1], c);
  float r2 = tap_value(xbc, ring, head, R, conv_dim, tap[0], c);
  float r3 = bf16f(xbc[(size_t)v * conv_dim + c]);
  return conv4_silu(w, b, r0, r1, r2, r3);
}

// Packed fp32 FMA on a pair of lanes held in one 64-bit register:
// d = a * b + c element-wise (sm_100+ `fma.rn.f32x2`), round-to-nearest.
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Packed pairs of fp32 (lower half = first value) for the f32x2 instructions.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(unsigned long long p) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(p));
  return r;
}
// d = a * b element-wise on a pair, round-to-nearest (sm_100+ `mul.rn.f32x2`).
__device__ __forceinline__ unsigned long long fmul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float pair_sum(unsigned long long p) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
  return lo + hi;
}

// fp32 -> (hi, lo) TF32 pair with hi + lo = x to ~2^-22 relative (round-to-nearest splits)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  const float r = x - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

// fp32 pair (x0, x1) -> packed bf16x2 hi (x0 in the lower half) and packed bf16x2 lo of the
// residuals: x = hi + lo to 2^-18 relative (round-to-nearest both times).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(x1), "f"(x0));
  const float r0 = x0 - __uint_as_float(hi << 16);
  const float r1 = x1 - __uint_as_float(hi & 0xffff0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(r1), "f"(r0));
}

// D += A·B on one m16n8k16 tile (bf16 inputs, fp32 accumulate), warp-wide.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// D += A·B on one m16n8k8 tile (TF32 inputs, fp32 accumulate), warp-wide.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void flag(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// cp.async (16-byte global -> shared, bypassing L1)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA) helpers.  Every wait is bounded: after one second
// of global time (or kWaitLimit unsuccessful polls, whichever comes first) it
// gives up and returns false, and the caller reports SSM_STATUS_TIMEOUT instead
// of spinning forever.
// ---------------------------------------------------------------------------
constexpr unsigned kWaitLimit = 1u << 26;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long global_time_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
// make initialised barriers visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// wait for phase `parity` of `bar`; false once limit_ns of global time (or kWaitLimit polls)
// have passed without it
// (the clock is first read after 64 unsuccessful polls, so a wait that succeeds at once costs
// no timer read)
__device__ __forceinline__ bool mbar_wait_ns(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  unsigned long long t0 = 0;
  for (unsigned it = 0; it < kWaitLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      const unsigned long long now = global_time_ns();
      if (t0 == 0)
        t0 = now;
      else if (now - t0 > limit_ns)
        return false;
    }
  }
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  return mbar_wait_ns(bar, parity, kWaitLimitNs);
}
// Programmatic dependent launch: the primary grid lets its dependent grid be scheduled;
// the dependent waits until the primary grid has completed and its writes are visible
// (a no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// 2-D tiled bulk tensor copy global -> shared, completion counted on `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// contiguous bulk copy global -> shared (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Kernel launchers (defined in the .cu files, called by api.cu).
struct VerifyArgs {
  int H, L, R, n_seq, n, max_depth;
  int gpc;      // head groups per CTA (set by launch_verify)
  int prep_hb;  // CTAs per instance of the prep kernel (set by launch_verify)
  const float *conv_w, *conv_b, *dt_bias, *A_log, *D;
  const ssm_node* layout;
  const uint16_t *xBC, *dt, *ring;
  const float* h0;
  const int32_t* ring_head;
  float* y;
  int32_t* status;
  // commit of the previous step's accepted path folded into this verify (LP = 0: plain verify).
  // LP bounds the path length; h_w / ring_w / head_w are the writable views of h0 / ring / ring_head.
  int LP, prev_n;
  const ssm_node* prev_layout;
  const int32_t *prev_path, *prev_path_len;
  const uint16_t *prev_xBC, *prev_dt;
  float* h_w;
  uint16_t* ring_w;
  int32_t* head_w;
};
// which: 0 = prep + main, 1 = prep only, 2 = main only (after a prep on the same workspace)
cudaError_t launch_verify(const VerifyArgs& a, void* workspace, cudaStream_t s, int which);
size_t verify_workspace_bytes(int n, int max_depth, int H, long long n_inst, int LP = 0);
int verify_heads_per_group(int n, int max_depth, int H, int LP = 0);  // 0: the plan does not fit in shared memory
int verify_prep_smem_bytes(int n, int max_depth, int H, int LP = 0);
// The same calls with the state contraction on tcgen05 (verify_tc.cu); launch_verify routes
// trees here unless the SSM_VERIFY_KERNEL override selects the warp-level kernels above.
cudaError_t launch_verify_tc(const VerifyArgs& a, void* workspace, cudaStream_t s, int which);
size_t verify_tc_workspace_bytes(int n, int max_depth, int H, int LP, long long n_inst);
bool verify_tc_fits(int n, int max_depth, int LP);
// Launch-plan overrides (0 = automatic).  Each starts at its environment variable, read once
// per process; ssm_set_tuning replaces it.  They never change results beyond rounding order.
enum TuneKey { TUNE_VERIFY_GPC, TUNE_VERIFY_G, TUNE_LINEAR_TCHUNK, TUNE_LINEAR_SPLITS, TUNE_LINEAR_STAGES,
               TUNE_VERIFY_KERNEL, TUNE_VERIFY_CTAS, TUNE_VERIFY_DEEP, TUNE_COUNT };
int tuning(TuneKey k);

// Projections (gemm.cu): D = A · Wᵀ (+ residual) with the output columns cut into segments.
struct GemmArgs {
  int M, N, K;
  int n_seg;
  int seg_col[4];         // first column of each segment (multiples of the tile width)
  long long seg_ld[4];    // row stride of each segment's output, elements
  int seg_f32[4];         // 1: fp32 output, 0: bf16
  void* seg_ptr[4];
  const float* residual;  // nullptr or fp32 [M][ldr], added to the accumulator
  long long ldr;
  int32_t* status;
  int tn, tchunk, splits, kb_per_split, tmem_cols, stages;  // tile plan, set by launch_gemm_bf16
};
int gemm_tile_cols();
cudaError_t launch_gemm_bf16(GemmArgs g, const void* A, long long lda, const void* W, long long ldw, cudaStream_t s);
// Row norms (norm.cu): RMSNorm of fp32 rows, and the gated form of y ⊙ SiLU(z).
cudaError_t launch_rmsnorm(int M, int C, const float* x, long long ldx, const uint16_t* z, long long ldz,
                           const float* w, float eps, uint16_t* out, long long ldo, cudaStream_t s);

// Chain trees: workspace bytes (one record per instance and 16-node chunk) and the launch.
size_t chain_workspace_bytes(int n, int H, long long n_inst);
cudaError_t launch_chain_verify(const VerifyArgs& a, void* workspace, cudaStream_t s);

struct AcceptArgs {
  int n_seq, n, max_path;
  const ssm_node* layout;
  const int32_t *tok, *tgt;
  int32_t *path, *path_len, *bonus, *status;
};
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s);

struct CommitArgs {
  int H, L, R, n_seq, n, max_path;
  const float *conv_w, *conv_b, *dt_bias, *A_log;
  const ssm_node* layout;
  const int32_t *path, *path_len;
  const uint16_t *xBC, *dt;
  float* h;
  uint16_t* ring;
  int32_t *ring_head, *status;
};
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s);

struct DraftArgs {
  int H, L, R, n_seq, step, log_cap;
  const float *conv_w, *conv_b, *dt_bias, *A_log, *D;
  const uint16_t *xBC_t, *dt_t;
  const float* h_in;
  float* h_out;
  uint16_t* ring;
  const int32_t* ring_head;
  float *log_delta, *log_B, *log_x;
  int32_t* log_len;
  float* y;
  int32_t* status;
};
cudaError_t launch_draft_step(const DraftArgs& a, cudaStream_t s);

struct ReplayArgs {
  int H, L, n_seq, log_cap;
  const float* A_log;
  const int32_t* k;
  const float *log_delta, *log_B, *log_x;
  int32_t* log_len;
  float* h;
  int32_t *ring_head, *status;
};
cudaError_t launch_replay(const ReplayArgs& a, cudaStream_t s);

// the bounded-wait self-test (one CTA waits on a barrier nothing arrives at)
cudaError_t launch_selftest_wait(int32_t* status, unsigned long long limit_ns, cudaStream_t s);
cudaError_t launch_selftest_silu(const float* v, float* out, long long n, cudaStream_t s);

}  // namespace ssmtree
