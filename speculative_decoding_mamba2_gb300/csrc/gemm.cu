// The projections of a Mamba2 block on the 5th-generation tensor cores.
//
// LightMamba page ("为什么 Mamba 难加速"): a Mamba block projects each token to
// X, B, C, Δ and Z (the input projection), runs X through the conv and the SSM,
// multiplies the SSM output by Z and projects back (the output projection).  Both
// projections are dense products of the tokens with a weight matrix:
//     D[t, o] = Σ_k A[t, k] · W[o, k]          (bf16 inputs, fp32 accumulation)
// with W stored row-major [out features][in features] (K contiguous), A [tokens][K].
//
// gemm_bf16_kernel is built for few tokens and wide weights (a decode/verify batch: a few
// hundred tokens against megabytes of weights), where the weights must stream from HBM once:
//  * the MMA computes Dᵀ = W · tokensᵀ: a CTA (4 warps) owns 128 output features (the MMA's
//    M, TMEM lanes), all tokens of a chunk of up to 256 (the MMA's N) and one K-split, so
//    each weight tile is read by exactly one CTA and each MMA does 128 x N x 16;
//  * each CTA loads its own weight tile and the chunk's token tile with 2-D bulk tensor copies
//    (TMA); a CTA runs alone (no cluster), so every copy lands in its own shared memory;
//  * K-splits, chosen on the host to fill the SMs, accumulate into an fp32 output with
//    vector reductions (used by the output projection, which adds into the residual
//    stream anyway);
//  * warp 0 feeds a ring of as many stages as shared memory holds (a stage is refilled once
//    the MMAs that read it have completed: their commit arrives on the stage's `empty`
//    barrier), warp 1 issues tcgen05.mma (operands from shared memory
//    through 128-byte-swizzle matrix descriptors) and commits; after the last k-block all
//    four warps read the accumulator (tcgen05.ld, warp w = TMEM lanes 32w..) into the now
//    idle stage memory as a [token][feature] tile and write it out row by row with
//    coalesced vector stores.
// The epilogue writes up to four column segments to separate outputs (the input
// projection's z, x|B|C and dt land where the next kernels read them), bf16 or fp32,
// optionally adding an fp32 residual.  Every wait on an mbarrier is bounded and polled by one
// thread while its warp (or the CTA) waits at a hardware barrier; a CTA that gives up waits
// (bounded again) for the copies it issued before it leaves.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace ssmtree {
namespace {

constexpr int GBK = 64, GTHREADS = 128;
constexpr int FM = 128;                            // output features per CTA (MMA M, TMEM lanes)
constexpr int MAX_TN = 256;                        // tokens per CTA (MMA N)
constexpr int MAX_STAGES = 8;
constexpr int GEMM_SMEM = 227 * 1024;              // the stage ring takes what the tile plan fits in here
constexpr int GEMM_RESERVED = 1024 /* alignment */ + 512 /* barriers */;
constexpr int SEG_ALIGN = 16;                      // segment boundaries: multiples of the narrowest tile

// ---- tcgen05 / TMEM helpers (inline PTX) ----
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the 128-byte swizzle:
// rows of 128 bytes, groups of 8 rows 1024 bytes apart (stride byte offset); the leading byte
// offset is not used by this layout.  Bits: start address >> 4 [0, 14), leading offset >> 4
// [16, 30), stride offset >> 4 [32, 46), descriptor version 1 [46, 48), swizzle mode [61, 64)
// (2 = 128-byte swizzle).  The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16 for bf16 x bf16 -> fp32, both operands K-major:
// D format [4, 6) = 1 (f32), A format [7, 10) = 1 (bf16), B format [10, 13) = 1 (bf16),
// transpose bits 15, 16 = 0, N >> 3 at [17, 23), M >> 4 at [24, 29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on `bar` once every tcgen05.mma this thread issued so far has completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Wait for phase `parity` of `bar` by polling the non-blocking test_wait from ONE thread (the
// rest of its warp or CTA waits at a hardware barrier): a thread suspended in try_wait is not
// always woken as soon as an asynchronous arrival (a bulk copy, an MMA commit) completes the
// phase.  Gives up after about one second of global time and returns false.
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  for (unsigned it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 1023) == 1023 && global_ns() - t0 > 1000000000ull) return false;
  }
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(GTHREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tw, GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int TN = g.tn, GSTAGES = g.stages;
  const int w_stage = FM * GBK * 2, t_stage = TN * GBK * 2;  // both multiples of 1024
  unsigned char* sw = smem;                      // [GSTAGES][w_stage]: weight rows (MMA operand A)
  unsigned char* st = smem + GSTAGES * w_stage;  // [GSTAGES][t_stage]: token rows (MMA operand B)
  unsigned long long* full = reinterpret_cast<unsigned long long*>(st + GSTAGES * t_stage);
  unsigned long long* empty = full + MAX_STAGES;
  unsigned long long* acc_bar = empty + MAX_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* issued = abort_flag + 1;  // k-blocks whose copies the producer issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f0 = blockIdx.x * FM, t0 = blockIdx.z * g.tchunk;
  const int KB = (g.K + GBK - 1) / GBK;
  const int kb0 = blockIdx.y * g.kb_per_split, kb1 = min(KB, kb0 + g.kb_per_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < GSTAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_bar), 1);
    *abort_flag = 0;
    *issued = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), (uint32_t)g.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Warp 0 feeds the ring and warp 1 issues the MMAs; each whole warp runs its loop (every lane
  // waits on the same barriers, lane 0 issues).
  if (warp == 0) {  // producer: this CTA's weight tile and the chunk's token tile
    for (int kb = kb0; kb < kb1; ++kb) {
      const int i = kb - kb0, s = i % GSTAGES, use = i / GSTAGES;
      int bad = 0;
      if (lane == 0) {
        if (use > 0 && !mbar_poll(smem_u32(&empty[s]), (use - 1) & 1)) {
          *abort_flag = 1;
          bad = 1;
        } else {
          mbar_arrive_expect_tx(smem_u32(&full[s]), (uint32_t)(w_stage + t_stage));
          tma_load_2d(smem_u32(sw + s * w_stage), &tw, kb * GBK, f0, smem_u32(&full[s]));
          tma_load_2d(smem_u32(st + s * t_stage), &ta, kb * GBK, t0, smem_u32(&full[s]));
          *issued = i + 1;
        }
      }
      if (__shfl_sync(0xffffffffu, bad, 0)) break;
    }
  } else if (warp == 1) {  // MMA issuer: D[128 features][TN tokens] += W · tokensᵀ
    const uint32_t idesc = idesc_bf16_f32(FM, TN);
    for (int kb = kb0; kb < kb1; ++kb) {
      const int i = kb - kb0, s = i % GSTAGES, use = i / GSTAGES;
      int bad = 0;
      if (lane == 0) {
        // no tcgen05 fence: the copies and the MMAs are both in the async proxy, and the
        // barrier's completion already orders the stage's data before the MMAs that read it
        if (*abort_flag || !mbar_poll(smem_u32(&full[s]), use & 1)) {
          *abort_flag = 1;
          bad = 1;
        } else {
          const uint64_t wd = desc_sw128(smem_u32(sw + s * w_stage));
          const uint64_t td = desc_sw128(smem_u32(st + s * t_stage));
#pragma unroll
          for (int k = 0; k < GBK / 16; ++k)  // next 16 columns: 32 bytes further in the swizzled rows
            umma_bf16(tmem, wd + 2 * k, td + 2 * k, idesc, (i | k) != 0);
          umma_commit(smem_u32(&empty[s]));  // the stage is free once these MMAs complete
        }
      }
      if (__shfl_sync(0xffffffffu, bad, 0)) break;
    }
    if (lane == 0) umma_commit(smem_u32(acc_bar));  // the accumulator is complete
    __syncwarp();
  }

  // ---- epilogue: thread = one output feature (TMEM lane); 16 tokens per tcgen05.ld ----
  // one thread watches the accumulator barrier; the CTA waits for it at a hardware barrier
  if (threadIdx.x == 64 && !mbar_poll(smem_u32(acc_bar), 0)) *abort_flag = 1;
  __syncthreads();
  tc_fence_after();
  if (*abort_flag) {  // CTA-uniform after the barrier: tcgen05.ld needs whole warps
    if (threadIdx.x == 0) {
      flag(g.status, SSM_STATUS_TIMEOUT);
      // copies issued into stages that no MMA waited for may still be in flight: give each
      // stage's latest use a bounded chance to land before the CTA's shared memory is released
      const int n_issued = *issued;
      for (int i = n_issued > GSTAGES ? n_issued - GSTAGES : 0; i < n_issued; ++i)
        mbar_poll(smem_u32(&full[i % GSTAGES]), (i / GSTAGES) & 1);
    }
  } else {
    // (1) accumulator -> shared memory, [token][feature] fp32 (the stage ring is free now: the
    //     last MMA has read it and every copy into it has landed)
    float* tile = reinterpret_cast<float*>(smem);  // TN x FM fp32 <= 128 KB
    const int fl = warp * 32 + lane;               // this thread's feature within the tile
#pragma unroll 1
    for (int c0 = 0; c0 < TN; c0 += 16) {
      float v[16];
      __syncwarp();
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);  // the whole warp takes part
#pragma unroll
      for (int i = 0; i < 16; ++i) tile[(c0 + i) * FM + fl] = v[i];  // lanes: consecutive words
    }
    __syncthreads();
    // (2) token rows out: 32 threads per row, 4 features each; a thread keeps its group of 4
    //     features (which lies in one segment) for every row, so the segment is resolved once
    const bool accumulate = g.splits > 1;  // fp32 output holding the residual: add the partial sums
    const int rows = min(TN, g.M - t0);
    const int fg = 4 * (threadIdx.x & (FM / 4 - 1)), f = f0 + fg;
    if (f < g.N) {
      int seg = 0;
      while (seg + 1 < g.n_seg && f >= g.seg_col[seg + 1]) ++seg;
      const int seg_end = seg + 1 < g.n_seg ? g.seg_col[seg + 1] : g.N;
      const int nc = min(4, seg_end - f);
      const bool vec = nc == 4 && seg_end - g.seg_col[seg] >= 16;  // 16-byte row strides guaranteed
      const long long ld = g.seg_ld[seg];
      const bool f32 = g.seg_f32[seg] != 0;
      unsigned char* base = static_cast<unsigned char*>(g.seg_ptr[seg]) +
                            (size_t)(f - g.seg_col[seg]) * (f32 || accumulate ? 4 : 2);
      const float* res = g.residual ? g.residual + f : nullptr;
      const long long ldr = g.ldr;
#pragma unroll 4
      for (int tr = threadIdx.x / (FM / 4); tr < rows; tr += GTHREADS / (FM / 4)) {
        const int t = t0 + tr;
        float4 v = *reinterpret_cast<const float4*>(tile + tr * FM + fg);
        if (accumulate) {
          float* d = reinterpret_cast<float*>(base) + (size_t)t * ld;
          if (vec) {
            atomicAdd(reinterpret_cast<float4*>(d), v);
          } else {
            const float vv[4] = {v.x, v.y, v.z, v.w};
            for (int i = 0; i < nc; ++i) atomicAdd(d + i, vv[i]);
          }
          continue;
        }
        if (res) {
          const float* rr = res + (size_t)t * ldr;
          v.x += rr[0];
          if (nc > 1) v.y += rr[1];
          if (nc > 2) v.z += rr[2];
          if (nc > 3) v.w += rr[3];
        }
        if (f32) {
          float* d = reinterpret_cast<float*>(base) + (size_t)t * ld;
          if (vec) {
            *reinterpret_cast<float4*>(d) = v;
          } else {
            const float vv[4] = {v.x, v.y, v.z, v.w};
            for (int i = 0; i < nc; ++i) d[i] = vv[i];
          }
        } else {
          uint16_t* d = reinterpret_cast<uint16_t*>(base) + (size_t)t * ld;
          if (vec) {
            *reinterpret_cast<uint2*>(d) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
          } else {
            const float vv[4] = {v.x, v.y, v.z, v.w};
            for (int i = 0; i < nc; ++i) d[i] = (uint16_t)(pack_bf16(vv[i], 0.f) & 0xffffu);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)g.tmem_cols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 gemm_encode_fn() {
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

// rows x cols bf16 matrix (row stride ld elements) as a 2-D tensor map with 128 x 64 boxes
bool encode_bf16(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = gemm_encode_fn();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)GBK, (cuuint32_t)box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int gemm_tile_cols() { return SEG_ALIGN; }

// Tile plan: 128 output features per CTA (the MMA's M), all tokens of a chunk of up to 256
// (the MMA's N, rounded up to a multiple of 16), and K-splits (only when the output is an fp32
// accumulator) so the grid fills the SMs with the least data per SM.  Tuning overrides:
// tokens per CTA, K-splits and ring stages (ssm_set_tuning).
void plan_gemm(GemmArgs& g, int sms, bool can_split) {
  const int o_tchunk = tuning(TUNE_LINEAR_TCHUNK);  // 64, 128 or 256 tokens per CTA
  const int o_splits = tuning(TUNE_LINEAR_SPLITS);  // K-splits (fp32 accumulator outputs only)
  const int o_stages = tuning(TUNE_LINEAR_STAGES);  // stages of the copy ring
  const int KB = (g.K + GBK - 1) / GBK;
  const int tiles = (g.N + FM - 1) / FM;
  // few feature tiles (a narrow projection) and no K-splits (a bf16 output): cut the tokens into
  // smaller chunks so more CTAs, each with a deeper ring of smaller stages, share the work
  g.tchunk = MAX_TN;
  while (!can_split && g.tchunk > 64 && g.M > g.tchunk / 2 &&
         (long long)tiles * ((g.M + g.tchunk / 2 - 1) / (g.tchunk / 2)) <= sms / 2)
    g.tchunk /= 2;
  if (o_tchunk == 64 || o_tchunk == 128 || o_tchunk == 256) g.tchunk = o_tchunk;
  const int chunk = g.M < g.tchunk ? g.M : g.tchunk;
  g.tn = (chunk + 15) / 16 * 16;
  const int tchunks = (g.M + g.tchunk - 1) / g.tchunk;
  double best = 1e300;
  g.splits = 1;
  g.kb_per_split = KB;
  for (int sp = 1; sp <= (can_split ? 16 : 1); ++sp) {
    const int kbp = (KB + sp - 1) / sp;
    if ((sp - 1) * kbp >= KB) continue;  // every split gets at least one k-block
    const long long ctas = (long long)tiles * sp * tchunks;
    const long long waves = (ctas + sms - 1) / sms;
    const double per_cta = (double)kbp * GBK * 2 * (FM + (double)g.tn);
    const double est = waves * per_cta * (1.0 + 0.02 * sp);  // small charge per split (reductions)
    if (est < best * 0.999) {
      best = est;
      g.splits = sp;
      g.kb_per_split = kbp;
    }
  }
  if (o_splits >= 1 && (o_splits == 1 || can_split) && (o_splits - 1) * ((KB + o_splits - 1) / o_splits) < KB) {
    g.splits = o_splits;
    g.kb_per_split = (KB + o_splits - 1) / o_splits;
  }
  int cols = 32;
  while (cols < g.tn) cols *= 2;
  g.tmem_cols = cols;
  const int stage_bytes = (FM + g.tn) * GBK * 2;
  g.stages = (GEMM_SMEM - GEMM_RESERVED) / stage_bytes;
  if (g.stages > MAX_STAGES) g.stages = MAX_STAGES;
  // the epilogue stages the fp32 [token][feature] tile in the ring's memory
  const int min_stages = (g.tn * FM * 4 + stage_bytes - 1) / stage_bytes;
  if (o_stages >= 2 && o_stages >= min_stages && o_stages < g.stages) g.stages = o_stages;
}

// dynamic shared memory of a plan: the stage ring (which also holds the epilogue tile), the
// barriers and the 1024-byte alignment of the ring
int gemm_smem_bytes(const GemmArgs& g) { return GEMM_RESERVED + g.stages * (FM + g.tn) * GBK * 2; }

cudaError_t launch_gemm_bf16(GemmArgs g, const void* A, long long lda, const void* W, long long ldw, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int configured[64] = {0};
  static int sm_count[64] = {0};
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) {
      sm_count[dev] = sms;
      configured[dev] = 1;
    }
  }
  const int sms = dev < 64 ? sm_count[dev] : 148;
  // K-splits add partial sums into the output: only for one fp32 segment that is its own residual
  const bool can_split = g.n_seg == 1 && g.seg_f32[0] && g.residual == g.seg_ptr[0] && g.ldr == g.seg_ld[0];
  plan_gemm(g, sms, can_split);
  CUtensorMap ta, tw;
  if (!encode_bf16(&ta, A, g.M, g.K, lda, g.tn) || !encode_bf16(&tw, W, g.N, g.K, ldw, FM))
    return cudaErrorInvalidValue;
  const int tiles = (g.N + FM - 1) / FM;
  const dim3 grid((unsigned)tiles, (unsigned)g.splits, (unsigned)((g.M + g.tchunk - 1) / g.tchunk));
  gemm_bf16_kernel<<<grid, GTHREADS, (size_t)gemm_smem_bytes(g), s>>>(ta, tw, g);
  return cudaGetLastError();
}

}  // namespace ssmtree
