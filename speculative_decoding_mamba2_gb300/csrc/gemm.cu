// The projections of a Mamba2 block on the 5th-generation tensor cores.
//
// LightMamba page ("为什么 Mamba 难加速"): a Mamba block projects each token to
// X, B, C, Δ and Z (the input projection), runs X through the conv and the SSM,
// multiplies the SSM output by Z and projects back (the output projection).  Both
// projections are dense products of the tokens with a weight matrix:
//     D[t, o] = Σ_k A[t, k] · W[o, k]          (bf16 inputs, fp32 accumulation)
// with W stored row-major [out features][in features] (K contiguous), A [tokens][K].
//
// gemm_bf16_kernel: one CTA (4 warps) per 128 x 128 output tile.  Thread 0 issues
// tensor-map bulk copies (TMA, 128-byte swizzle) of 128 x 64 tiles of A and W into a
// 4-stage shared-memory ring; thread 32 issues tcgen05.mma (M = 128, N = 128, K = 16,
// both operands from shared memory through matrix descriptors) into one fp32 TMEM
// accumulator and hands each stage back with tcgen05.commit; after the last k-block
// all four warps read the accumulator (tcgen05.ld, each warp its 32 TMEM lanes = rows)
// and store it.  The epilogue writes up to four column segments to separate outputs
// (the input projection's z, x|B|C and dt land where the next kernels read them),
// as bf16 or fp32, optionally adding an fp32 residual (the output projection updates
// the residual stream in place).  Every wait on an mbarrier is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace ssmtree {
namespace {

constexpr int GBM = 128, GBN = 128, GBK = 64, GSTAGES = 4, GTHREADS = 128;
constexpr int A_STAGE = GBM * GBK * 2;  // 16 KB: 128 rows of 128 bytes
constexpr int B_STAGE = GBN * GBK * 2;  // 16 KB
constexpr int TMEM_COLS = GBN;          // one fp32 accumulator column per output column
constexpr int GEMM_SMEM = GSTAGES * (A_STAGE + B_STAGE) + 1024 /* alignment */ + 256 /* barriers */;

static_assert(TMEM_COLS >= 32 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM is allocated in powers of two >= 32");

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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(GTHREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tw, GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* sa = smem;                              // [GSTAGES][A_STAGE]
  unsigned char* sw = smem + GSTAGES * A_STAGE;          // [GSTAGES][B_STAGE]
  unsigned long long* full = reinterpret_cast<unsigned long long*>(sw + GSTAGES * B_STAGE);
  unsigned long long* empty = full + GSTAGES;
  unsigned long long* acc_bar = empty + GSTAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * GBM, n0 = blockIdx.y * GBN;
  const int KB = (g.K + GBK - 1) / GBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GSTAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {  // producer: TMA tiles of A (tokens) and W (features)
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % GSTAGES, use = kb / GSTAGES;
      if (use > 0 && !mbar_wait(smem_u32(&empty[s]), (use - 1) & 1)) {
        *abort_flag = 1;
        break;
      }
      mbar_arrive_expect_tx(smem_u32(&full[s]), A_STAGE + B_STAGE);
      tma_load_2d(smem_u32(sa + s * A_STAGE), &ta, kb * GBK, m0, smem_u32(&full[s]));
      tma_load_2d(smem_u32(sw + s * B_STAGE), &tw, kb * GBK, n0, smem_u32(&full[s]));
    }
  } else if (threadIdx.x == 32) {  // MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(GBM, GBN);
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % GSTAGES, use = kb / GSTAGES;
      if (*abort_flag || !mbar_wait(smem_u32(&full[s]), use & 1)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint64_t ad = desc_sw128(smem_u32(sa + s * A_STAGE));
      const uint64_t wd = desc_sw128(smem_u32(sw + s * B_STAGE));
#pragma unroll
      for (int k = 0; k < GBK / 16; ++k)  // next 16 columns: 32 bytes further in the swizzled rows
        umma_bf16(tmem, ad + 2 * k, wd + 2 * k, idesc, (kb | k) != 0);
      umma_commit(smem_u32(&empty[s]));  // the stage is free once these have read it
    }
    umma_commit(smem_u32(acc_bar));  // the accumulator is complete
  }

  // ---- epilogue: warp w holds rows m0 + 32w .. m0 + 32w + 31 (TMEM lanes 32w ..) ----
  const bool ok = mbar_wait(smem_u32(acc_bar), 0);
  __syncwarp();
  tc_fence_after();
  if (__any_sync(0xffffffffu, !ok || *abort_flag)) {  // warp-uniform: tcgen05.ld needs the whole warp
    if (threadIdx.x == 0) flag(g.status, SSM_STATUS_TIMEOUT);
  } else {
    int seg = 0;
    while (seg + 1 < g.n_seg && n0 >= g.seg_col[seg + 1]) ++seg;
    const int seg_end = seg + 1 < g.n_seg ? g.seg_col[seg + 1] : g.N;
    const int row = m0 + warp * 32 + lane;
    const long long ld = g.seg_ld[seg];
    const int c_base = n0 - g.seg_col[seg];  // column of this tile inside its segment
    const int cols = min(GBN, seg_end - n0);
#pragma unroll 1
    for (int c0 = 0; c0 < GBN; c0 += 16) {
      float v[16];
      __syncwarp();
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);  // warp-wide: every lane takes part
      if (row >= g.M || c0 >= cols) continue;
      const int nc = min(16, cols - c0);
      if (g.residual) {
        const float* rr = g.residual + (size_t)row * g.ldr + n0 + c0;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < nc) v[i] += rr[i];
      }
      if (g.seg_f32[seg]) {
        float* d = static_cast<float*>(g.seg_ptr[seg]) + (size_t)row * ld + c_base + c0;
        if (nc == 16) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4*>(d + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < nc) d[i] = v[i];
        }
      } else {
        uint16_t* d = static_cast<uint16_t*>(g.seg_ptr[seg]) + (size_t)row * ld + c_base + c0;
        if (nc == 16) {
          uint4 p0, p1;
          p0.x = pack_bf16(v[0], v[1]);
          p0.y = pack_bf16(v[2], v[3]);
          p0.z = pack_bf16(v[4], v[5]);
          p0.w = pack_bf16(v[6], v[7]);
          p1.x = pack_bf16(v[8], v[9]);
          p1.y = pack_bf16(v[10], v[11]);
          p1.z = pack_bf16(v[12], v[13]);
          p1.w = pack_bf16(v[14], v[15]);
          reinterpret_cast<uint4*>(d)[0] = p0;
          reinterpret_cast<uint4*>(d)[1] = p1;
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < nc) d[i] = (uint16_t)(pack_bf16(v[i], 0.f) & 0xffffu);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
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

int gemm_tile_cols() { return GBN; }

cudaError_t launch_gemm_bf16(const GemmArgs& g, const void* A, long long lda, const void* W, long long ldw,
                             cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  CUtensorMap ta, tw;
  if (!encode_bf16(&ta, A, g.M, g.K, lda, GBM) || !encode_bf16(&tw, W, g.N, g.K, ldw, GBN))
    return cudaErrorInvalidValue;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = 1;
  }
  const dim3 grid((unsigned)((g.M + GBM - 1) / GBM), (unsigned)((g.N + GBN - 1) / GBN));
  gemm_bf16_kernel<<<grid, GTHREADS, GEMM_SMEM, s>>>(ta, tw, g);
  return cudaGetLastError();
}

}  // namespace ssmtree
