// C ABI of the block's dense steps (ssm_layer.h): host-side validation, then launches.
#include <stdint.h>
#include <stdio.h>

#include <string>

#include "common.cuh"
#include "ssm_layer.h"

namespace ssmtree {
void set_error(const std::string& msg);
}

using namespace ssmtree;

namespace {

int lfail(int code, const char* fn, const char* what) {
  char buf[320];
  snprintf(buf, sizeof buf, "%s: %s", fn, what);
  set_error(buf);
  return code;
}

int lfinish(const char* fn, cudaError_t e) {
  if (e != cudaSuccess) {
    char buf[320];
    snprintf(buf, sizeof buf, "%s: CUDA error %d (%s)", fn, (int)e, cudaGetErrorString(e));
    set_error(buf);
    return SSM_ERR_CUDA;
  }
  set_error("");
  return SSM_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

int check_norm(const char* fn, int32_t M, int32_t C, const void* x, int64_t ldx, const float* w, const void* out,
               int64_t ldo) {
  if (M < 0) return lfail(SSM_ERR_INVALID_ARG, fn, "M must be >= 0");
  if (C < 1 || C > 8192) return lfail(SSM_ERR_INVALID_ARG, fn, "C must be in [1, 8192]");
  if (M > 0 && (!x || !w || !out)) return lfail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (ldx < C || ldo < C) return lfail(SSM_ERR_INVALID_ARG, fn, "row strides must be >= C");
  return SSM_OK;
}

}  // namespace

extern "C" int32_t ssm_linear_tile_cols(void) { return gemm_tile_cols(); }

extern "C" int ssm_linear(int32_t M, int32_t N, int32_t K, const uint16_t* A, int64_t lda, const uint16_t* W,
                          int64_t ldw, int32_t n_seg, const ssm_out_segment* seg, const float* residual,
                          int64_t ldr, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_linear";
  if (M < 0 || N < 1 || K < 1) return lfail(SSM_ERR_INVALID_ARG, fn, "need M >= 0, N >= 1, K >= 1");
  if (!A || !W) return lfail(SSM_ERR_INVALID_ARG, fn, "A or W is NULL");
  if (lda < K || ldw < K || (lda & 7) || (ldw & 7))
    return lfail(SSM_ERR_INVALID_ARG, fn, "lda and ldw must be >= K and multiples of 8");
  if (!aligned16(A) || !aligned16(W)) return lfail(SSM_ERR_INVALID_ARG, fn, "A and W must be 16-byte aligned");
  if (n_seg < 1 || n_seg > 4 || !seg) return lfail(SSM_ERR_INVALID_ARG, fn, "n_seg must be in [1, 4]");
  const int tile = gemm_tile_cols();
  GemmArgs g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.n_seg = n_seg;
  for (int i = 0; i < n_seg; ++i) {
    const ssm_out_segment& s = seg[i];
    if (!s.ptr) return lfail(SSM_ERR_INVALID_ARG, fn, "a segment pointer is NULL");
    if (i == 0 ? s.col != 0 : (s.col <= seg[i - 1].col || s.col >= N))
      return lfail(SSM_ERR_INVALID_ARG, fn, "segment columns must start at 0, increase and stay below N");
    if (s.col % tile) return lfail(SSM_ERR_INVALID_ARG, fn, "segment columns must be multiples of the tile width");
    const int end = i + 1 < n_seg ? seg[i + 1].col : N;
    if (s.ld < end - s.col) return lfail(SSM_ERR_INVALID_ARG, fn, "a segment's ld is below its width");
    // 16-column chunks are stored as 16-byte vectors: a segment at least that wide needs
    // 16-byte row strides; narrower ones are stored element by element
    if (!aligned16(s.ptr) || (end - s.col >= 16 && (s.f32 ? (s.ld & 3) : (s.ld & 7))))
      return lfail(SSM_ERR_INVALID_ARG, fn,
                   "segment outputs must be 16-byte aligned, with 16-byte row strides when 16 or more columns wide");
    g.seg_col[i] = s.col;
    g.seg_ld[i] = s.ld;
    g.seg_f32[i] = s.f32 ? 1 : 0;
    g.seg_ptr[i] = s.ptr;
  }
  if (residual && ldr < N) return lfail(SSM_ERR_INVALID_ARG, fn, "ldr must be >= N");
  g.residual = residual;
  g.ldr = ldr;
  g.status = dev_status;
  return lfinish(fn, launch_gemm_bf16(g, A, lda, W, ldw, (cudaStream_t)stream));
}

extern "C" int ssm_rmsnorm(int32_t M, int32_t C, const float* x, int64_t ldx, const float* w, float eps,
                           uint16_t* out, int64_t ldo, void* stream) {
  const char* fn = "ssm_rmsnorm";
  if (int rc = check_norm(fn, M, C, x, ldx, w, out, ldo)) return rc;
  return lfinish(fn, launch_rmsnorm(M, C, x, ldx, nullptr, 0, w, eps, out, ldo, (cudaStream_t)stream));
}

extern "C" int ssm_gated_rmsnorm(int32_t M, int32_t C, const float* y, int64_t ldy, const uint16_t* z, int64_t ldz,
                                 const float* w, float eps, uint16_t* out, int64_t ldo, void* stream) {
  const char* fn = "ssm_gated_rmsnorm";
  if (int rc = check_norm(fn, M, C, y, ldy, w, out, ldo)) return rc;
  if (M > 0 && !z) return lfail(SSM_ERR_INVALID_ARG, fn, "z is NULL");
  if (ldz < C) return lfail(SSM_ERR_INVALID_ARG, fn, "ldz must be >= C");
  return lfinish(fn, launch_rmsnorm(M, C, y, ldy, z, ldz, w, eps, out, ldo, (cudaStream_t)stream));
}
