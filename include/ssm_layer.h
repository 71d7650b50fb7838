/*
 * ssm_layer.h -- the dense steps around the selective-SSM path of a Mamba2 block,
 * so that a whole block can verify a draft tree on the GPU:
 *
 *   x (residual stream, fp32) -> RMSNorm -> input projection -> z | x B C | dt
 *   -> conv + SSM over the tree (ssm_tree.h) -> y -> y · SiLU(z), RMSNorm
 *   -> output projection, added to x.
 *
 * The block structure is the one the LightMamba page ("为什么 Mamba 难加速")
 * describes: the input projection makes X, B, C, Δ and Z; X goes through the conv
 * and the SSM; the output Y is multiplied by Z and projected back.  The page names
 * an RMSNorm before the input projection and a second one after the SSM
 * ("旋转辅助量化"); the gated form y · SiLU(z) followed by RMSNorm is Mamba2's, the
 * reading this library takes.
 *
 * Same conventions as ssm_tree.h: device pointers are caller-owned, every call is
 * asynchronous on `stream` (NULL = the legacy default stream), returns an SSM_*
 * status and leaves a message for ssm_last_error() on failure.
 */
#ifndef SSM_LAYER_H_
#define SSM_LAYER_H_

#include <stdint.h>

#include "ssm_tree.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One output column segment of ssm_linear: columns [col, next segment's col) of
 * the product land in ptr[row * ld + (column - col)], as bf16 (f32 = 0) or fp32
 * (f32 = 1).  ptr is 16-byte aligned; a segment 16 or more columns wide needs ld a
 * multiple of 8 (bf16) or 4 (fp32). */
typedef struct {
  int32_t col;
  int32_t f32;
  int64_t ld;
  void *ptr;
} ssm_out_segment;

/*
 * ssm_linear -- a projection of the block: D[t][o] = sum_k A[t][k] * W[o][k]
 * (+ residual[t][o]), bf16 operands, fp32 accumulation on the tensor cores
 * (tcgen05, accumulator in tensor memory).
 *   M, N, K     tokens, output features, input features (all >= 1)
 *   A           device bf16 [M][lda], lda >= K, lda a multiple of 8, 16-byte aligned
 *   W           device bf16 [N][ldw] (row-major by output feature), same rules
 *   n_seg, seg  1..4 output segments; seg[0].col = 0, cols increasing, each a
 *               multiple of ssm_linear_tile_cols() and < N
 *   residual    NULL, or device fp32 [M][ldr] added to the accumulator; it may be
 *               the output itself (one fp32 segment over all columns: x += D)
 *   dev_status  NULL or device int32: SSM_STATUS_TIMEOUT if a bounded wait on a
 *               copy gave up (the output is then not valid)
 * Errors: SSM_ERR_INVALID_ARG for NULL pointers, bad sizes, strides or alignment;
 * SSM_ERR_CUDA for a launch failure.
 */
int ssm_linear(int32_t M, int32_t N, int32_t K, const uint16_t *A, int64_t lda, const uint16_t *W, int64_t ldw,
               int32_t n_seg, const ssm_out_segment *seg, const float *residual, int64_t ldr, int32_t *dev_status,
               void *stream);

/* Column tile of ssm_linear (segment boundaries are multiples of it). */
int32_t ssm_linear_tile_cols(void);

/*
 * ssm_rmsnorm -- out[t][c] = w[c] * x[t][c] / sqrt(mean_c x[t][c]^2 + eps).
 *   x    device fp32 [M][ldx]     w   device fp32 [C]
 *   out  device bf16 [M][ldo]     1 <= C <= 8192
 */
int ssm_rmsnorm(int32_t M, int32_t C, const float *x, int64_t ldx, const float *w, float eps, uint16_t *out,
                int64_t ldo, void *stream);

/*
 * ssm_gated_rmsnorm -- g = y * SiLU(z), out[t][c] = w[c] * g[t][c] / sqrt(mean_c g[t][c]^2 + eps).
 *   y    device fp32 [M][ldy] (the SSM output)   z   device bf16 [M][ldz]
 *   w    device fp32 [C]                          out device bf16 [M][ldo]
 */
int ssm_gated_rmsnorm(int32_t M, int32_t C, const float *y, int64_t ldy, const uint16_t *z, int64_t ldz,
                      const float *w, float eps, uint16_t *out, int64_t ldo, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_LAYER_H_ */
