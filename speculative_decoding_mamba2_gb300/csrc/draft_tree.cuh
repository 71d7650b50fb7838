// Launch arguments of the draft-tree kernels (draft_tree.cu).
#pragma once

#include "common.cuh"

namespace ssmtree {

// One depth level of each sequence's draft tree.
struct DraftTreeArgs {
  int H, L, R, n_seq, n, level;
  const float *conv_w, *conv_b, *dt_bias, *A_log, *D;
  const ssm_node* layout;               // [S][n]
  const uint16_t *xBC, *dt;             // [I][n][conv_dim], [I][n][H]
  const float* h;                       // [I][H][P][N] committed draft state (read only)
  const uint16_t* ring;                 // [I][R][conv_dim]
  const int32_t* ring_head;             // [I]
  float *log_delta, *log_B, *log_x;     // [I][n][H], [I][n][N], [I][n][d_inner]
  float* y;                             // [I][n][d_inner]
  int32_t* status;
};
// workspace: per instance the level's C rows, e^{S_v} and path sums, draft_tree_workspace_bytes()
size_t draft_tree_workspace_bytes(int n, int H, long long n_inst);
cudaError_t launch_draft_tree_level(const DraftTreeArgs& a, void* workspace, cudaStream_t s);

// The accepted path's logged updates into the committed draft state, its rows into the ring.
struct DraftTreeCommitArgs {
  int H, L, R, n_seq, n, max_path;
  const float* A_log;
  const ssm_node* layout;
  const int32_t *path, *path_len;       // [S][max_path], [S]
  const float *log_delta, *log_B, *log_x;
  const uint16_t* xBC;                  // [I][n][conv_dim]
  float* h;
  uint16_t* ring;
  int32_t *ring_head, *status;
};
cudaError_t launch_draft_tree_commit(const DraftTreeCommitArgs& a, cudaStream_t s);

}  // namespace ssmtree
