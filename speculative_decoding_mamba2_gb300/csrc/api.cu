// libssmtree C ABI: argument validation on the host, then kernel launches on
// the caller's stream.  Nothing here allocates device memory.
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <stddef.h>

#include <string>

#include "common.cuh"
#include "draft_tree.cuh"

namespace ssmtree {

static thread_local std::string g_error;

void set_error(const std::string& msg) { g_error = msg; }

namespace {

int fail(int code, const char* fn, const char* what) {
  char buf[320];
  snprintf(buf, sizeof buf, "%s: %s", fn, what);
  g_error = buf;
  return code;
}

int cuda_fail(const char* fn, cudaError_t e) {
  char buf[320];
  snprintf(buf, sizeof buf, "%s: CUDA error %d (%s)", fn, (int)e, cudaGetErrorString(e));
  g_error = buf;
  return SSM_ERR_CUDA;
}

// Shape checks common to every device call.
int check_dims(const char* fn, const ssm_dims* d, bool need_params, const ssm_params* p) {
  if (!d) return fail(SSM_ERR_INVALID_ARG, fn, "dims is NULL");
  if (d->n_heads < 1) return fail(SSM_ERR_INVALID_ARG, fn, "n_heads must be >= 1");
  if (d->head_dim != kP) return fail(SSM_ERR_INVALID_ARG, fn, "head_dim must be 64 in this library");
  if (d->d_state != kN) return fail(SSM_ERR_INVALID_ARG, fn, "d_state must be 128 in this library");
  if (d->conv_width != kW) return fail(SSM_ERR_INVALID_ARG, fn, "conv_width must be 4");
  if (d->n_layers < 1) return fail(SSM_ERR_INVALID_ARG, fn, "n_layers must be >= 1");
  if (d->ring_cap < 3) return fail(SSM_ERR_INVALID_ARG, fn, "ring_cap must be >= 3");
  if ((long long)d->n_heads * kP > (1 << 24)) return fail(SSM_ERR_CAPACITY, fn, "n_heads too large");
  if (need_params) {
    if (!p) return fail(SSM_ERR_INVALID_ARG, fn, "params is NULL");
    if (!p->conv_w || !p->conv_b || !p->dt_bias || !p->A_log || !p->D)
      return fail(SSM_ERR_INVALID_ARG, fn, "a parameter pointer is NULL");
  }
  return SSM_OK;
}

int finish(const char* fn, cudaError_t e) {
  if (e != cudaSuccess) return cuda_fail(fn, e);
  g_error.clear();
  return SSM_OK;
}

}  // namespace
}  // namespace ssmtree

using namespace ssmtree;

extern "C" int32_t ssm_version(void) { return 100; }

extern "C" const char* ssm_last_error(void) { return g_error.c_str(); }

namespace {
const char* const kTuneNames[TUNE_COUNT] = {"SSM_VERIFY_GROUPS_PER_CTA", "SSM_VERIFY_HEADS_PER_GROUP",
                                            "SSM_LINEAR_TCHUNK",         "SSM_LINEAR_SPLITS",
                                            "SSM_LINEAR_STAGES",         "SSM_VERIFY_KERNEL",
                                            "SSM_VERIFY_CTAS",           "SSM_VERIFY_DEEP"};
struct TuneTable {
  int v[TUNE_COUNT];
  TuneTable() {
    for (int k = 0; k < TUNE_COUNT; ++k) {
      const char* e = getenv(kTuneNames[k]);
      const int x = e ? atoi(e) : 0;
      v[k] = x > 0 ? x : 0;
    }
  }
};
TuneTable& tune_table() {
  static TuneTable t;  // environment read once, on first use
  return t;
}
}  // namespace

int ssmtree::tuning(TuneKey k) { return tune_table().v[k]; }

extern "C" int ssm_set_tuning(const char* name, int32_t value) {
  static const char* fn = "ssm_set_tuning";
  if (!name) return fail(SSM_ERR_INVALID_ARG, fn, "name is NULL");
  if (value < 0) return fail(SSM_ERR_INVALID_ARG, fn, "value must be >= 0");
  for (int k = 0; k < TUNE_COUNT; ++k)
    if (strcmp(name, kTuneNames[k]) == 0) {
      tune_table().v[k] = value;
      g_error.clear();
      return SSM_OK;
    }
  return fail(SSM_ERR_INVALID_ARG, fn, "unknown tuning name");
}

namespace {
// A tree whose deepest node sits at depth n-1 is a chain; long chains take the chain kernel.
bool long_chain(int32_t n_nodes, int32_t max_depth) {
  return max_depth == n_nodes - 1 && max_depth > SSM_MAX_DEPTH;
}

int check_verify_shape(const char* fn, const ssm_dims* dims, int32_t n_seq, int32_t n_nodes, int32_t max_depth) {
  if (int rc = check_dims(fn, dims, false, nullptr)) return rc;
  if (n_seq < 0) return fail(SSM_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
  if (n_nodes < 1) return fail(SSM_ERR_INVALID_ARG, fn, "n_nodes must be >= 1");
  if (max_depth < 0 || max_depth >= n_nodes) return fail(SSM_ERR_RANGE, fn, "max_depth must be in [0, n_nodes)");
  if (long_chain(n_nodes, max_depth)) {
    if (n_nodes > SSM_MAX_CHAIN_NODES) return fail(SSM_ERR_CAPACITY, fn, "chain longer than SSM_MAX_CHAIN_NODES");
    return SSM_OK;
  }
  if (n_nodes > SSM_MAX_NODES) return fail(SSM_ERR_CAPACITY, fn, "n_nodes exceeds SSM_MAX_NODES");
  if (max_depth > SSM_MAX_DEPTH) return fail(SSM_ERR_CAPACITY, fn, "max_depth exceeds SSM_MAX_DEPTH");
  if (verify_heads_per_group(n_nodes, max_depth, dims->n_heads) == 0 ||
      verify_prep_smem_bytes(n_nodes, max_depth, dims->n_heads) > 232448)
    return fail(SSM_ERR_CAPACITY, fn, "tree too large for the shared-memory plan of this library");
  return SSM_OK;
}
}  // namespace

extern "C" size_t ssm_tree_verify_workspace_size(const ssm_dims* dims, int32_t n_seq, int32_t n_nodes,
                                                 int32_t max_depth) {
  const char* fn = "ssm_tree_verify_workspace_size";
  if (check_verify_shape(fn, dims, n_seq, n_nodes, max_depth) != SSM_OK) return 0;
  g_error.clear();
  const size_t b = long_chain(n_nodes, max_depth)
                       ? chain_workspace_bytes(n_nodes, dims->n_heads, (long long)n_seq * dims->n_layers)
                       : verify_workspace_bytes(n_nodes, max_depth, dims->n_heads, (long long)n_seq * dims->n_layers);
  return b ? b : 16;
}

extern "C" int ssm_tree_verify(const ssm_dims* dims, const ssm_params* prm, int32_t n_seq, int32_t n_nodes,
                               int32_t max_depth, const ssm_node* layout, const uint16_t* xBC, const uint16_t* dt,
                               const float* h0, const uint16_t* ring, const int32_t* ring_head, float* y,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_tree_verify";
  if (int rc = check_verify_shape(fn, dims, n_seq, n_nodes, max_depth)) return rc;
  if (int rc = check_dims(fn, dims, true, prm)) return rc;
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!layout || !xBC || !dt || !h0 || !ring || !ring_head || !y || !workspace)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (((uintptr_t)xBC | (uintptr_t)h0 | (uintptr_t)ring | (uintptr_t)layout | (uintptr_t)workspace) & 15)
    return fail(SSM_ERR_INVALID_ARG, fn, "xBC, h0, ring, layout and workspace must be 16-byte aligned");
  const bool chain = long_chain(n_nodes, max_depth);
  const long long n_inst = (long long)n_seq * dims->n_layers;
  if (workspace_bytes < (chain ? chain_workspace_bytes(n_nodes, dims->n_heads, n_inst)
                               : verify_workspace_bytes(n_nodes, max_depth, dims->n_heads, n_inst)))
    return fail(SSM_ERR_CAPACITY, fn, "workspace smaller than ssm_tree_verify_workspace_size()");
  VerifyArgs a{};
  a.gpc = 1;
  a.H = dims->n_heads;
  a.L = dims->n_layers;
  a.R = dims->ring_cap;
  a.n_seq = n_seq;
  a.n = n_nodes;
  a.max_depth = max_depth;
  a.conv_w = prm->conv_w;
  a.conv_b = prm->conv_b;
  a.dt_bias = prm->dt_bias;
  a.A_log = prm->A_log;
  a.D = prm->D;
  a.layout = layout;
  a.xBC = xBC;
  a.dt = dt;
  a.ring = ring;
  a.h0 = h0;
  a.ring_head = ring_head;
  a.y = y;
  a.status = dev_status;
  return finish(fn, chain ? launch_chain_verify(a, workspace, (cudaStream_t)stream)
                         : launch_verify(a, workspace, (cudaStream_t)stream, 0));
}

namespace {
int check_commit_verify_shape(const char* fn, const ssm_dims* dims, int32_t n_seq, int32_t prev_n_nodes,
                              int32_t prev_max_path, int32_t n_nodes, int32_t max_depth) {
  if (int rc = check_verify_shape(fn, dims, n_seq, n_nodes, max_depth)) return rc;
  if (long_chain(n_nodes, max_depth))
    return fail(SSM_ERR_CAPACITY, fn, "chain trees deeper than SSM_MAX_DEPTH take ssm_commit + ssm_tree_verify");
  if (prev_n_nodes < 1 || prev_n_nodes > SSM_MAX_NODES)
    return fail(SSM_ERR_RANGE, fn, "prev_n_nodes must be in [1, SSM_MAX_NODES]");
  if (prev_max_path < 1 || prev_max_path > SSM_MAX_DEPTH + 1)
    return fail(SSM_ERR_RANGE, fn, "prev_max_path must be in [1, SSM_MAX_DEPTH + 1]");
  if (dims->ring_cap < prev_max_path + 3)
    return fail(SSM_ERR_CAPACITY, fn, "ring_cap must be >= prev_max_path + 3 (the rows before the path are read after the path is written)");
  if (verify_heads_per_group(n_nodes, max_depth, dims->n_heads, prev_max_path) == 0 ||
      verify_prep_smem_bytes(n_nodes, max_depth, dims->n_heads, prev_max_path) > 232448)
    return fail(SSM_ERR_CAPACITY, fn, "tree and path too large for the shared-memory plan of this library");
  return SSM_OK;
}
}  // namespace

extern "C" size_t ssm_commit_verify_workspace_size(const ssm_dims* dims, int32_t n_seq, int32_t n_nodes,
                                                   int32_t max_depth, int32_t prev_max_path) {
  const char* fn = "ssm_commit_verify_workspace_size";
  if (check_commit_verify_shape(fn, dims, n_seq, 1, prev_max_path, n_nodes, max_depth) != SSM_OK) return 0;
  g_error.clear();
  const size_t b =
      verify_workspace_bytes(n_nodes, max_depth, dims->n_heads, (long long)n_seq * dims->n_layers, prev_max_path);
  return b ? b : 16;
}

namespace {
// which: 0 = the whole folded call, 1 = its prep kernel only, 2 = its main kernel only
int commit_verify_call(const char* fn, int which, const ssm_dims* dims, const ssm_params* prm, int32_t n_seq,
                       int32_t prev_n_nodes, const ssm_node* prev_layout, int32_t prev_max_path,
                       const int32_t* prev_path, const int32_t* prev_path_len, const uint16_t* prev_xBC,
                       const uint16_t* prev_dt, int32_t n_nodes, int32_t max_depth, const ssm_node* layout,
                       const uint16_t* xBC, const uint16_t* dt, float* h, uint16_t* ring, int32_t* ring_head, float* y,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (int rc = check_commit_verify_shape(fn, dims, n_seq, prev_n_nodes, prev_max_path, n_nodes, max_depth)) return rc;
  if (int rc = check_dims(fn, dims, true, prm)) return rc;
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!prev_layout || !prev_path || !prev_path_len || !prev_xBC || !prev_dt || !layout || !xBC || !dt || !h || !ring ||
      !ring_head || !y || !workspace)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (((uintptr_t)prev_xBC | (uintptr_t)xBC | (uintptr_t)h | (uintptr_t)ring | (uintptr_t)layout |
       (uintptr_t)workspace) & 15)
    return fail(SSM_ERR_INVALID_ARG, fn, "prev_xBC, xBC, h, ring, layout and workspace must be 16-byte aligned");
  if (workspace_bytes <
      verify_workspace_bytes(n_nodes, max_depth, dims->n_heads, (long long)n_seq * dims->n_layers, prev_max_path))
    return fail(SSM_ERR_CAPACITY, fn, "workspace smaller than ssm_commit_verify_workspace_size()");
  VerifyArgs a{};
  a.gpc = 1;
  a.H = dims->n_heads;
  a.L = dims->n_layers;
  a.R = dims->ring_cap;
  a.n_seq = n_seq;
  a.n = n_nodes;
  a.max_depth = max_depth;
  a.conv_w = prm->conv_w;
  a.conv_b = prm->conv_b;
  a.dt_bias = prm->dt_bias;
  a.A_log = prm->A_log;
  a.D = prm->D;
  a.layout = layout;
  a.xBC = xBC;
  a.dt = dt;
  a.ring = ring;
  a.h0 = h;
  a.ring_head = ring_head;
  a.y = y;
  a.status = dev_status;
  a.LP = prev_max_path;
  a.prev_n = prev_n_nodes;
  a.prev_layout = prev_layout;
  a.prev_path = prev_path;
  a.prev_path_len = prev_path_len;
  a.prev_xBC = prev_xBC;
  a.prev_dt = prev_dt;
  a.h_w = h;
  a.ring_w = ring;
  a.head_w = ring_head;
  return finish(fn, launch_verify(a, workspace, (cudaStream_t)stream, which));
}
}  // namespace

#define SSM_COMMIT_VERIFY_ARGS                                                                                      \
  const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t prev_n_nodes, const ssm_node *prev_layout,   \
      int32_t prev_max_path, const int32_t *prev_path, const int32_t *prev_path_len, const uint16_t *prev_xBC,     \
      const uint16_t *prev_dt, int32_t n_nodes, int32_t max_depth, const ssm_node *layout, const uint16_t *xBC,     \
      const uint16_t *dt, float *h, uint16_t *ring, int32_t *ring_head, float *y, void *workspace,                 \
      size_t workspace_bytes, int32_t *dev_status, void *stream
#define SSM_COMMIT_VERIFY_PASS                                                                                      \
  dims, prm, n_seq, prev_n_nodes, prev_layout, prev_max_path, prev_path, prev_path_len, prev_xBC, prev_dt, n_nodes, \
      max_depth, layout, xBC, dt, h, ring, ring_head, y, workspace, workspace_bytes, dev_status, stream

extern "C" int ssm_commit_verify(SSM_COMMIT_VERIFY_ARGS) {
  return commit_verify_call("ssm_commit_verify", 0, SSM_COMMIT_VERIFY_PASS);
}
extern "C" int ssm_commit_verify_prep(SSM_COMMIT_VERIFY_ARGS) {
  return commit_verify_call("ssm_commit_verify_prep", 1, SSM_COMMIT_VERIFY_PASS);
}
extern "C" int ssm_commit_verify_main(SSM_COMMIT_VERIFY_ARGS) {
  return commit_verify_call("ssm_commit_verify_main", 2, SSM_COMMIT_VERIFY_PASS);
}

extern "C" int ssm_accept_path(int32_t n_seq, int32_t n_nodes, int32_t max_path, const ssm_node* layout,
                               const int32_t* tok, const int32_t* tgt, int32_t* path, int32_t* path_len,
                               int32_t* bonus, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_accept_path";
  if (n_seq < 0) return fail(SSM_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
  if (n_nodes < 1) return fail(SSM_ERR_INVALID_ARG, fn, "n_nodes must be >= 1");
  if (max_path < 1 || max_path > SSM_MAX_PATH) return fail(SSM_ERR_RANGE, fn, "max_path must be in [1, SSM_MAX_PATH]");
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!layout || !tok || !tgt || !path || !path_len || !bonus)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  AcceptArgs a;
  a.n_seq = n_seq;
  a.n = n_nodes;
  a.max_path = max_path;
  a.layout = layout;
  a.tok = tok;
  a.tgt = tgt;
  a.path = path;
  a.path_len = path_len;
  a.bonus = bonus;
  a.status = dev_status;
  return finish(fn, launch_accept(a, (cudaStream_t)stream));
}

extern "C" int ssm_commit(const ssm_dims* dims, const ssm_params* prm, int32_t n_seq, int32_t n_nodes,
                          const ssm_node* layout, int32_t max_path, const int32_t* path, const int32_t* path_len,
                          const uint16_t* xBC, const uint16_t* dt, float* h, uint16_t* ring, int32_t* ring_head,
                          int32_t* dev_status, void* stream) {
  const char* fn = "ssm_commit";
  if (int rc = check_dims(fn, dims, true, prm)) return rc;
  if (n_seq < 0) return fail(SSM_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
  if (n_nodes < 1) return fail(SSM_ERR_INVALID_ARG, fn, "n_nodes must be >= 1");
  if (max_path < 1 || max_path > SSM_MAX_PATH) return fail(SSM_ERR_RANGE, fn, "max_path must be in [1, SSM_MAX_PATH]");
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!layout || !path || !path_len || !xBC || !dt || !h || !ring || !ring_head)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (((uintptr_t)xBC | (uintptr_t)h | (uintptr_t)ring) & 15)
    return fail(SSM_ERR_INVALID_ARG, fn, "xBC, h and ring must be 16-byte aligned");
  CommitArgs a;
  a.H = dims->n_heads;
  a.L = dims->n_layers;
  a.R = dims->ring_cap;
  a.n_seq = n_seq;
  a.n = n_nodes;
  a.max_path = max_path;
  a.conv_w = prm->conv_w;
  a.conv_b = prm->conv_b;
  a.dt_bias = prm->dt_bias;
  a.A_log = prm->A_log;
  a.layout = layout;
  a.path = path;
  a.path_len = path_len;
  a.xBC = xBC;
  a.dt = dt;
  a.h = h;
  a.ring = ring;
  a.ring_head = ring_head;
  a.status = dev_status;
  return finish(fn, launch_commit(a, (cudaStream_t)stream));
}

extern "C" int ssm_draft_step(const ssm_dims* dims, const ssm_params* prm, int32_t n_seq, int32_t step,
                              int32_t log_cap, const uint16_t* xBC_t, const uint16_t* dt_t, const float* h_in,
                              float* h_out, uint16_t* ring, const int32_t* ring_head, float* log_delta, float* log_B,
                              float* log_x, int32_t* log_len, float* y, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_draft_step";
  if (int rc = check_dims(fn, dims, true, prm)) return rc;
  if (n_seq < 0) return fail(SSM_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
  if (log_cap < 1) return fail(SSM_ERR_INVALID_ARG, fn, "log_cap must be >= 1");
  if (step < 0 || step >= log_cap) return fail(SSM_ERR_RANGE, fn, "step must be in [0, log_cap)");
  if (step + 3 >= dims->ring_cap)
    return fail(SSM_ERR_CAPACITY, fn, "ring_cap too small: need step + 3 < ring_cap so the committed rows survive");
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!xBC_t || !dt_t || !h_in || !h_out || !ring || !ring_head || !log_delta || !log_B || !log_x || !log_len || !y)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (((uintptr_t)h_in | (uintptr_t)h_out) & 15) return fail(SSM_ERR_INVALID_ARG, fn, "h_in and h_out must be 16-byte aligned");
  DraftArgs a;
  a.H = dims->n_heads;
  a.L = dims->n_layers;
  a.R = dims->ring_cap;
  a.n_seq = n_seq;
  a.step = step;
  a.log_cap = log_cap;
  a.conv_w = prm->conv_w;
  a.conv_b = prm->conv_b;
  a.dt_bias = prm->dt_bias;
  a.A_log = prm->A_log;
  a.D = prm->D;
  a.xBC_t = xBC_t;
  a.dt_t = dt_t;
  a.h_in = h_in;
  a.h_out = h_out;
  a.ring = ring;
  a.ring_head = ring_head;
  a.log_delta = log_delta;
  a.log_B = log_B;
  a.log_x = log_x;
  a.log_len = log_len;
  a.y = y;
  a.status = dev_status;
  return finish(fn, launch_draft_step(a, (cudaStream_t)stream));
}

extern "C" int ssm_replay(const ssm_dims* dims, const ssm_params* prm, int32_t n_seq, int32_t log_cap,
                          const int32_t* k, const float* log_delta, const float* log_B, const float* log_x,
                          int32_t* log_len, float* h_ckpt, int32_t* ring_head, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_replay";
  if (int rc = check_dims(fn, dims, false, nullptr)) return rc;
  if (!prm || !prm->A_log) return fail(SSM_ERR_INVALID_ARG, fn, "params->A_log is NULL");
  if (n_seq < 0) return fail(SSM_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
  if (log_cap < 1) return fail(SSM_ERR_INVALID_ARG, fn, "log_cap must be >= 1");
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!k || !log_delta || !log_B || !log_x || !log_len || !h_ckpt || !ring_head)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (((uintptr_t)h_ckpt | (uintptr_t)log_B) & 15)
    return fail(SSM_ERR_INVALID_ARG, fn, "h_ckpt and log_B must be 16-byte aligned");
  ReplayArgs a;
  a.H = dims->n_heads;
  a.L = dims->n_layers;
  a.n_seq = n_seq;
  a.log_cap = log_cap;
  a.A_log = prm->A_log;
  a.k = k;
  a.log_delta = log_delta;
  a.log_B = log_B;
  a.log_x = log_x;
  a.log_len = log_len;
  a.h = h_ckpt;
  a.ring_head = ring_head;
  a.status = dev_status;
  return finish(fn, launch_replay(a, (cudaStream_t)stream));
}

extern "C" int ssm_draft_tree_level(const ssm_dims* dims, const ssm_params* prm, int32_t n_seq, int32_t n_nodes,
                                    int32_t level, const ssm_node* layout, const uint16_t* xBC, const uint16_t* dt,
                                    const float* h_ckpt, const uint16_t* ring, const int32_t* ring_head,
                                    float* log_delta, float* log_B, float* log_x, float* y, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_draft_tree_level";
  if (int rc = check_dims(fn, dims, true, prm)) return rc;
  if (n_seq < 0) return fail(SSM_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
  if (n_nodes < 1) return fail(SSM_ERR_INVALID_ARG, fn, "n_nodes must be >= 1");
  if (n_nodes > SSM_MAX_NODES) return fail(SSM_ERR_CAPACITY, fn, "n_nodes exceeds SSM_MAX_NODES");
  if (level < 0 || level > SSM_MAX_DEPTH) return fail(SSM_ERR_RANGE, fn, "level must be in [0, SSM_MAX_DEPTH]");
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!layout || !xBC || !dt || !h_ckpt || !ring || !ring_head || !log_delta || !log_B || !log_x || !y)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (!workspace) return fail(SSM_ERR_INVALID_ARG, fn, "workspace is NULL");
  if (((uintptr_t)h_ckpt | (uintptr_t)log_B | (uintptr_t)prm->conv_w | (uintptr_t)workspace) & 15)
    return fail(SSM_ERR_INVALID_ARG, fn, "h_ckpt, log_B, params->conv_w and workspace must be 16-byte aligned");
  if (workspace_bytes < draft_tree_workspace_bytes(n_nodes, dims->n_heads, (long long)n_seq * dims->n_layers))
    return fail(SSM_ERR_CAPACITY, fn, "workspace smaller than ssm_draft_tree_workspace_size()");
  DraftTreeArgs a;
  a.H = dims->n_heads;
  a.L = dims->n_layers;
  a.R = dims->ring_cap;
  a.n_seq = n_seq;
  a.n = n_nodes;
  a.level = level;
  a.conv_w = prm->conv_w;
  a.conv_b = prm->conv_b;
  a.dt_bias = prm->dt_bias;
  a.A_log = prm->A_log;
  a.D = prm->D;
  a.layout = layout;
  a.xBC = xBC;
  a.dt = dt;
  a.h = h_ckpt;
  a.ring = ring;
  a.ring_head = ring_head;
  a.log_delta = log_delta;
  a.log_B = log_B;
  a.log_x = log_x;
  a.y = y;
  a.status = dev_status;
  return finish(fn, launch_draft_tree_level(a, workspace, (cudaStream_t)stream));
}

extern "C" size_t ssm_draft_tree_workspace_size(const ssm_dims* dims, int32_t n_seq, int32_t n_nodes) {
  const char* fn = "ssm_draft_tree_workspace_size";
  if (check_dims(fn, dims, false, nullptr)) return 0;
  if (n_seq < 0 || n_nodes < 1 || n_nodes > SSM_MAX_NODES) {
    fail(SSM_ERR_INVALID_ARG, fn, "need n_seq >= 0 and 1 <= n_nodes <= SSM_MAX_NODES");
    return 0;
  }
  const size_t b = draft_tree_workspace_bytes(n_nodes, dims->n_heads, (long long)n_seq * dims->n_layers);
  return b ? b : 16;
}

extern "C" int ssm_draft_tree_commit(const ssm_dims* dims, const ssm_params* prm, int32_t n_seq, int32_t n_nodes,
                                     const ssm_node* layout, int32_t max_path, const int32_t* path,
                                     const int32_t* path_len, const float* log_delta, const float* log_B,
                                     const float* log_x, const uint16_t* xBC, float* h_ckpt, uint16_t* ring,
                                     int32_t* ring_head, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_draft_tree_commit";
  if (int rc = check_dims(fn, dims, false, nullptr)) return rc;
  if (!prm || !prm->A_log) return fail(SSM_ERR_INVALID_ARG, fn, "params->A_log is NULL");
  if (n_seq < 0) return fail(SSM_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
  if (n_nodes < 1) return fail(SSM_ERR_INVALID_ARG, fn, "n_nodes must be >= 1");
  if (n_nodes > SSM_MAX_NODES) return fail(SSM_ERR_CAPACITY, fn, "n_nodes exceeds SSM_MAX_NODES");
  if (max_path < 1 || max_path > SSM_MAX_PATH) return fail(SSM_ERR_RANGE, fn, "max_path must be in [1, SSM_MAX_PATH]");
  if (n_seq == 0) return finish(fn, cudaSuccess);
  if (!layout || !path || !path_len || !log_delta || !log_B || !log_x || !xBC || !h_ckpt || !ring || !ring_head)
    return fail(SSM_ERR_INVALID_ARG, fn, "a tensor pointer is NULL");
  if (((uintptr_t)h_ckpt | (uintptr_t)log_B | (uintptr_t)xBC | (uintptr_t)ring) & 15)
    return fail(SSM_ERR_INVALID_ARG, fn, "h_ckpt, log_B, xBC and ring must be 16-byte aligned");
  DraftTreeCommitArgs a;
  a.H = dims->n_heads;
  a.L = dims->n_layers;
  a.R = dims->ring_cap;
  a.n_seq = n_seq;
  a.n = n_nodes;
  a.max_path = max_path;
  a.A_log = prm->A_log;
  a.layout = layout;
  a.path = path;
  a.path_len = path_len;
  a.log_delta = log_delta;
  a.log_B = log_B;
  a.log_x = log_x;
  a.xBC = xBC;
  a.h = h_ckpt;
  a.ring = ring;
  a.ring_head = ring_head;
  a.status = dev_status;
  return finish(fn, launch_draft_tree_commit(a, (cudaStream_t)stream));
}

extern "C" int ssm_selftest_bounded_wait(int32_t limit_us, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_selftest_bounded_wait";
  if (limit_us < 1 || limit_us > 1000000) return fail(SSM_ERR_RANGE, fn, "limit_us must be in [1, 1000000]");
  if (!dev_status) return fail(SSM_ERR_INVALID_ARG, fn, "dev_status is NULL");
  return finish(fn, launch_selftest_wait(dev_status, (unsigned long long)limit_us * 1000ull, (cudaStream_t)stream));
}

extern "C" int ssm_selftest_silu(const float* v, float* out, int64_t n, void* stream) {
  const char* fn = "ssm_selftest_silu";
  if (n < 0) return fail(SSM_ERR_RANGE, fn, "n must be >= 0");
  if (n > 0 && (!v || !out)) return fail(SSM_ERR_INVALID_ARG, fn, "v or out is NULL");
  return finish(fn, launch_selftest_silu(v, out, (long long)n, (cudaStream_t)stream));
}
