/*
 * ssm_tree.h -- C ABI of libssmtree: SpecMamba-style tree verification for a
 * Mamba2 selective-SSM layer, on one GB300 (sm_103a).
 *
 * Method, by page and section:
 *   - "FPGA加速Mamba推理：SpecMamba方案与优化实践" §1.2: a draft model proposes
 *     tokens, the target model verifies them in parallel; §2.1: a rejection
 *     forces the SSM state back to the last accepted token; §3.1: the draft
 *     keeps only light intermediates (Δ, A, B, X) and recovers from them, the
 *     target recomputes only the affected path; §3.2: the token tree is
 *     flattened breadth-first and each node's children are updated from the
 *     node's state, which is released once they are done; §5.2: tree_config
 *     (max_branches, max_depth).
 *   - "FPGA 加速器完全拆解（二）…LightMamba", section "为什么 Mamba 难加速":
 *     X, B, C, Δ from the input projection; X through conv1d into the SSM with
 *     state h_t; the update terms Ā·h_{t-1} and B̄·X.
 * Read in the Mamba2 form (ngroups = 1):
 *     post = SiLU(conv_b + Σ_k conv_w[k]·row[k])      (width-4 causal conv, oldest tap first)
 *     x | B | C = post split as [d_inner | N | N]    (head h owns x[h·P, (h+1)·P))
 *     Δ = softplus(dt + dt_bias),  A = -exp(A_log),  Ā = exp(Δ·A)   (per head)
 *     h_v = Ā_v·h_parent(v) + Δ_v·(x_v ⊗ B_v),   h_parent(root) = h0
 *     y_v = C_v·h_v + D·x_v
 *
 * Conventions for every call:
 *   - Sizes: H heads, P head_dim, N d_state, W conv width (= 4),
 *     d_inner = H·P, conv_dim = d_inner + 2·N, L layers, S sequences,
 *     I = S·L instances, instance i = seq·L + layer (sequence-major), n nodes
 *     per tree.  Every array is dense, row-major, in the order its comment gives.
 *   - "device" pointers are CUDA device memory owned by the caller; the library
 *     never allocates, frees or keeps them.  "host" pointers are host memory.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device calls
 *     only enqueue work on it and return; results are ready when the stream is.
 *   - Return value: SSM_OK or a negative SSM_ERR_*; on error nothing was
 *     enqueued and ssm_last_error() (thread-local) says why.
 *   - `dev_status` (device, may be NULL): one int32 that kernels OR the
 *     SSM_STATUS_* bits into when device-resident data is inconsistent (a
 *     layout record out of range, a path or k out of range).  The offending item
 *     is clamped or skipped, never read or written out of bounds.  The caller
 *     zeroes it and reads it back when it wants to know.
 */
#ifndef SSM_TREE_H
#define SSM_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSM_OK 0
#define SSM_ERR_INVALID_ARG (-1) /* null pointer, bad size, unsupported shape   */
#define SSM_ERR_BAD_TREE (-2)    /* parent[] not a breadth-first tree          */
#define SSM_ERR_CAPACITY (-3)    /* tree or ring larger than the caps          */
#define SSM_ERR_CUDA (-4)        /* a CUDA runtime call failed                 */
#define SSM_ERR_RANGE (-5)       /* a scalar argument out of range             */

#define SSM_STATUS_BAD_LAYOUT 1  /* a layout record points outside its tree     */
#define SSM_STATUS_PATH_RANGE 2  /* path_len or a path entry out of range       */
#define SSM_STATUS_K_RANGE 4     /* replay k larger than the logged steps       */
#define SSM_STATUS_WALK_TRUNCATED 8 /* accept walk longer than max_path         */
#define SSM_STATUS_TIMEOUT 16    /* a bounded wait on a copy gave up (results   */
                                 /* of that call are invalid)                   */

/* Limits of this library (checked on the host; larger inputs get SSM_ERR_CAPACITY). */
#define SSM_MAX_NODES 64         /* nodes per branching tree (ssm_tree_verify)  */
#define SSM_MAX_DEPTH 15         /* deepest node below the root (branching)     */
#define SSM_MAX_CHAIN_NODES 4096 /* nodes of a chain (parent[v] = v-1)          */
#define SSM_MAX_PATH 256         /* accept / commit path length                 */

typedef struct ssm_dims {
  int32_t n_heads;    /* H                                                     */
  int32_t head_dim;   /* P (this library: 64)                                  */
  int32_t d_state;    /* N (this library: 128)                                 */
  int32_t conv_width; /* W (must be 4)                                         */
  int32_t n_layers;   /* L                                                     */
  int32_t ring_cap;   /* R: conv-ring rows per instance (>= 3)                 */
} ssm_dims;

/* Per-layer parameters, all device fp32. */
typedef struct ssm_params {
  const float *conv_w;  /* [L][conv_dim][W], tap 0 is the oldest row          */
  const float *conv_b;  /* [L][conv_dim]                                      */
  const float *dt_bias; /* [L][H]                                             */
  const float *A_log;   /* [L][H]  (A = -exp(A_log))                          */
  const float *D;       /* [L][H]                                             */
} ssm_params;

/* One node of a breadth-first token tree (32 bytes). */
typedef struct ssm_node {
  int32_t parent;      /* -1 for the root (node 0)                             */
  int32_t depth;       /* 0 for the root                                        */
  int32_t child_begin; /* children are the contiguous range                     */
  int32_t child_count; /*   [child_begin, child_begin + child_count)            */
  int32_t tap[3];      /* source of the pre-conv row d = 1, 2, 3 positions back */
                       /* on the node's path: node index >= 0, or -j meaning   */
                       /* conv-ring position ring_head - j (j = 1..3)           */
  int32_t reserved;    /* 0                                                     */
} ssm_node;

/* Library version (major*10000 + minor*100 + patch). */
int32_t ssm_version(void);

/* Thread-local text of the last error returned on this thread ("" if none). */
const char *ssm_last_error(void);

/*
 * ssm_tree_layout_build -- host-only (no CUDA call).  SpecMamba page §3.2
 * (breadth-first flattening), §5.2 (max_branches, max_depth).
 *   parent     host int32 [n_seq][n_nodes]: parent[0] = -1, 0 <= parent[v] < v,
 *              non-decreasing (breadth-first: siblings contiguous).
 *   max_branches, max_depth: caps (<= 0 means "no cap").
 *   layout     host ssm_node [n_seq][n_nodes], written.
 *   depth_out  host, may be NULL: deepest node over all trees.
 * Errors: SSM_ERR_BAD_TREE (first offending sequence/node in ssm_last_error),
 *         SSM_ERR_CAPACITY (a cap exceeded), SSM_ERR_INVALID_ARG.
 */
int ssm_tree_layout_build(const int32_t *parent, int32_t n_seq, int32_t n_nodes, int32_t max_branches,
                          int32_t max_depth, ssm_node *layout, int32_t *depth_out);

/*
 * ssm_tree_verify -- SpecMamba page §3.2 (tree verification) with the Mamba2
 * update above: for every node v of every instance, y_v = C_v·h_v + D·x_v where
 * h_v is the state after the node's root-to-node path applied to h0.  The
 * per-node states never reach memory; only h0, the inputs and y do.
 *   layout     device ssm_node [S][n] (from ssm_tree_layout_build), max_depth
 *              = its deepest node.  Branching trees: n <= SSM_MAX_NODES and
 *              max_depth <= SSM_MAX_DEPTH.  A tree with max_depth = n-1 is a
 *              chain; chains up to SSM_MAX_CHAIN_NODES are verified by walking
 *              them in 16-node chunks with the state on chip (the workspace
 *              then holds each chunk's B | C tables, 17 KB per instance and
 *              chunk).
 *   xBC        device bf16 [I][n][conv_dim]  pre-conv rows of the tree nodes
 *   dt         device bf16 [I][n][H]         raw dt
 *   h0         device fp32 [I][H][P][N]      committed state (read only)
 *   ring       device bf16 [I][R][conv_dim]  conv ring (read only)
 *   ring_head  device int32 [I]               committed positions; the rows
 *              before the root are ring positions head-3 .. head-1 (mod R)
 *   y          device fp32 [I][n][d_inner]    written
 *   workspace  device, 16-byte aligned, >= ssm_tree_verify_workspace_size()
 *              bytes, caller-owned scratch; its contents on entry do not
 *              matter and on return are unspecified.  Calls that overlap on
 *              the GPU must not share one workspace.
 */
int ssm_tree_verify(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t n_nodes,
                    int32_t max_depth, const ssm_node *layout, const uint16_t *xBC, const uint16_t *dt,
                    const float *h0, const uint16_t *ring, const int32_t *ring_head, float *y,
                    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * ssm_tree_verify_workspace_size -- host-only.  Bytes of device workspace
 * ssm_tree_verify needs for this shape (per-instance conv outputs, path
 * tables and path coefficients, written and read within one call); 0 if the
 * shape is rejected (reason in ssm_last_error()).
 */
size_t ssm_tree_verify_workspace_size(const ssm_dims *dims, int32_t n_seq, int32_t n_nodes, int32_t max_depth);

/*
 * ssm_accept_path -- SpecMamba page §1.2 (target verifies the draft): greedy
 * walk from the root; at node u move to the first child c (breadth-first
 * order) with tok[c] == tgt[u]; stop when none matches.
 *   layout   device ssm_node [S][n]
 *   tok      device int32 [S][n]   draft token of each node (tok[0] unused)
 *   tgt      device int32 [S][n]   target's greedy token after each node
 *   path     device int32 [S][max_path]  written: root..last, then -1 padding
 *   path_len device int32 [S]            written (>= 1)
 *   bonus    device int32 [S]            written: tgt[last]
 * A walk longer than max_path stops there and sets SSM_STATUS_WALK_TRUNCATED.
 */
int ssm_accept_path(int32_t n_seq, int32_t n_nodes, int32_t max_path, const ssm_node *layout,
                    const int32_t *tok, const int32_t *tgt, int32_t *path, int32_t *path_len, int32_t *bonus,
                    int32_t *dev_status, void *stream);

/*
 * ssm_commit -- SpecMamba page §3.1 (target: selective recomputation of the
 * affected path only) and §2.1 (roll back to the last accepted token).  The
 * accepted path is re-run from h0; h is overwritten with the state after its
 * last node, the last min(len, 3) pre-conv path rows go to ring positions
 * head+len-3.. head+len-1 (mod R) and ring_head advances by len.  Ring rows
 * outside the three before the new head are unspecified afterwards.
 *   path, path_len  device int32 [S][max_path], [S] (from ssm_accept_path)
 *   xBC, dt         as for ssm_tree_verify
 *   h               device fp32 [I][H][P][N]  in: h0, out: committed state
 *   ring, ring_head device, updated
 */
int ssm_commit(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t n_nodes, const ssm_node *layout,
               int32_t max_path, const int32_t *path, const int32_t *path_len, const uint16_t *xBC,
               const uint16_t *dt, float *h, uint16_t *ring, int32_t *ring_head, int32_t *dev_status,
               void *stream);

/*
 * ssm_commit_verify -- ssm_commit of the previous step's accepted path
 * followed by ssm_tree_verify of the next tree, in one pass over the state.
 * SpecMamba page §3.1 (selective recomputation of the accepted path) and §3.2
 * (FIFO tree verification): the commit is a rank-len update of h, so it is
 * applied to each state chunk as the verify streams it in; h is read once and
 * written once, where the separate calls read it twice and write it once.
 * Results equal ssm_commit(prev...) then ssm_tree_verify(next...) up to fp32
 * rounding order.  The pages describe the two steps, not this schedule.
 *   prev_n_nodes, prev_layout       the previous tree (n' nodes): ssm_node [S][n']
 *   prev_max_path                   row stride of prev_path, 1 <= .. <= SSM_MAX_DEPTH+1
 *   prev_path, prev_path_len        device int32 [S][prev_max_path], [S] (ssm_accept_path)
 *   prev_xBC, prev_dt               device bf16 [I][n'][conv_dim], [I][n'][H]: the previous
 *                                   tree's inputs (only the accepted path's rows are read)
 *   n_nodes .. dt                   the next tree, as for ssm_tree_verify (max_depth <= 15)
 *   h                               device fp32 [I][H][P][N]: in the state before the
 *                                   commit, out the committed state (the state the next
 *                                   tree was verified from)
 *   ring, ring_head                 device, updated as ssm_commit updates them;
 *                                   ring_cap >= prev_max_path + 3
 *   y                               device fp32 [I][n][d_inner], the next tree's outputs
 *   workspace                       ssm_commit_verify_workspace_size() bytes
 * A path entry that is not the root followed by children in order ends the
 * path there and sets SSM_STATUS_PATH_RANGE (as ssm_commit does).  Returns
 * SSM_ERR_CAPACITY for chain trees beyond SSM_MAX_DEPTH (they take the
 * separate calls) or a too-small workspace.
 */
size_t ssm_commit_verify_workspace_size(const ssm_dims *dims, int32_t n_seq, int32_t n_nodes, int32_t max_depth,
                                        int32_t prev_max_path);
int ssm_commit_verify(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t prev_n_nodes,
                      const ssm_node *prev_layout, int32_t prev_max_path, const int32_t *prev_path,
                      const int32_t *prev_path_len, const uint16_t *prev_xBC, const uint16_t *prev_dt,
                      int32_t n_nodes, int32_t max_depth, const ssm_node *layout, const uint16_t *xBC,
                      const uint16_t *dt, float *h, uint16_t *ring, int32_t *ring_head, float *y, void *workspace,
                      size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * ssm_commit_verify_prep / ssm_commit_verify_main -- the two halves of
 * ssm_commit_verify, same arguments.  Issued back to back on one stream they are
 * exactly ssm_commit_verify.  They exist so that the SSM can start as soon as Δ, B
 * and C exist: the LightMamba page ("计算重排序与细粒度分块融合") reorders the input
 * projection to produce Δ, B, C first and starts the SSM while X and Z are still
 * being produced.
 *   _prep reads, of this step's tree, only the B | C channels of xBC and dt (plus
 *         the previous path's rows, the ring, the layouts and the parameters); it
 *         writes the workspace and the committed ring rows' B | C channels; it reads
 *         ring_head and leaves it as it was.
 *   _main reads the x channels of xBC, h and what _prep wrote; it must run after
 *         _prep on the same workspace (same stream, or ordered by the caller) and
 *         after the x channels are in place.  It writes h, the ring's x channels,
 *         ring_head (advanced by the committed path's length) and y.
 * Both validate every argument as ssm_commit_verify does.
 */
int ssm_commit_verify_prep(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t prev_n_nodes,
                           const ssm_node *prev_layout, int32_t prev_max_path, const int32_t *prev_path,
                           const int32_t *prev_path_len, const uint16_t *prev_xBC, const uint16_t *prev_dt,
                           int32_t n_nodes, int32_t max_depth, const ssm_node *layout, const uint16_t *xBC,
                           const uint16_t *dt, float *h, uint16_t *ring, int32_t *ring_head, float *y,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);
int ssm_commit_verify_main(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t prev_n_nodes,
                           const ssm_node *prev_layout, int32_t prev_max_path, const int32_t *prev_path,
                           const int32_t *prev_path_len, const uint16_t *prev_xBC, const uint16_t *prev_dt,
                           int32_t n_nodes, int32_t max_depth, const ssm_node *layout, const uint16_t *xBC,
                           const uint16_t *dt, float *h, uint16_t *ring, int32_t *ring_head, float *y,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * ssm_draft_step -- one draft token per instance (a one-node tree), SpecMamba
 * page §3.1 (the draft logs only Δ, A, B, X).  Position = ring_head + step:
 * the token's pre-conv row is written to that ring position, the conv window
 * is the three ring rows before it, and
 *     h_out = Ā·h_in + Δ·(x ⊗ B),   y = C·h_out + D·x,
 * then log row `step` = {Δ [H], B [N], x [d_inner]} (fp32, post-conv) and
 * log_len = step + 1.  A is constant per head, so Δ stands for A in the log.
 *   step       0 <= step < log_cap and step + 3 < R
 *   xBC_t      device bf16 [I][conv_dim]   dt_t device bf16 [I][H]
 *   h_in/h_out device fp32 [I][H][P][N] (may be the same buffer)
 *   ring       device bf16 [I][R][conv_dim] (row written), ring_head device [I] (read)
 *   log_delta  device fp32 [I][log_cap][H]; log_B [I][log_cap][N];
 *   log_x      [I][log_cap][d_inner]; log_len device int32 [I]
 *   y          device fp32 [I][d_inner]
 */
int ssm_draft_step(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t step, int32_t log_cap,
                   const uint16_t *xBC_t, const uint16_t *dt_t, const float *h_in, float *h_out, uint16_t *ring,
                   const int32_t *ring_head, float *log_delta, float *log_B, float *log_x, int32_t *log_len,
                   float *y, int32_t *dev_status, void *stream);

/*
 * ssm_replay -- SpecMamba page §3.1 (draft state recovery from the light log):
 * h_ckpt <- the k[seq] logged updates applied in order (no conv, no input
 * re-read; the same fp32 operations as ssm_draft_step, so the result equals
 * the state that step k left, bit for bit); ring_head += k; log_len = 0.
 *   k          device int32 [S], 0 <= k <= log_len (else clamped + status bit)
 *   log_*      as written by ssm_draft_step (log_B 16-byte aligned)
 *   h_ckpt     device fp32 [I][H][P][N], in/out, 16-byte aligned
 */
int ssm_replay(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t log_cap, const int32_t *k,
               const float *log_delta, const float *log_B, const float *log_x, int32_t *log_len, float *h_ckpt,
               int32_t *ring_head, int32_t *dev_status, void *stream);

/*
 * ssm_draft_tree_level -- draft-side tree drafting, one depth level per call.
 * SpecMamba page §3.1 (the draft keeps only the light intermediates Δ, A, B, X
 * and recovers states from them) and §3.2 (a node's children continue from the
 * node's state).  A draft tree grows one depth at a time: the tokens of depth
 * level+1 come from the outputs of depth `level`.  For every node v of depth
 * `level` (in every instance): its pre-conv row goes through the tree conv
 * (taps over its ancestors, then the conv ring) and SiLU, Δ = softplus(dt +
 * dt_bias), and
 *     y_v = C_v·h_v + D·x_v,  h_v = h_ckpt followed by the logged updates of
 *     v's ancestors (root first) and then v's own update.
 * h_v is never formed: the call reads h_ckpt once and the ancestors' log rows,
 * and writes v's log row {Δ [H], B [N], x [d_inner]} (fp32, post-conv) and y_v.
 * No state is written, so every branch shares the one committed state.
 *   n_nodes    1..SSM_MAX_NODES;  level 0..SSM_MAX_DEPTH (a level with no
 *              node is a no-op)
 *   layout     device ssm_node [S][n] (ssm_tree_layout_build of the draft tree)
 *   xBC, dt    device bf16 [I][n][conv_dim], [I][n][H]: rows of the nodes of
 *              depth <= level must be written (read only)
 *   h_ckpt     device fp32 [I][H][P][N], 16-byte aligned (read only)
 *   ring, ring_head  as for ssm_tree_verify (read only)
 *   log_delta  device fp32 [I][n][H]; log_B [I][n][N] (16-byte aligned);
 *   log_x      [I][n][d_inner]: rows of depth < level are read (the earlier
 *              levels' calls wrote them), rows of depth == level are written
 *   y          device fp32 [I][n][d_inner]: rows of depth == level written
 *   workspace  device, 16-byte aligned, >= ssm_draft_tree_workspace_size()
 *              bytes, caller-owned scratch (per level node: C, e^{S_v} per
 *              head, the path sums of every row and the B·C products along
 *              its path, written and read within the call); calls that
 *              overlap on the GPU must not share one
 * A layout record that points outside its tree sets SSM_STATUS_BAD_LAYOUT and
 * the instance writes nothing.
 */
int ssm_draft_tree_level(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t n_nodes,
                         int32_t level, const ssm_node *layout, const uint16_t *xBC, const uint16_t *dt,
                         const float *h_ckpt, const uint16_t *ring, const int32_t *ring_head, float *log_delta,
                         float *log_B, float *log_x, float *y, void *workspace, size_t workspace_bytes,
                         int32_t *dev_status, void *stream);

/*
 * ssm_draft_tree_workspace_size -- host-only.  Bytes of device workspace
 * ssm_draft_tree_level needs: about n_nodes * (N + H + d_inner + 16) * 4 per
 * instance (each part padded to 128 bytes); 0 if the shape is rejected
 * (reason in ssm_last_error()).
 */
size_t ssm_draft_tree_workspace_size(const ssm_dims *dims, int32_t n_seq, int32_t n_nodes);

/*
 * ssm_draft_tree_commit -- after the target accepts a path of the draft tree
 * (ssm_accept_path), move the draft's committed state along it from the log:
 * h_ckpt <- the logged updates of path[0 .. path_len) applied in order (no conv,
 * no input re-read; the same fp32 operations as ssm_draft_step, so on a chain
 * the result equals the stepped state bit for bit), the path's pre-conv rows
 * appended to the conv ring (the last three are written) and ring_head +=
 * path_len.  Every node on the path must have been drafted (its log row written).
 *   path       device int32 [S][max_path]: path[0] = 0, each entry a child of
 *              the one before; path_len device int32 [S], 0..max_path.  A bad
 *              entry sets SSM_STATUS_PATH_RANGE and only the valid prefix commits.
 *   log_*      as written by ssm_draft_tree_level (log_B 16-byte aligned)
 *   xBC        device bf16 [I][n][conv_dim] (16-byte aligned)
 *   h_ckpt     device fp32 [I][H][P][N], in/out, 16-byte aligned
 *   ring       device bf16 [I][R][conv_dim] (16-byte aligned), ring_head [I]
 */
int ssm_draft_tree_commit(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t n_nodes,
                          const ssm_node *layout, int32_t max_path, const int32_t *path, const int32_t *path_len,
                          const float *log_delta, const float *log_B, const float *log_x, const uint16_t *xBC,
                          float *h_ckpt, uint16_t *ring, int32_t *ring_head, int32_t *dev_status, void *stream);

/*
 * ssm_selftest_bounded_wait -- failure detection self-test (no counterpart in the
 * pages).  Every copy pipeline of this library waits on mbarriers with a bounded
 * wait: after one second of global time it gives up, sets SSM_STATUS_TIMEOUT in
 * the caller's status word and the kernel returns, so a lost copy never hangs
 * the GPU.  This call runs that wait on a barrier nothing arrives at, with a
 * limit of limit_us microseconds, so the give-up path can be checked: on return
 * (after a synchronize) *dev_status has SSM_STATUS_TIMEOUT set and the context
 * is usable.
 *   limit_us   1..1000000
 *   dev_status device int32 (required)
 */
int ssm_selftest_bounded_wait(int32_t limit_us, int32_t *dev_status, void *stream);

/*
 * ssm_selftest_silu -- the SiLU forms the kernels evaluate, on n given inputs (no
 * counterpart in the pages; SiLU is the activation after the conv, LightMamba page
 * "为什么 Mamba 难加速").  For each v[i]:
 *   out[i]        the FMA-pipe form of the tree kernel's x conv: v / (1 + 2^t),
 *                 t = -v·log2(e), 2^t by Cody-Waite reduction and a degree-6
 *                 Taylor series, the reciprocal by three Newton-Raphson steps;
 *   out[n + i]    the special-function form (fast exp and divide intrinsics) of
 *                 the prep kernels' B | C conv;
 *   out[2n + i]   v / (1 + expf(-v)) with a rounded divide (commit, draft step).
 *   v    device fp32 [n]     out device fp32 [3][n]
 */
int ssm_selftest_silu(const float *v, float *out, int64_t n, void *stream);

/*
 * ssm_set_tuning -- process-wide launch-plan overrides (no counterpart in the
 * pages; they change how work is spread over the GPU, never the results beyond
 * fp32 rounding order).  Each knob starts at the value of the environment
 * variable of the same name, read once when the library is first used, or 0
 * (automatic plan) when unset; this call replaces it for later calls.
 *   name   "SSM_VERIFY_GROUPS_PER_CTA"   head groups per CTA of the tree kernel (1..8)
 *          "SSM_VERIFY_HEADS_PER_GROUP"  heads per group of the tree kernel (2 or 4)
 *          "SSM_LINEAR_TCHUNK"           tokens per CTA of ssm_linear (64, 128 or 256)
 *          "SSM_LINEAR_SPLITS"           K-splits of ssm_linear (fp32 accumulator outputs)
 *          "SSM_LINEAR_STAGES"           copy-ring stages of ssm_linear
 *          "SSM_VERIFY_KERNEL"           tree kernels of ssm_tree_verify / ssm_commit_verify:
 *                                        0 or 1 = warp-level mma.sync (the default),
 *                                        2 = the state contraction on tcgen05 with tensor-
 *                                        memory accumulators (measured slower here)
 *          "SSM_VERIFY_CTAS"             at most this many CTAs of the persistent tcgen05 tree
 *                                        kernel (each walks a run of head pairs)
 *          "SSM_VERIFY_DEEP"             one CTA per SM with a deep pipeline of state chunks:
 *                                        0 = when the head groups are few per SM, 1 = never,
 *                                        2 = wherever its shared memory fits
 *   value  0 = automatic; a value the plan cannot use is ignored at launch.
 * Not thread-safe against calls that launch concurrently on other threads.
 * Errors: SSM_ERR_INVALID_ARG for an unknown name or a negative value.
 */
int ssm_set_tuning(const char *name, int32_t value);

/*
 * ssm_tree_verify_noalloc -- ssm_tree_verify for callers that cannot allocate
 * device memory (a runtime that gives a plugin only the current op's tensors
 * and owns all other device memory, an embedding with allocation forbidden
 * after start-up, a C-ABI-only host with no allocator of its own).  The pages
 * have no counterpart: this is a deployment convenience of this library.
 * Same arguments and results as ssm_tree_verify, without the workspace: the
 * scratch is one array of SSM_NOALLOC_WORKSPACE_BYTES bytes compiled into the
 * library, held by every GPU that loads it until the process exits.  A batch
 * whose ssm_tree_verify_workspace_size() exceeds that gets SSM_ERR_CAPACITY.
 * Nothing here calls cudaMalloc/cudaFree or any allocating routine.  The first
 * call on a device looks up the array's address (cudaGetSymbolAddress) with
 * that device current and keeps it for the process; make it before any stream
 * capture.  A cudaDeviceReset of that device invalidates the kept address, so
 * do not call this entry point after one.  All calls share the array, so calls
 * whose GPU work overlaps race; serialise them.
 */
#define SSM_NOALLOC_WORKSPACE_BYTES (16u << 20)
int ssm_tree_verify_noalloc(const ssm_dims *dims, const ssm_params *prm, int32_t n_seq, int32_t n_nodes,
                            int32_t max_depth, const ssm_node *layout, const uint16_t *xBC, const uint16_t *dt,
                            const float *h0, const uint16_t *ring, const int32_t *ring_head, float *y,
                            int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_TREE_H */
