// Tree-layout module (host only): validates breadth-first parent[] arrays and
// derives the per-node records the kernels read.
//
// SpecMamba page ("FPGA加速Mamba推理：SpecMamba方案与优化实践") §3.2: the token
// tree is flattened breadth-first into a processing sequence; §5.2: the
// tree_config caps max_branches and max_depth.  In breadth-first order the
// parent index never decreases, so the children of a node form one contiguous,
// increasing index range, which is what child_begin / child_count record.
#include <stdio.h>

#include <string>
#include <vector>

#include "ssm_tree.h"

namespace ssmtree {
void set_error(const std::string& msg);
}

extern "C" int ssm_tree_layout_build(const int32_t* parent, int32_t n_seq, int32_t n_nodes, int32_t max_branches,
                                     int32_t max_depth, ssm_node* layout, int32_t* depth_out) {
  using ssmtree::set_error;
  char buf[256];
  if (n_seq < 0 || n_nodes < 1) {
    set_error("ssm_tree_layout_build: n_seq must be >= 0 and n_nodes >= 1");
    return SSM_ERR_INVALID_ARG;
  }
  if (n_seq > 0 && (parent == nullptr || layout == nullptr)) {
    set_error("ssm_tree_layout_build: null parent or layout");
    return SSM_ERR_INVALID_ARG;
  }
  int32_t deepest = 0;
  std::vector<int32_t> nchild(n_nodes);
  for (int32_t s = 0; s < n_seq; ++s) {
    const int32_t* par = parent + (size_t)s * n_nodes;
    ssm_node* out = layout + (size_t)s * n_nodes;
    if (par[0] != -1) {
      snprintf(buf, sizeof buf, "ssm_tree_layout_build: sequence %d: parent[0] = %d, must be -1", s, par[0]);
      set_error(buf);
      return SSM_ERR_BAD_TREE;
    }
    for (int32_t v = 1; v < n_nodes; ++v) {
      if (par[v] < 0 || par[v] >= v) {
        snprintf(buf, sizeof buf, "ssm_tree_layout_build: sequence %d: parent[%d] = %d is not an earlier node", s, v,
                 par[v]);
        set_error(buf);
        return SSM_ERR_BAD_TREE;
      }
      if (v >= 2 && par[v] < par[v - 1]) {
        snprintf(buf, sizeof buf, "ssm_tree_layout_build: sequence %d: parent[] is not breadth-first at node %d", s,
                 v);
        set_error(buf);
        return SSM_ERR_BAD_TREE;
      }
    }
    for (int32_t v = 0; v < n_nodes; ++v) {
      nchild[v] = 0;
      out[v].parent = par[v];
      out[v].depth = v == 0 ? 0 : out[par[v]].depth + 1;
      out[v].child_begin = n_nodes;
      out[v].child_count = 0;
      out[v].reserved = 0;
    }
    for (int32_t v = 1; v < n_nodes; ++v) {
      ssm_node& p = out[par[v]];
      if (p.child_count == 0) p.child_begin = v;
      p.child_count += 1;
    }
    for (int32_t v = 0; v < n_nodes; ++v) {
      if (max_branches > 0 && out[v].child_count > max_branches) {
        snprintf(buf, sizeof buf, "ssm_tree_layout_build: sequence %d: node %d has %d children > max_branches %d", s,
                 v, out[v].child_count, max_branches);
        set_error(buf);
        return SSM_ERR_CAPACITY;
      }
      if (max_depth > 0 && out[v].depth > max_depth) {
        snprintf(buf, sizeof buf, "ssm_tree_layout_build: sequence %d: node %d at depth %d > max_depth %d", s, v,
                 out[v].depth, max_depth);
        set_error(buf);
        return SSM_ERR_CAPACITY;
      }
      if (out[v].depth > deepest) deepest = out[v].depth;
      // conv taps: the node d positions back on v's path, or ring row head-(d-depth)
      int32_t anc = v;
      for (int d = 1; d <= 3; ++d) {
        if (anc >= 0) anc = out[anc].parent;
        out[v].tap[d - 1] = anc >= 0 ? anc : -(d - out[v].depth);
      }
    }
  }
  if (depth_out) *depth_out = deepest;
  return SSM_OK;
}
