"""SpecMamba-style tree verification for Mamba2 on GB300 (sm_103a).

The compute path is libssmtree.so (hand-written CUDA, C ABI in
include/ssm_tree.h and include/ssm_layer.h); this package holds its sources
(csrc/), its build step (build.py) and a thin ctypes binding (binding.py) with
the same names.
"""
from .binding import (  # noqa: F401
    Dims,
    SSMError,
    lib,
    library_path,
    ssm_accept_path,
    ssm_commit,
    ssm_commit_verify,
    ssm_commit_verify_workspace_size,
    ssm_draft_step,
    ssm_draft_tree_commit,
    ssm_draft_tree_level,
    ssm_draft_tree_workspace_size,
    ssm_gated_rmsnorm,
    ssm_last_error,
    ssm_linear,
    ssm_linear_tile_cols,
    ssm_replay,
    ssm_rmsnorm,
    ssm_selftest_bounded_wait,
    ssm_selftest_silu,
    ssm_set_tuning,
    ssm_tree_layout_build,
    ssm_tree_verify,
    ssm_tree_verify_noalloc,
    ssm_tree_verify_workspace_size,
    ssm_version,
)
from .binding import (  # noqa: F401
    SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_BAD_TREE, SSM_ERR_CAPACITY, SSM_ERR_CUDA, SSM_ERR_RANGE,
    SSM_STATUS_BAD_LAYOUT, SSM_STATUS_PATH_RANGE, SSM_STATUS_K_RANGE, SSM_STATUS_WALK_TRUNCATED,
    SSM_STATUS_TIMEOUT, SSM_MAX_NODES, SSM_MAX_DEPTH, SSM_MAX_PATH, SSM_NOALLOC_WORKSPACE_BYTES, NODE_WORDS,
)
