"""fp64 CPU oracle -- test infrastructure only (see ssm_oracle's header)."""
from .ssm_oracle import (  # noqa: F401
    BadTree,
    softplus,
    silu,
    tree_layout,
    node_window,
    conv_silu,
    split_xbc,
    ssm_step,
    ssm_out,
    verify,
    accept,
    commit,
    draft_step,
    replay,
    draft_tree_level,
    draft_tree_commit,
)
from .block_oracle import (  # noqa: F401
    to_bf16,
    linear,
    rmsnorm,
    gated_rmsnorm,
    block_verify,
)
