"""Seeded synthetic inputs for SpecMamba-style tree verification on Mamba2 shapes.

This package only draws random numbers and lays them out.  It holds none of the
method's arithmetic (no conv, no softplus, no recurrence), so both the fp64
oracle and the CUDA path can consume the same buffers without sharing code.
"""
from .workloads import (  # noqa: F401
    Shape,
    Workload,
    WORKLOADS,
    workload,
    to_bf16_bits,
    bf16_bits_to_f32,
    layer_params,
    tree_parents,
    tree_tokens,
    instance_state,
    node_inputs,
    draft_inputs,
    replay_k,
    batch,
    batch_parallel,
    draft_batch,
)
