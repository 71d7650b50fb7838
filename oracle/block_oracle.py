"""fp64 CPU oracle for the dense steps around the SSM in a Mamba2 block.

TEST INFRASTRUCTURE ONLY, like ``ssm_oracle`` (same rules: imported by tests/,
smoke() and the CPU legs of bench.py only; shares no code with the CUDA path).

Sources (page title, then section):

* "FPGA 加速器完全拆解（二）…FlightLLM、CXL-SpecKV 与 LightMamba", section
  "为什么 Mamba 难加速": the input projection makes X, B, C, Δ and Z from each
  token; X goes through the conv and the SSM; the SSM output Y is multiplied
  elementwise by Z and the output projection restores the model width.
* Same page, section "旋转辅助量化": the block has an RMSNorm before the input
  projection and a second RMSNorm after the SSM.

Readings where the pages are silent (also listed in the design notes): the
second norm is Mamba2's gated form RMSNorm(y · SiLU(z)) with a learned weight;
the input projection's output columns are ordered [z | x B C | dt]; the output
projection's result is added to the residual stream; activations passed between
the steps are stored as bf16 (round to nearest even) exactly where the GPU path
stores them, everything else is fp64.
"""
from __future__ import annotations

import numpy as np

from .ssm_oracle import silu, verify


def to_bf16(a):
    """Round float64/float32 values to the nearest bf16 (ties to even), returned as float64."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return ((r << 16).astype(np.uint32)).view(np.float32).astype(np.float64)


def linear(A, W):
    """D[t, o] = Σ_k A[t, k] · W[o, k]  (a projection; W is [out features][in features])."""
    return np.asarray(A, np.float64) @ np.asarray(W, np.float64).T


def rmsnorm(x, w, eps):
    """w · x / sqrt(mean(x²) + eps) over the last axis."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(w, np.float64)


def gated_rmsnorm(y, z, w, eps):
    """RMSNorm of g = y · SiLU(z) with weight w."""
    return rmsnorm(np.asarray(y, np.float64) * silu(np.asarray(z, np.float64)), w, eps)


def block_verify(blk, ssm_params, parent, x_in, h0, ring, head, H, P=64, N=128, eps=1e-5):
    """One Mamba2 block over a draft tree of one sequence.

    x_in [n][d_model] is the residual stream at the tree's tokens.  Returns
    (x_out, y): the residual stream after the block and the SSM output.
    blk: norm_w [d_model], W_in [2·d_inner + 2N + H][d_model], gnorm_w [d_inner],
    W_out [d_model][d_inner]."""
    d_inner = H * P
    conv_dim = d_inner + 2 * N
    u = to_bf16(rmsnorm(x_in, blk["norm_w"], eps))
    proj = linear(u, blk["W_in"])
    z = to_bf16(proj[:, :d_inner])
    xBC = to_bf16(proj[:, d_inner:d_inner + conv_dim])
    dt = to_bf16(proj[:, d_inner + conv_dim:d_inner + conv_dim + H])
    y = verify(ssm_params, parent, xBC, dt, h0, ring, head)
    g = to_bf16(gated_rmsnorm(y, z, blk["gnorm_w"], eps))
    return np.asarray(x_in, np.float64) + linear(g, blk["W_out"]), y
