"""Test-side glue: widen generator outputs for the oracle and run it per instance."""
from __future__ import annotations

import numpy as np

import oracle
from synth import bf16_bits_to_f32


def f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def params_at(params: dict, j: int) -> dict:
    """Layer j's parameters, widened to fp64."""
    return {k: np.asarray(v[j], np.float64) for k, v in params.items()}


def oracle_verify_instance(b: dict, i: int, j: int, return_states=False):
    """Run the oracle on instance (sequence index i, layer index j) of a synth batch."""
    return oracle.verify(params_at(b["params"], j), b["parent"][i], f64(b["xBC"][i, j]), f64(b["dt"][i, j]),
                         b["h0"][i, j].astype(np.float64), f64(b["ring"][i, j]), int(b["ring_head"][i, j]),
                         return_states=return_states)


def rel_err(got, ref):
    """max |got - ref| / (1 + |ref|)  (the parity bound's left side)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


# ---------------------------------------------------------------------------
# device-side glue for the GPU tests (torch is only the allocator here)
# ---------------------------------------------------------------------------
def bf16_dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def params_dev(params):
    return {k: dev(np.ascontiguousarray(v, np.float32)) for k, v in params.items()}


def upload_tree_batch(b, w):
    """Synth batch -> device tensors + Dims + layout (built by the library's host call)."""
    from speculative_decoding_mamba2_gb300 import Dims, ssm_tree_layout_build
    S, L = len(b["seqs"]), len(b["layers"])
    n = b["n_nodes"]
    dims = Dims(n_heads=w.shape.H, n_layers=L, ring_cap=w.ring_cap)
    layout, depth = ssm_tree_layout_build(b["parent"])
    I = S * L
    d = dict(dims=dims, n_seq=S, n=n, depth=depth, layout=dev(layout), params=params_dev(b["params"]),
             xBC=bf16_dev(b["xBC"]).view(I, n, dims.conv_dim), dt=bf16_dev(b["dt"]).view(I, n, dims.n_heads),
             h0=dev(b["h0"]).view(I, dims.n_heads, dims.head_dim, dims.d_state),
             ring=bf16_dev(b["ring"]).view(I, w.ring_cap, dims.conv_dim), ring_head=dev(b["ring_head"]).view(I),
             tok=dev(b["tok"]), tgt=dev(b["tgt"]))
    return d


def run_tree_step(d, max_path=None, commit=True):
    """verify -> accept -> commit through the C ABI; returns host copies."""
    import torch
    from speculative_decoding_mamba2_gb300 import (ssm_accept_path, ssm_commit, ssm_tree_verify,
                                                   ssm_tree_verify_workspace_size)
    dims, S, n = d["dims"], d["n_seq"], d["n"]
    I = S * dims.n_layers
    max_path = d["depth"] + 1 if max_path is None else max_path
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full((I, n, dims.d_inner), float("nan"), device="cuda")
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, d["depth"]), dtype=torch.uint8, device="cuda")
    ssm_tree_verify(dims, d["params"], S, n, d["depth"], d["layout"], d["xBC"], d["dt"], d["h0"], d["ring"],
                    d["ring_head"], y, ws, status)
    path = torch.empty((S, max_path), dtype=torch.int32, device="cuda")
    plen = torch.empty(S, dtype=torch.int32, device="cuda")
    bonus = torch.empty(S, dtype=torch.int32, device="cuda")
    ssm_accept_path(S, n, max_path, d["layout"], d["tok"], d["tgt"], path, plen, bonus, status)
    out = dict(y=y, path=path, path_len=plen, bonus=bonus)
    if commit:
        h = d["h0"].clone()
        ring = d["ring"].clone()
        head = d["ring_head"].clone()
        ssm_commit(dims, d["params"], S, n, d["layout"], max_path, path, plen, d["xBC"], d["dt"], h, ring, head,
                   status)
        out.update(h=h, ring=ring, ring_head=head)
    torch.cuda.synchronize()
    out["status"] = status
    return out


def ring_window(ring_rows, head):
    """The three conv-state rows before `head`, oldest first."""
    R = ring_rows.shape[0]
    return np.stack([ring_rows[(head - 3 + i) % R] for i in range(3)])
