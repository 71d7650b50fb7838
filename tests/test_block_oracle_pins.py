"""Pins for the block oracle (oracle/block_oracle.py), on the CPU: each function checked
against something other than itself (a library routine, brute force, values worked out
by hand, constructions whose result is known), and plausible mistakes planted in it are
caught by at least one pin."""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.block_oracle as bo
from synth import Shape, Workload, batch


def test_to_bf16_matches_torch_rounding():
    rng = np.random.default_rng(91)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.0078125, 1.01171875, -3.5]])  # includes exact ties
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.to_bf16(v), ref)


def test_linear_matches_brute_force():
    rng = np.random.default_rng(92)
    A = rng.standard_normal((3, 5))
    W = rng.standard_normal((4, 5))
    D = np.zeros((3, 4))
    for t in range(3):
        for o in range(4):
            for k in range(5):
                D[t, o] += A[t, k] * W[o, k]
    np.testing.assert_allclose(oracle.linear(A, W), D, rtol=1e-14, atol=0)


def test_rmsnorm_hand_values():
    # x = [3, 4]: mean square 12.5, so x / sqrt(12.5) = [0.8485281374238570, 1.1313708498984760]
    np.testing.assert_allclose(oracle.rmsnorm([[3.0, 4.0]], [1.0, 1.0], 0.0),
                               [[0.8485281374238570, 1.1313708498984760]], rtol=1e-15)
    np.testing.assert_allclose(oracle.rmsnorm([[3.0, 4.0]], [2.0, -1.0], 0.0),
                               [[1.6970562748477140, -1.1313708498984760]], rtol=1e-15)
    # eps enters under the root: [1, 1] with eps 3 -> 1 / sqrt(4)
    np.testing.assert_allclose(oracle.rmsnorm([[1.0, 1.0]], [1.0, 1.0], 3.0), [[0.5, 0.5]], rtol=1e-15)
    # each row on its own: scale of one row does not touch the other
    np.testing.assert_allclose(oracle.rmsnorm([[3.0, 4.0], [30.0, 40.0]], [1.0, 1.0], 0.0),
                               [[0.8485281374238570, 1.1313708498984760]] * 2, rtol=1e-15)


def test_gated_rmsnorm_hand_values():
    # z = ln 3: SiLU = ln 3 · 3/4 = 0.8239592165010822; z = 0: SiLU = 0.  g = [0.82396, 0],
    # mean square g0²/2, so g / rms = [sqrt 2, 0]
    np.testing.assert_allclose(oracle.gated_rmsnorm([[1.0, 2.0]], [[math.log(3.0), 0.0]], [1.0, 1.0], 0.0),
                               [[1.4142135623730951, 0.0]], rtol=1e-15, atol=1e-300)
    # z = ±ln 3: SiLU = ln 3 · [3/4, -1/4], so g / rms = [0.75, -0.25] / sqrt(0.3125)
    np.testing.assert_allclose(oracle.gated_rmsnorm([[1.0, 1.0]], [[math.log(3.0), -math.log(3.0)]], [1.0, 1.0], 0.0),
                               [[1.3416407864998738, -0.4472135954999579]], rtol=1e-14)
    # z = 40: SiLU = 40 to 1e-17, g = [80, -40], rms = sqrt(4000)
    np.testing.assert_allclose(oracle.gated_rmsnorm([[2.0, -1.0]], [[40.0, 40.0]], [1.0, 1.0], 0.0),
                               [[1.2649110640673518, -0.6324555320336759]], rtol=1e-14)


def _block_case(seed, H=2):
    w = Workload(seed, "block pin", Shape(H=H), n_layers=1, batch=1, trees=(("random", 8, 3, 3),))
    b = batch(w)
    prm = {k: np.asarray(v[0], np.float64) for k, v in b["params"].items()}
    d_inner, conv_dim = H * 64, H * 64 + 256
    return b, prm, d_inner, conv_dim


def _run(blk, b, prm, x_in, H, eps):
    ring = ((b["ring"][0, 0].astype(np.uint32)) << 16).view(np.float32).astype(np.float64)
    return oracle.block_verify(blk, prm, b["parent"][0], x_in, b["h0"][0, 0].astype(np.float64), ring,
                               int(b["ring_head"][0, 0]), H, eps=eps)


def test_block_residual_gate_and_slices():
    H = 2
    b, prm, d_inner, conv_dim = _block_case(93, H)
    n = b["n_nodes"]
    d_model = conv_dim + H
    rng = np.random.default_rng(94)
    signs = np.where(rng.random((n, d_model)) < 0.5, -1.0, 1.0)  # rows of ±1: mean square 1
    blk = {"norm_w": np.full(d_model, 0.5),  # so the normed input is exactly ±0.5
           "W_in": np.zeros((2 * d_inner + 256 + H, d_model)),
           "gnorm_w": np.ones(d_inner),
           "W_out": rng.standard_normal((d_model, d_inner))}
    # x|B|C and dt copy the normed input's first conv_dim + H columns; z stays 0
    for c in range(conv_dim + H):
        blk["W_in"][d_inner + c, c] = 1.0
    eps = 2.0 ** -20  # > 0, so a closed gate normalises zeros to zeros; the ±0.5 still round to ±0.5
    x_out, y = _run(blk, b, prm, signs, H, eps)
    ring = ((b["ring"][0, 0].astype(np.uint32)) << 16).view(np.float32).astype(np.float64)
    y_ref = oracle.verify(prm, b["parent"][0], 0.5 * signs[:, :conv_dim], 0.5 * signs[:, conv_dim:],
                          b["h0"][0, 0].astype(np.float64), ring, int(b["ring_head"][0, 0]))
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)  # the x|B|C and dt slices
    np.testing.assert_array_equal(x_out, signs)  # z = 0 closes the gate: the block adds nothing
    # open the gate (z = the normed input's first d_inner columns) but zero the output projection
    for c in range(d_inner):
        blk["W_in"][c, c] = 1.0
    blk["W_out"][:] = 0.0
    x_out, _ = _run(blk, b, prm, signs, H, eps)
    np.testing.assert_array_equal(x_out, signs)  # the residual passes through unchanged
    # with the gate open and an output projection, the block changes the stream
    blk["W_out"] = rng.standard_normal((d_model, d_inner))
    x_out, _ = _run(blk, b, prm, signs, H, eps)
    assert np.abs(x_out - signs).max() > 1e-3


# ---- planted mistakes ----
def _silu_identity(v):
    return np.asarray(v, np.float64)


def _rmsnorm_sum(x, w, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * np.asarray(w, np.float64)


def _block_no_residual(blk, ssm_params, parent, x_in, h0, ring, head, H, P=64, N=128, eps=1e-5):
    x_out, y = _orig_block(blk, ssm_params, parent, x_in, h0, ring, head, H, P, N, eps)
    return x_out - np.asarray(x_in, np.float64), y


def _block_z_from_xbc(blk, ssm_params, parent, x_in, h0, ring, head, H, P=64, N=128, eps=1e-5):
    d_inner = H * P
    shifted = dict(blk)
    W = np.array(blk["W_in"])
    W[:d_inner] = W[d_inner:2 * d_inner]  # z taken from the x columns
    shifted["W_in"] = W
    return _orig_block(shifted, ssm_params, parent, x_in, h0, ring, head, H, P, N, eps)


_orig_block = bo.block_verify

MUTATIONS = {
    "gate without SiLU": ("silu", _silu_identity),
    "RMS over the sum, not the mean": ("rmsnorm", _rmsnorm_sum),
    "residual dropped": ("block_verify", _block_no_residual),
    "z read from the x columns": ("block_verify", _block_z_from_xbc),
}

PINS = [test_rmsnorm_hand_values, test_gated_rmsnorm_hand_values, test_block_residual_gate_and_slices]


def _any_pin_fails():
    for t in PINS:
        try:
            t()
        except AssertionError:
            return True
    return False


def test_unmutated_block_oracle_passes_every_pin():
    assert not _any_pin_fails()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_block_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(bo, attr, fn)
    if hasattr(oracle, attr) and attr != "silu":
        monkeypatch.setattr(oracle, attr, fn)
    with np.errstate(all="ignore"):
        assert _any_pin_fails(), f"no pin caught: {name}"
