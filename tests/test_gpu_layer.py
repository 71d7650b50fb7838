"""The block's dense steps on the GPU against the fp64 oracle, through the C ABI:
the tensor-core projection (tcgen05) with its column segments and residual add,
the two RMSNorms, and a whole Mamba2 block verifying a draft tree.

Bars: fp32 outputs of a projection within 1e-4·(1+|ref|) (bf16 products are exact in
fp32; only the accumulation order differs); bf16 outputs within one bf16 rounding of the
reference (2^-8 relative).  A whole block stores its activations as bf16 between the
steps.  Where the GPU's fp32 value and the oracle's fp64 value of an activation fall on
either side of a bf16 rounding point, the two round apart by one bf16 step (2^-8
relative); at the 2.7B-like K this happens to about one value in 2000.  A flipped x|B|C
value moves the conv output of up to four nodes by |w|·2^-8 ≈ 1e-3 and, through the
state, every descendant's y.  So the block bar is: every element within 1e-2·(1+|ref|)
and the median within 1e-4·(1+|ref|).  A wrong slice, a missing gate or residual is an
O(1) error in most elements."""
import numpy as np
import pytest
import torch

import oracle
from synth import Shape, Workload, batch
from tests.helpers import f64, params_at

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def bf16_host(rng, shape, scale=1.0):
    """Seeded bf16 values (as float64 on the host) and their bit patterns."""
    v = oracle.to_bf16(rng.standard_normal(shape) * scale)
    bits = v.astype(np.float32).view(np.uint32) >> 16
    return v, bits.astype(np.uint16)


def dev_bf16(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)


def host(t):
    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.double().cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (100, 200, 100), (128, 384, 2560), (300, 1000, 520),
                                   (256, 10576, 2560)])
def test_linear_fp32_against_oracle(M, N, K):
    from speculative_decoding_mamba2_gb300 import ssm_linear
    rng = np.random.default_rng([71, M, N, K])
    A, a_bits = bf16_host(rng, (M, K))
    W, w_bits = bf16_host(rng, (N, K), 0.05)
    Kp = (K + 7) // 8 * 8  # row strides are multiples of 8 elements; K itself need not be
    pad = lambda bits: np.pad(bits, ((0, 0), (0, Kp - K)))  # noqa: E731
    out = torch.full((M, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm_linear(dev_bf16(pad(a_bits))[:, :K], dev_bf16(pad(w_bits))[:, :K], [(0, out)], status=status)
    torch.cuda.synchronize()
    assert int(status) == 0
    ref = oracle.linear(A, W)
    assert (np.abs(host(out) - ref) <= 1e-4 * (1 + np.abs(ref))).all()


def test_linear_segments_and_strides():
    # the input projection's shape at H = 4: [z 256 | x B C 512 | dt 4], outputs in their own
    # buffers with row strides wider than the segment
    from speculative_decoding_mamba2_gb300 import ssm_linear
    rng = np.random.default_rng(72)
    M, K, H = 77, 192, 4
    N = 256 + 512 + H
    A, a_bits = bf16_host(rng, (M, K))
    W, w_bits = bf16_host(rng, (N, K), 0.1)
    z = torch.full((M, 264), float("nan"), device="cuda", dtype=torch.bfloat16)
    xbc = torch.full((M, 512), float("nan"), device="cuda", dtype=torch.float32)
    dt = torch.full((M, 8), float("nan"), device="cuda", dtype=torch.bfloat16)
    Ad = dev_bf16(a_bits)
    ssm_linear(Ad, dev_bf16(w_bits), [(0, z[:, :256]), (256, xbc), (768, dt[:, :H])])
    torch.cuda.synchronize()
    ref = oracle.linear(A, W)
    zb, rb = host(z[:, :256]), ref[:, :256]
    assert (np.abs(zb - rb) <= 2.0 ** -8 * np.abs(rb) + 1e-30).all()
    assert (np.abs(host(xbc) - ref[:, 256:768]) <= 1e-4 * (1 + np.abs(ref[:, 256:768]))).all()
    assert (np.abs(host(dt[:, :H]) - ref[:, 768:]) <= 2.0 ** -8 * np.abs(ref[:, 768:]) + 1e-30).all()
    assert torch.isnan(z[:, 256:].float()).all() and torch.isnan(dt[:, H:].float()).all()  # nothing past a segment


def test_linear_residual_in_place():
    from speculative_decoding_mamba2_gb300 import ssm_linear
    rng = np.random.default_rng(73)
    M, N, K = 130, 256, 320
    A, a_bits = bf16_host(rng, (M, K))
    W, w_bits = bf16_host(rng, (N, K), 0.1)
    x0 = rng.standard_normal((M, N)).astype(np.float32)
    x = torch.from_numpy(x0.copy()).cuda()
    ssm_linear(dev_bf16(a_bits), dev_bf16(w_bits), [(0, x)], residual=x)
    torch.cuda.synchronize()
    ref = x0.astype(np.float64) + oracle.linear(A, W)
    assert (np.abs(host(x) - ref) <= 1e-4 * (1 + np.abs(ref))).all()


@pytest.mark.parametrize("C", [256, 2560, 5120, 1000, 1002])  # 1002: no 16-byte rows, element loads
def test_rmsnorm_and_gated_rmsnorm(C):
    from speculative_decoding_mamba2_gb300 import ssm_gated_rmsnorm, ssm_rmsnorm
    rng = np.random.default_rng([74, C])
    M, eps = 37, 1e-5
    x = rng.standard_normal((M, C)).astype(np.float32) * 3
    w = (1 + 0.1 * rng.standard_normal(C)).astype(np.float32)
    z, z_bits = bf16_host(rng, (M, C), 2.0)
    out = torch.empty((M, C), device="cuda", dtype=torch.bfloat16)
    xd, wd = torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda()
    ssm_rmsnorm(xd, wd, eps, out)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(x, w, eps)
    assert (np.abs(host(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6).all()
    ssm_gated_rmsnorm(xd, dev_bf16(z_bits), wd, eps, out)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(x, z, w, eps)
    assert (np.abs(host(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6).all()


def block_setup(seed, H=4, d_model=256, n_seq=2):
    """A Mamba2 block at a small shape with seeded synthetic weights, and a draft tree batch
    (one layer) whose pre-conv rows the block's own input projection will produce."""
    w = Workload(seed, "block", Shape(H=H), n_layers=1, batch=n_seq, trees=(("random", 16, 3, 4),))
    b = batch(w)
    rng = np.random.default_rng([seed, 1])
    d_inner, conv_dim = H * 64, H * 64 + 256
    n_in = d_inner + conv_dim + H
    blk = {"norm_w": (1 + 0.1 * rng.standard_normal(d_model)),
           "W_in": oracle.to_bf16(rng.standard_normal((n_in, d_model)) / np.sqrt(d_model)),
           "gnorm_w": (1 + 0.1 * rng.standard_normal(d_inner)),
           "W_out": oracle.to_bf16(rng.standard_normal((d_model, d_inner)) / np.sqrt(d_inner))}
    blk["norm_w"] = blk["norm_w"].astype(np.float32).astype(np.float64)
    blk["gnorm_w"] = blk["gnorm_w"].astype(np.float32).astype(np.float64)
    x_in = rng.standard_normal((n_seq, b["n_nodes"], d_model)).astype(np.float32)
    return w, b, blk, x_in


def bits_of(v):
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_block_verify_against_oracle():
    """x → RMSNorm → input projection (z | x B C | dt) → tree verify → gated RMSNorm →
    output projection added to x, all through the C ABI, against oracle.block_verify."""
    from speculative_decoding_mamba2_gb300 import (Dims, ssm_gated_rmsnorm, ssm_linear, ssm_rmsnorm,
                                                   ssm_tree_layout_build, ssm_tree_verify,
                                                   ssm_tree_verify_workspace_size)
    H, d_model, S = 4, 256, 2
    w, b, blk, x_in = block_setup(81, H, d_model, S)
    n = b["n_nodes"]
    d_inner, conv_dim = H * 64, H * 64 + 256
    T, eps = S * n, 1e-5
    dims = Dims(n_heads=H, n_layers=1, ring_cap=w.ring_cap)
    x = torch.from_numpy(x_in.reshape(T, d_model).copy()).cuda()
    u = torch.empty((T, d_model), device="cuda", dtype=torch.bfloat16)
    z = torch.empty((T, d_inner), device="cuda", dtype=torch.bfloat16)
    xBC = torch.empty((T, conv_dim), device="cuda", dtype=torch.bfloat16)
    dt = torch.empty((T, H), device="cuda", dtype=torch.bfloat16)
    y = torch.empty((T, d_inner), device="cuda")
    g = torch.empty((T, d_inner), device="cuda", dtype=torch.bfloat16)
    W_in, W_out = dev_bf16(bits_of(blk["W_in"])), dev_bf16(bits_of(blk["W_out"]))
    nw = torch.from_numpy(blk["norm_w"].astype(np.float32)).cuda()
    gw = torch.from_numpy(blk["gnorm_w"].astype(np.float32)).cuda()
    prm = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda() for k, v in b["params"].items()}
    lay, depth = ssm_tree_layout_build(b["parent"])
    layout = torch.from_numpy(lay).cuda()
    h0 = torch.from_numpy(b["h0"]).cuda()
    ring = dev_bf16(b["ring"].reshape(S, -1))
    head = torch.from_numpy(b["ring_head"]).cuda()
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, depth), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm_rmsnorm(x, nw, eps, u)
    ssm_linear(u, W_in, [(0, z), (d_inner, xBC), (d_inner + conv_dim, dt)], status=status)
    ssm_tree_verify(dims, prm, S, n, depth, layout, xBC, dt, h0, ring, head, y, ws, status)
    ssm_gated_rmsnorm(y, z, gw, eps, g)
    ssm_linear(g, W_out, [(0, x)], residual=x, status=status)
    torch.cuda.synchronize()
    assert int(status) == 0
    x_out = host(x).reshape(S, n, d_model)
    y_gpu = host(y).reshape(S, n, d_inner)
    for i in range(S):
        ref_x, ref_y = oracle.block_verify(blk, params_at(b["params"], 0), b["parent"][i], x_in[i],
                                           b["h0"][i, 0].astype(np.float64), f64(b["ring"][i, 0]),
                                           int(b["ring_head"][i, 0]), H, eps=eps)
        for got, ref in ((y_gpu[i], ref_y), (x_out[i], ref_x)):
            e = np.abs(got - ref) / (1 + np.abs(ref))
            assert e.max() <= 1e-2, (i, e.max())
            assert np.median(e) <= 1e-4, (i, np.median(e))


def _check_bf16_step(got, ref, what):
    """A bf16 activation against the oracle's value of the same step (fed the GPU's own inputs)
    rounded to bf16: equal, except where the GPU's fp32 value and the fp64 value fall on either
    side of a rounding point -- then one bf16 step apart -- or where the value is so small that
    the fp32 accumulation's absolute error (about 1e-5 for a 2560- or 5120-term sum of O(1)
    size) decides its bf16 neighbour; at most 1 % of the values differ at all."""
    r = oracle.to_bf16(ref)
    d = np.abs(got - r)
    assert (d <= 2.0 ** -7 * np.abs(r) + 1e-4).all(), (what, float((d - 2.0 ** -7 * np.abs(r)).max()))
    assert np.mean(d > 0) <= 1e-2, (what, float(np.mean(d > 0)))


@pytest.mark.parametrize("layer", [0, 63])
def test_block_steps_2p7b_shape(layer):
    """A whole Mamba2 block at the 2.7B shape (d_model 2560, 80 heads, d_inner 5120), two
    sequences of 16-node trees, step by step: each step's oracle is fed the GPU's own bf16
    intermediates, so a rounding flip in one step cannot propagate into the next.  fp32 outputs
    (y, the residual stream) within 1e-3·(1+|ref|); bf16 outputs per _check_bf16_step."""
    from speculative_decoding_mamba2_gb300 import (Dims, ssm_gated_rmsnorm, ssm_linear, ssm_rmsnorm,
                                                   ssm_tree_layout_build, ssm_tree_verify,
                                                   ssm_tree_verify_workspace_size)
    H, d_model, S, eps = 80, 2560, 2, 1e-5
    w = Workload(3, "block steps 2.7B", Shape(H=H), n_layers=64, batch=S, trees=(("random", 16, 3, 4),))
    b = batch(w, layers=[layer])
    n = b["n_nodes"]
    d_inner, conv_dim = H * 64, H * 64 + 256
    T = S * n
    rng = np.random.default_rng([90, layer])
    n_in = d_inner + conv_dim + H
    W_in = oracle.to_bf16(rng.standard_normal((n_in, d_model)) / np.sqrt(d_model))
    W_out = oracle.to_bf16(rng.standard_normal((d_model, d_inner)) / np.sqrt(d_inner))
    nw = (1 + 0.1 * rng.standard_normal(d_model)).astype(np.float32)
    gw = (1 + 0.1 * rng.standard_normal(d_inner)).astype(np.float32)
    x_in = rng.standard_normal((T, d_model)).astype(np.float32)
    dims = Dims(n_heads=H, n_layers=1, ring_cap=w.ring_cap)
    x = torch.from_numpy(x_in.copy()).cuda()
    u = torch.empty((T, d_model), device="cuda", dtype=torch.bfloat16)
    z = torch.empty((T, d_inner), device="cuda", dtype=torch.bfloat16)
    xBC = torch.empty((T, conv_dim), device="cuda", dtype=torch.bfloat16)
    dt = torch.empty((T, H), device="cuda", dtype=torch.bfloat16)
    y = torch.empty((T, d_inner), device="cuda")
    g = torch.empty((T, d_inner), device="cuda", dtype=torch.bfloat16)
    prm = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda() for k, v in b["params"].items()}
    lay, depth = ssm_tree_layout_build(b["parent"])
    layout = torch.from_numpy(lay).cuda()
    h0 = torch.from_numpy(b["h0"]).cuda()
    ring = dev_bf16(b["ring"].reshape(S, -1))
    head = torch.from_numpy(b["ring_head"]).cuda()
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, depth), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm_rmsnorm(x, torch.from_numpy(nw).cuda(), eps, u)
    ssm_linear(u, dev_bf16(bits_of(W_in)), [(0, z), (d_inner, xBC), (d_inner + conv_dim, dt)], status=status)
    ssm_tree_verify(dims, prm, S, n, depth, layout, xBC, dt, h0, ring, head, y, ws, status)
    ssm_gated_rmsnorm(y, z, torch.from_numpy(gw).cuda(), eps, g)
    ssm_linear(g, dev_bf16(bits_of(W_out)), [(0, x)], residual=x, status=status)
    torch.cuda.synchronize()
    assert int(status) == 0
    u_g, z_g, xbc_g, dt_g, y_g, g_g, x_g = (host(t) for t in (u, z, xBC, dt, y, g, x))
    # 1. RMSNorm of the residual stream
    _check_bf16_step(u_g, oracle.rmsnorm(x_in, nw.astype(np.float64), eps), "rmsnorm")
    # 2. input projection of the GPU's u, cut into z | x B C | dt
    proj = oracle.linear(u_g, W_in)
    _check_bf16_step(z_g, proj[:, :d_inner], "z")
    _check_bf16_step(xbc_g, proj[:, d_inner:d_inner + conv_dim], "xBC")
    _check_bf16_step(dt_g, proj[:, d_inner + conv_dim:], "dt")
    # 3. tree verify of the GPU's x B C and dt, every element
    prm0 = params_at(b["params"], 0)
    for i in range(S):
        rows = slice(i * n, (i + 1) * n)
        ref_y = oracle.verify(prm0, b["parent"][i], xbc_g[rows], dt_g[rows], b["h0"][i, 0].astype(np.float64),
                              f64(b["ring"][i, 0]), int(b["ring_head"][i, 0]))
        assert (np.abs(y_g[rows] - ref_y) <= 1e-3 * (1 + np.abs(ref_y))).all(), ("y", i)
    # 4. gated RMSNorm of the GPU's y and z
    _check_bf16_step(g_g, oracle.gated_rmsnorm(y_g, z_g, gw.astype(np.float64), eps), "gated rmsnorm")
    # 5. output projection of the GPU's g added to the residual stream
    ref_x = x_in.astype(np.float64) + oracle.linear(g_g, W_out)
    assert (np.abs(x_g - ref_x) <= 1e-3 * (1 + np.abs(ref_x))).all(), "residual out"
