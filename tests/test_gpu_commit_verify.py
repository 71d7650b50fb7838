"""ssm_commit_verify (commit of the previous tree's accepted path folded into the
next tree's verify) against the fp64 oracle, oracle.commit then oracle.verify,
and against the separate GPU calls ssm_commit then ssm_tree_verify.

Bar: accepted path, ring rows and heads bit-exact; y and the committed state
max |gpu - ref| <= 1e-3 * (1 + |ref|) against the oracle; the fused and the
separate GPU calls agree to 5e-5 * (1 + |ref|).  They round differently: the fused
call contracts C with the state as read and adds the commit's rank-len update to y
through the products C_v·B_j (y = e^S·(E·C·h + Σ_j u_j·C·B_j)), and forms the
committed state's update U·Bᵀ from bf16 hi/lo splits (~2^-16 of the update); the
separate calls contract C with the committed state."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from synth import Shape, Workload, batch, workload
from tests.helpers import bf16_dev, dev, f64, params_at, rel_err, ring_window, upload_tree_batch

pytestmark = pytest.mark.gpu
TOL = 1e-3
TOL_GPU = 5e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def next_workload(w, index, tree):
    """Same shape and sizes as w, another seed stream and tree: the next speculative step."""
    return dataclasses.replace(w, index=index, name=w.name + " (next step)", trees=(tree,))


def run_both(b0, w0, b1, path=None, plen=None):
    """Accept on the previous tree (unless a path is given), then the fused call and the
    separate calls from the same state; returns host-side results of both."""
    from speculative_decoding_mamba2_gb300 import (ssm_accept_path, ssm_commit, ssm_commit_verify,
                                                   ssm_commit_verify_workspace_size, ssm_tree_layout_build,
                                                   ssm_tree_verify, ssm_tree_verify_workspace_size)
    d0 = upload_tree_batch(b0, w0)
    dims, S, n0 = d0["dims"], d0["n_seq"], d0["n"]
    I = S * dims.n_layers
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if path is None:
        mp = d0["depth"] + 1
        path = torch.empty((S, mp), dtype=torch.int32, device="cuda")
        plen = torch.empty(S, dtype=torch.int32, device="cuda")
        bonus = torch.empty(S, dtype=torch.int32, device="cuda")
        ssm_accept_path(S, n0, mp, d0["layout"], d0["tok"], d0["tgt"], path, plen, bonus, status)
    else:
        mp = path.shape[1]
    n1 = b1["n_nodes"]
    lay1_h, depth1 = ssm_tree_layout_build(b1["parent"])
    lay1 = dev(lay1_h)
    xBC1 = bf16_dev(b1["xBC"]).view(I, n1, dims.conv_dim)
    dt1 = bf16_dev(b1["dt"]).view(I, n1, dims.n_heads)

    h = d0["h0"].clone()
    ring = d0["ring"].clone()
    head = d0["ring_head"].clone()
    y = torch.full((I, n1, dims.d_inner), float("nan"), device="cuda")
    ws = torch.empty(ssm_commit_verify_workspace_size(dims, S, n1, depth1, mp), dtype=torch.uint8, device="cuda")
    fstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm_commit_verify(dims, d0["params"], S, n0, d0["layout"], mp, path, plen, d0["xBC"], d0["dt"], n1, depth1,
                      lay1, xBC1, dt1, h, ring, head, y, ws, fstatus)

    h2 = d0["h0"].clone()
    ring2 = d0["ring"].clone()
    head2 = d0["ring_head"].clone()
    y2 = torch.full_like(y, float("nan"))
    ws2 = torch.empty(ssm_tree_verify_workspace_size(dims, S, n1, depth1), dtype=torch.uint8, device="cuda")
    sstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm_commit(dims, d0["params"], S, n0, d0["layout"], mp, path, plen, d0["xBC"], d0["dt"], h2, ring2, head2,
               sstatus)
    ssm_tree_verify(dims, d0["params"], S, n1, depth1, lay1, xBC1, dt1, h2, ring2, head2, y2, ws2, sstatus)
    torch.cuda.synchronize()
    cpu = lambda t: t.cpu()  # noqa: E731
    return dict(y=cpu(y), h=cpu(h), ring=cpu(ring), head=cpu(head), status=int(fstatus.item()),
                y_sep=cpu(y2), h_sep=cpu(h2), ring_sep=cpu(ring2), head_sep=cpu(head2),
                sep_status=int(sstatus.item()) | int(status.item()),
                path=cpu(path), plen=cpu(plen))


def check_oracle(b0, b1, out, pairs, paths=None):
    """Sampled instances (seq index i, layer index j): oracle.commit then oracle.verify."""
    L = len(b0["layers"])
    for i, j in pairs:
        inst = i * L + j
        prm = params_at(b0["params"], j)
        if paths is None:
            path_ref, _ = oracle.accept(b0["parent"][i], b0["tok"][i], b0["tgt"][i])
            assert out["path"][i, :int(out["plen"][i])].tolist() == path_ref
        else:
            path_ref = paths[i]
        head0 = int(b0["ring_head"][i, j])
        h_c, ring_c, head_c = oracle.commit(prm, b0["parent"][i], path_ref, f64(b0["xBC"][i, j]),
                                            f64(b0["dt"][i, j]), b0["h0"][i, j].astype(np.float64),
                                            f64(b0["ring"][i, j]), head0)
        y_ref = oracle.verify(prm, b1["parent"][i], f64(b1["xBC"][i, j]), f64(b1["dt"][i, j]), h_c, ring_c, head_c)
        e = rel_err(out["y"][inst].double().numpy(), y_ref)
        assert e <= TOL, f"y of instance ({i},{j}): {e}"
        e = rel_err(out["h"][inst].double().numpy(), h_c)
        assert e <= TOL, f"committed h of instance ({i},{j}): {e}"
        assert int(out["head"][inst]) == head_c
        ring_gpu = out["ring"][inst].view(torch.int16).numpy().view(np.uint16)
        ring_exp = b0["ring"][i, j].copy()
        R = ring_exp.shape[0]
        for jj, m in enumerate(path_ref):
            ring_exp[(head0 + jj) % R] = b0["xBC"][i, j, m]
        np.testing.assert_array_equal(ring_window(ring_gpu, head_c), ring_window(ring_exp, head_c))


def check_separate(out):
    """Fused against the separate GPU calls, every element."""
    assert torch.isfinite(out["y"]).all()
    assert rel_err(out["y"].double().numpy(), out["y_sep"].double().numpy()) <= TOL_GPU
    assert rel_err(out["h"].double().numpy(), out["h_sep"].double().numpy()) <= TOL_GPU
    assert torch.equal(out["head"], out["head_sep"])
    for inst in range(out["head"].shape[0]):
        hd = int(out["head"][inst])
        np.testing.assert_array_equal(ring_window(out["ring"][inst].view(torch.int16).numpy(), hd),
                                      ring_window(out["ring_sep"][inst].view(torch.int16).numpy(), hd))


def test_tiny_130m_tree15_every_element():
    w0 = workload(0)
    w1 = next_workload(w0, 60, ("random", 16, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(0, 0)])
    check_separate(out)


def test_ragged_heads_and_trees_of_different_sizes():
    # H = 6: the last head group of 4 is ragged (its rows past the 6 heads are another
    # instance's state and must not be written); 40-node previous tree, 16-node next tree
    w0 = Workload(61, "ragged", Shape(H=6), n_layers=2, batch=3, trees=(("full", 3, 3),), p_accept=0.9)
    w1 = next_workload(w0, 62, ("random", 16, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(3) for j in range(2)])
    check_separate(out)


@pytest.mark.parametrize("gpc", ["2", "3"])
def test_several_head_groups_per_cta(gpc, tuning):
    # per-group committed-path rows arrive while the previous group is still being consumed
    tuning("SSM_VERIFY_GROUPS_PER_CTA", gpc)
    w0 = Workload(63, "groups", Shape(H=24), n_layers=2, batch=2, trees=(("random", 16, 3, 4),), p_accept=0.9)
    w1 = next_workload(w0, 64, ("full", 2, 3))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(2)])
    check_separate(out)


@pytest.mark.parametrize("deep", [1, 2])
def test_root_only_and_longest_paths(deep, tuning):
    tuning("SSM_VERIFY_DEEP", deep)  # 1: two CTAs per SM, 3 chunks in flight; 2: one, 8
    # a 16-node chain accepted to its end (path of 16 = the longest the fused call takes),
    # and a root-only path, in one batch
    w0 = Workload(65, "chain16", Shape(H=8), n_layers=2, batch=2, trees=(("chain", 16),), p_accept=1.0)
    w1 = next_workload(w0, 66, ("random", 16, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    full = list(range(16))
    path = torch.full((2, 16), -1, dtype=torch.int32)
    path[0] = torch.tensor(full, dtype=torch.int32)
    path[1, 0] = 0
    plen = torch.tensor([16, 1], dtype=torch.int32)
    out = run_both(b0, w0, b1, path=path.cuda(), plen=plen.cuda())
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(2)], paths=[full, [0]])
    check_separate(out)


@pytest.mark.parametrize("deep", [1, 2])
def test_bad_path_is_cut_and_flagged_like_commit(deep, tuning):
    tuning("SSM_VERIFY_DEEP", deep)  # 1: two CTAs per SM, 3 chunks in flight; 2: one, 8
    from speculative_decoding_mamba2_gb300 import SSM_STATUS_PATH_RANGE
    # the prep fetches the path's rows as given, clamped into the tree, before the path is
    # checked: a cut path uses only the rows before the cut, a bad root fetches node 0 again
    w0 = Workload(67, "badpath", Shape(H=8), n_layers=2, batch=5, trees=(("full", 2, 3),), p_accept=1.0)
    w1 = next_workload(w0, 68, ("random", 16, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    lay = oracle.tree_layout(b0["parent"][0])
    good = lay["path"][b0["n_nodes"] - 1]  # root .. deepest node
    path = torch.full((5, 4), -1, dtype=torch.int32)
    path[0] = torch.tensor(good, dtype=torch.int32)
    path[1] = torch.tensor([good[0], good[1], 999, good[3]], dtype=torch.int32)  # out of range at 2
    path[2] = torch.tensor([5, good[1], good[2], good[3]], dtype=torch.int32)    # bad root
    path[3] = torch.tensor([-2, good[1], good[2], good[3]], dtype=torch.int32)   # bad root below the tree
    path[4] = torch.tensor(good, dtype=torch.int32)                               # length 0: root only
    plen = torch.tensor([4, 4, 4, 4, 0], dtype=torch.int32)
    out = run_both(b0, w0, b1, path=path.cuda(), plen=plen.cuda())
    assert out["status"] & SSM_STATUS_PATH_RANGE
    assert out["sep_status"] & SSM_STATUS_PATH_RANGE
    check_oracle(b0, b1, out, [(i, j) for i in range(5) for j in range(2)],
                 paths=[good, good[:2], [0], [0], [0]])
    check_separate(out)


def test_2p7b_batch16_full_size_sampled():
    # the default benchmark's launch configuration: 16 sequences x 64 layers, 80 heads
    w0 = workload(3)
    w1 = next_workload(w0, 69, ("random", 16, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(0, 0), (15, 63), (7, 40), (3, 5)])
    check_separate(out)


@pytest.mark.parametrize("nxt", [("full", 2, 4), ("full", 3, 3), ("random", 64, 4, 15)])
def test_next_tree_of_several_node_tiles(nxt):
    # 31-, 40- and 64-node next trees (two, three and four node tiles, each with accumulators
    # sized to it): several node tiles per head group (the next group's x conv
    # runs in the last tile; the path-term product spans several k-steps), depth up to 15
    w0 = Workload(70, "tiles", Shape(H=8), n_layers=2, batch=2, trees=(("random", 16, 3, 4),), p_accept=0.9)
    w1 = next_workload(w0, 71, nxt)
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(2)])
    check_separate(out)


def test_stress_shape_ternary_next_tree_sampled():
    # the stress workload's shape (48 heads) and its 40-node ternary tree after a committed path
    w0 = workload(4)
    w1 = next_workload(w0, 72, ("full", 3, 3))
    b0, b1 = batch(w0, seqs=[0, 21, 63], tree=0), batch(w1, seqs=[0, 21, 63])
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(0, 0), (1, 24), (2, 47)])
    check_separate(out)


@pytest.mark.parametrize("gpc", ["2", "3"])
def test_several_head_groups_and_node_tiles(gpc, tuning):
    # several head groups per CTA (H = 10: the last one ragged) with a 40-node next tree
    tuning("SSM_VERIFY_GROUPS_PER_CTA", gpc)
    w0 = Workload(73, "groups x tiles", Shape(H=10), n_layers=2, batch=2, trees=(("random", 16, 3, 4),),
                  p_accept=0.9)
    w1 = next_workload(w0, 74, ("full", 3, 3))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(2)])
    check_separate(out)


def test_ring_positions_wrap_around():
    # ring heads just below the ring size and far beyond it: the committed rows and the
    # rows before the next root wrap around the 20-row ring
    w0 = Workload(75, "wrap", Shape(H=8), n_layers=2, batch=2, trees=(("chain", 8),), p_accept=1.0)
    w1 = next_workload(w0, 76, ("random", 16, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    b0["ring_head"][:] = np.array([[18, 19], [37, 1000001]], np.int32)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(2)])
    check_separate(out)


def test_split_prep_then_main_is_the_folded_call():
    """ssm_commit_verify_prep, then ssm_commit_verify_main on the same workspace, equals the
    one folded call bit for bit -- also when the x channels of the new tree's rows only
    arrive between the two (the prep reads B | C and dt only)."""
    from speculative_decoding_mamba2_gb300 import (ssm_accept_path, ssm_commit_verify, ssm_commit_verify_workspace_size,
                                                   ssm_tree_layout_build)
    w0 = Workload(91, "split", Shape(H=6), n_layers=2, batch=3, trees=(("random", 16, 3, 4),), p_accept=0.9)
    b0, b1 = batch(w0), batch(Workload(92, "split next", Shape(H=6), n_layers=2, batch=3,
                                       trees=(("random", 16, 3, 4),)))
    d0 = upload_tree_batch(b0, w0)
    dims, S, n0 = d0["dims"], d0["n_seq"], d0["n"]
    I = S * dims.n_layers
    mp = d0["depth"] + 1
    path = torch.empty((S, mp), dtype=torch.int32, device="cuda")
    plen = torch.empty(S, dtype=torch.int32, device="cuda")
    bonus = torch.empty(S, dtype=torch.int32, device="cuda")
    ssm_accept_path(S, n0, mp, d0["layout"], d0["tok"], d0["tgt"], path, plen, bonus)
    n1 = b1["n_nodes"]
    lay1_h, depth1 = ssm_tree_layout_build(b1["parent"])
    lay1 = dev(lay1_h)
    xBC1 = bf16_dev(b1["xBC"]).view(I, n1, dims.conv_dim)
    dt1 = bf16_dev(b1["dt"]).view(I, n1, dims.n_heads)
    outs = []
    for mode in ("all", "split", "late x"):
        h, ring, head = d0["h0"].clone(), d0["ring"].clone(), d0["ring_head"].clone()
        y = torch.full((I, n1, dims.d_inner), float("nan"), device="cuda")
        ws = torch.empty(ssm_commit_verify_workspace_size(dims, S, n1, depth1, mp), dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = (dims, d0["params"], S, n0, d0["layout"], mp, path, plen, d0["xBC"], d0["dt"], n1, depth1, lay1)
        x_in = xBC1.clone()
        if mode == "late x":
            x_in[..., :dims.d_inner] = float("nan")  # the x channels land after the prep
        if mode == "all":
            ssm_commit_verify(*args, x_in, dt1, h, ring, head, y, ws, status)
        else:
            ssm_commit_verify(*args, x_in, dt1, h, ring, head, y, ws, status, part="prep")
            # the prep leaves the ring head to the main half (every prep CTA reads the old one)
            assert torch.equal(head, d0["ring_head"])
            if mode == "late x":
                x_in[..., :dims.d_inner] = xBC1[..., :dims.d_inner]
            ssm_commit_verify(*args, x_in, dt1, h, ring, head, y, ws, status, part="main")
        torch.cuda.synchronize()
        assert int(status) == 0
        outs.append((y.cpu(), h.cpu(), ring.cpu(), head.cpu()))
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                               b.view(torch.int32) if b.dtype == torch.float32 else b)


@pytest.mark.parametrize("ctas", [1, 3, 0])
def test_persistent_ctas_walk_many_items(ctas, tuning):
    # the tensor-memory tree kernels are persistent: with 1 or 3 CTAs each walks many (instance,
    # head pair) items across instance boundaries (tables reloaded, accumulators and stages
    # reused); 0 = the default grid
    tuning("SSM_VERIFY_KERNEL", 2)
    tuning("SSM_VERIFY_CTAS", ctas)
    w0 = Workload(82, "multi-item", Shape(H=10), n_layers=3, batch=2, trees=(("random", 16, 3, 4),), p_accept=0.9)
    w1 = next_workload(w0, 83, ("random", 16, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(3)])
    check_separate(out)


@pytest.mark.parametrize("kernel", [1, 2])
def test_both_tree_kernel_sets(kernel, tuning):
    # 1: warp-level mma.sync (the default); 2: state contraction on tcgen05 with tensor-memory
    # accumulators
    tuning("SSM_VERIFY_KERNEL", kernel)
    w0 = Workload(84, "kernel sets", Shape(H=6), n_layers=2, batch=2, trees=(("random", 16, 3, 4),), p_accept=0.9)
    w1 = next_workload(w0, 85, ("full", 3, 3))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(2)])
    check_separate(out)


@pytest.mark.parametrize("deep", [1, 2])
def test_deep_and_shallow_pipelines(deep, tuning):
    # 1: two CTAs per SM, 3 state chunks in flight each; 2: one CTA per SM with the deep
    # pipeline (8 chunks in flight: more stages than a group's 8 chunks, so the next group's
    # chunks land during a group's epilogue); 2 groups per CTA, the last ragged
    tuning("SSM_VERIFY_DEEP", deep)
    tuning("SSM_VERIFY_GROUPS_PER_CTA", 2)
    w0 = Workload(86, "pipelines", Shape(H=10), n_layers=2, batch=2, trees=(("random", 16, 3, 4),), p_accept=0.9)
    w1 = next_workload(w0, 87, ("random", 14, 3, 4))
    b0, b1 = batch(w0), batch(w1)
    out = run_both(b0, w0, b1)
    assert out["status"] == 0 and out["sep_status"] == 0
    check_oracle(b0, b1, out, [(i, j) for i in range(2) for j in range(2)])
    check_separate(out)
