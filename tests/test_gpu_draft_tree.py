"""Draft-side tree drafting on the GPU: ssm_draft_tree_level (one depth level per call,
branch states from the log) and ssm_draft_tree_commit (the accepted path from the log),
against the oracle's draft_tree_level / draft_tree_commit, and bit for bit against the
one-token draft step on a chain."""
import numpy as np
import pytest
import torch

import oracle
from synth import Shape, Workload, batch, workload
from tests.helpers import bf16_dev, dev, f64, params_at, params_dev, rel_err, ring_window

pytestmark = pytest.mark.gpu
TOL = 1e-3       # y: |got - ref| <= 1e-3 (1 + |ref|)
LOG_TOL = 1e-5   # logged Δ, B, x: conv + SiLU + softplus in fp32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def upload(b, w):
    from speculative_decoding_mamba2_gb300 import Dims, ssm_tree_layout_build
    S, L, n = len(b["seqs"]), len(b["layers"]), b["n_nodes"]
    I = S * L
    dims = Dims(n_heads=w.shape.H, n_layers=L, ring_cap=w.ring_cap)
    layout, depth = ssm_tree_layout_build(b["parent"])
    return dict(dims=dims, S=S, n=n, I=I, depth=depth, layout=dev(layout), prm=params_dev(b["params"]),
                xBC=bf16_dev(b["xBC"]).view(I, n, dims.conv_dim), dt=bf16_dev(b["dt"]).view(I, n, dims.n_heads),
                h=dev(b["h0"]).view(I, dims.n_heads, dims.head_dim, dims.d_state),
                ring=bf16_dev(b["ring"]).view(I, w.ring_cap, dims.conv_dim), head=dev(b["ring_head"]).view(I),
                tok=dev(b["tok"]), tgt=dev(b["tgt"]))


def draft_levels(d, levels=None):
    from speculative_decoding_mamba2_gb300 import ssm_draft_tree_level, ssm_draft_tree_workspace_size
    dims, I, n = d["dims"], d["I"], d["n"]
    ws = torch.empty(ssm_draft_tree_workspace_size(dims, d["S"], n), dtype=torch.uint8, device="cuda")
    logs = dict(delta=torch.full((I, n, dims.n_heads), float("nan"), device="cuda"),
                B=torch.full((I, n, dims.d_state), float("nan"), device="cuda"),
                x=torch.full((I, n, dims.d_inner), float("nan"), device="cuda"))
    y = torch.full((I, n, dims.d_inner), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for lv in (range(d["depth"] + 1) if levels is None else levels):
        ssm_draft_tree_level(dims, d["prm"], d["S"], n, lv, d["layout"], d["xBC"], d["dt"], d["h"], d["ring"],
                             d["head"], logs["delta"], logs["B"], logs["x"], y, ws, status)
    torch.cuda.synchronize()
    return y, logs, status


def oracle_levels(b, i, j):
    prm = params_at(b["params"], j)
    parent = b["parent"][i]
    lay = oracle.tree_layout(parent)
    xBC, dt = f64(b["xBC"][i, j]), f64(b["dt"][i, j])
    h0, ring, head = b["h0"][i, j].astype(np.float64), f64(b["ring"][i, j]), int(b["ring_head"][i, j])
    ys, log = {}, {}
    for lv in range(max(lay["depth"]) + 1):
        y_l, rows = oracle.draft_tree_level(prm, parent, lv, xBC, dt, h0, ring, head, log)
        ys.update(y_l)
        log.update(rows)
    return np.stack([ys[v] for v in range(len(parent))]), log


def check_levels(b, w, d, y, logs, pairs):
    L = len(b["layers"])
    for i, j in pairs:
        ref_y, ref_log = oracle_levels(b, i, j)
        inst = i * L + j
        assert rel_err(y[inst].cpu().numpy(), ref_y) <= TOL
        for v, (dl, Bv, xv) in ref_log.items():
            assert rel_err(logs["delta"][inst, v].cpu().numpy(), dl) <= LOG_TOL
            assert rel_err(logs["B"][inst, v].cpu().numpy(), Bv) <= LOG_TOL
            assert rel_err(logs["x"][inst, v].cpu().numpy(), xv) <= LOG_TOL


def test_draft_tree_levels_small():
    # two sequences with different random trees, three heads (the last CTA holds one head)
    w = Workload(50, "draft tree small", Shape(H=3), n_layers=2, batch=2, trees=(("random", 14, 3, 4),))
    b = batch(w)
    d = upload(b, w)
    y, logs, status = draft_levels(d)
    assert int(status) == 0
    check_levels(b, w, d, y, logs, [(i, j) for i in range(2) for j in range(2)])


def test_draft_tree_wide_level_and_max_nodes():
    # a root with 40 children, then 23 grandchildren: level 1 takes five 8-node passes;
    # 64 nodes is the cap
    parent = [-1] + [0] * 40 + [1 + (k * 7) % 40 for k in range(23)]
    parent = [-1] + sorted(parent[1:])
    w = Workload(51, "draft tree wide", Shape(H=2), n_layers=1, batch=1, trees=(("random", 64, 64, 2),))
    b = batch(w)
    b["parent"][0] = np.asarray(parent, np.int32)
    d = upload(b, w)
    y, logs, status = draft_levels(d)
    assert int(status) == 0
    check_levels(b, w, d, y, logs, [(0, 0)])


def test_draft_tree_level_without_nodes_is_a_no_op():
    w = Workload(52, "draft tree empty level", Shape(H=2), n_layers=1, batch=1, trees=(("random", 6, 2, 2),))
    b = batch(w)
    d = upload(b, w)
    y, logs, status = draft_levels(d, levels=[d["depth"] + 1, 15])
    assert int(status) == 0
    assert torch.isnan(y).all() and torch.isnan(logs["x"]).all() and torch.isnan(logs["delta"]).all()


def commit(d, logs, path, plen, max_path):
    from speculative_decoding_mamba2_gb300 import ssm_draft_tree_commit
    h, ring, head = d["h"].clone(), d["ring"].clone(), d["head"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm_draft_tree_commit(d["dims"], d["prm"], d["S"], d["n"], d["layout"], max_path, path, plen, logs["delta"],
                          logs["B"], logs["x"], d["xBC"], h, ring, head, status)
    torch.cuda.synchronize()
    return h, ring, head, int(status)


def test_draft_tree_accept_and_commit():
    from speculative_decoding_mamba2_gb300 import ssm_accept_path
    w = Workload(53, "draft tree commit", Shape(H=4), n_layers=2, batch=3, trees=(("random", 16, 3, 4),))
    b = batch(w)
    d = upload(b, w)
    y, logs, status = draft_levels(d)
    max_path = d["depth"] + 1
    path = torch.empty((d["S"], max_path), dtype=torch.int32, device="cuda")
    plen = torch.empty(d["S"], dtype=torch.int32, device="cuda")
    bonus = torch.empty(d["S"], dtype=torch.int32, device="cuda")
    ssm_accept_path(d["S"], d["n"], max_path, d["layout"], d["tok"], d["tgt"], path, plen, bonus, status)
    h, ring, head, st = commit(d, logs, path, plen, max_path)
    assert int(status) == 0 and st == 0
    L, R = len(b["layers"]), w.ring_cap
    for i in range(d["S"]):
        ref_path, _ = oracle.accept(b["parent"][i], b["tok"][i], b["tgt"][i])
        assert path[i, :plen[i]].tolist() == ref_path
        for j in range(L):
            inst = i * L + j
            _, ref_log = oracle_levels(b, i, j)
            h_ref, ring_ref, head_ref = oracle.draft_tree_commit(
                params_at(b["params"], j)["A_log"], b["parent"][i], ref_path, ref_log, f64(b["xBC"][i, j]),
                b["h0"][i, j].astype(np.float64), f64(b["ring"][i, j]), int(b["ring_head"][i, j]))
            assert rel_err(h[inst].cpu().numpy(), h_ref) <= TOL
            assert int(head[inst]) == head_ref
            got = ring_window(f64(ring[inst].view(torch.int16).cpu().numpy().view(np.uint16)), head_ref)
            np.testing.assert_array_equal(got, ring_window(ring_ref, head_ref))


def test_draft_tree_commit_bad_and_empty_paths():
    w = Workload(54, "draft tree bad path", Shape(H=2), n_layers=1, batch=2, trees=(("random", 10, 3, 3),))
    b = batch(w)
    d = upload(b, w)
    _, logs, _ = draft_levels(d)
    lay = oracle.tree_layout(b["parent"][0])
    leaf_path = lay["path"][len(b["parent"][0]) - 1]
    max_path = d["depth"] + 1
    p = np.full((2, max_path), -1, np.int32)
    p[0, :len(leaf_path)] = leaf_path
    p[0, len(leaf_path) - 1] = 0  # the last entry is not a child of the one before
    h, ring, head, st = commit(d, logs, dev(p), dev(np.array([len(leaf_path), 0], np.int32)), max_path)
    assert st & 2  # SSM_STATUS_PATH_RANGE
    # sequence 0 commits the valid prefix, sequence 1 (path_len 0) nothing
    _, ref_log = oracle_levels(b, 0, 0)
    prefix = leaf_path[:-1]
    h_ref, _, head_ref = oracle.draft_tree_commit(params_at(b["params"], 0)["A_log"], b["parent"][0], prefix, ref_log,
                                                  f64(b["xBC"][0, 0]), b["h0"][0, 0].astype(np.float64),
                                                  f64(b["ring"][0, 0]), int(b["ring_head"][0, 0]))
    assert rel_err(h[0].cpu().numpy(), h_ref) <= TOL and int(head[0]) == head_ref
    assert torch.equal(h[1], d["h"][1]) and torch.equal(ring[1], d["ring"][1]) and int(head[1]) == int(d["head"][1])


def test_draft_tree_chain_bit_exact_with_draft_steps():
    # a 16-node chain drafted level by level logs exactly what sixteen ssm_draft_step calls
    # log, and committing k path nodes gives the stepped state k bit for bit
    from speculative_decoding_mamba2_gb300 import Dims, ssm_draft_step
    T = 16
    w = Workload(55, "draft tree chain", Shape(H=4), n_layers=2, batch=1, trees=(("chain", T),), ring_cap=20)
    b = batch(w)
    d = upload(b, w)
    y, logs, status = draft_levels(d)
    dims, I = d["dims"], d["I"]
    h_work = torch.empty_like(d["h"])
    ring, head = d["ring"].clone(), d["head"].clone()
    sl = dict(delta=torch.zeros(I, T, dims.n_heads, device="cuda"), B=torch.zeros(I, T, dims.d_state, device="cuda"),
              x=torch.zeros(I, T, dims.d_inner, device="cuda"), len=torch.zeros(I, dtype=torch.int32, device="cuda"))
    states = []
    ys = []
    for t in range(T):
        yt = torch.empty(I, dims.d_inner, device="cuda")
        ssm_draft_step(dims, d["prm"], 1, t, T, d["xBC"][:, t].contiguous(), d["dt"][:, t].contiguous(),
                       d["h"] if t == 0 else h_work, h_work, ring, head, sl["delta"], sl["B"], sl["x"], sl["len"], yt,
                       status)
        states.append(h_work.clone())
        ys.append(yt)
    torch.cuda.synchronize()
    assert int(status) == 0
    assert torch.equal(logs["delta"], sl["delta"]) and torch.equal(logs["B"], sl["B"]) and torch.equal(logs["x"], sl["x"])
    assert rel_err(y.cpu().numpy(), torch.stack(ys, 1).cpu().numpy()) <= TOL
    for k in (1, 7, T):
        path = dev(np.arange(T, dtype=np.int32)[None])
        h, _, hd, st = commit(d, logs, path, dev(np.array([k], np.int32)), T)
        assert st == 0 and torch.equal(h, states[k - 1]) and int(hd[0]) == int(d["head"][0]) + k


def test_draft_tree_full_size_sampled():
    # the 370M draft shape, 48 layers, the 16-node random tree: every level, sampled layers
    w = workload(5)
    b = batch(w)
    d = upload(b, w)
    y, logs, status = draft_levels(d)
    assert int(status) == 0
    assert not torch.isnan(y).any()
    check_levels(b, w, d, y, logs, [(0, 0), (0, 23), (0, 47)])


def test_draft_tree_runs_across_sequences():
    # 2 sequences x 8 layers x 32 heads = 512 (instance, head) items for the level kernel's
    # persistent CTAs: runs cross instances and, at the middle, sequences (different trees)
    w = Workload(58, "draft tree runs", Shape(H=32), n_layers=8, batch=2, trees=(("random", 16, 3, 4),))
    b = batch(w)
    d = upload(b, w)
    y, logs, status = draft_levels(d)
    assert int(status) == 0
    check_levels(b, w, d, y, logs, [(i, j) for i in range(2) for j in (0, 3, 7)])


def test_draft_tree_bad_layout_is_flagged_and_writes_nothing():
    # sequence 1's node 3 takes a conv tap from a later node: that sequence's instances write
    # no log row and no y at any level, the status says so, sequence 0 is unaffected
    from speculative_decoding_mamba2_gb300 import SSM_STATUS_BAD_LAYOUT
    w = Workload(59, "draft tree bad layout", Shape(H=3), n_layers=2, batch=2, trees=(("random", 12, 3, 4),))
    b = batch(w)
    d = upload(b, w)
    lay = d["layout"].view(2, d["n"], 8)
    lay[1, 3, 4] = 5  # tap d = 1 of node 3 -> node 5
    y, logs, status = draft_levels(d)
    assert int(status) & SSM_STATUS_BAD_LAYOUT
    L = len(b["layers"])
    bad = slice(L, 2 * L)
    assert torch.isnan(y[bad]).all() and torch.isnan(logs["x"][bad]).all()
    assert torch.isnan(logs["B"][bad]).all() and torch.isnan(logs["delta"][bad]).all()
    check_levels(b, w, d, y, logs, [(0, 0), (0, 1)])
