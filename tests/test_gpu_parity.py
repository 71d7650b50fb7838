"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Bar: indices (layout, accepted path, bonus, ring rows, heads) bit-exact;
floats max |gpu - ref| <= 1e-3 * (1 + |ref|) (fp32 state, bf16 inputs)."""
import numpy as np
import pytest
import torch

import oracle
from synth import WORKLOADS, Shape, Workload, batch, workload
from tests.helpers import (f64, oracle_verify_instance, params_at, rel_err, ring_window, run_tree_step,
                           upload_tree_batch)

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def check_instances(b, out, pairs, commit=True):
    """Compare sampled instances (seq index i, layer index j) with the oracle."""
    L = len(b["layers"])
    for i, j in pairs:
        inst = i * L + j
        y_ref, st = oracle_verify_instance(b, i, j, return_states=True)
        y = out["y"][inst].double().cpu().numpy()
        e = rel_err(y, y_ref)
        assert e <= TOL, f"y of instance ({i},{j}): {e}"
        path_ref, bonus_ref = oracle.accept(b["parent"][i], b["tok"][i], b["tgt"][i])
        plen = int(out["path_len"][i])
        assert out["path"][i, :plen].cpu().tolist() == path_ref
        assert int(out["bonus"][i]) == bonus_ref
        if not commit:
            continue
        h_ref, ring_ref, head_ref = oracle.commit(params_at(b["params"], j), b["parent"][i], path_ref,
                                                  f64(b["xBC"][i, j]), f64(b["dt"][i, j]),
                                                  b["h0"][i, j].astype(np.float64), f64(b["ring"][i, j]),
                                                  int(b["ring_head"][i, j]))
        np.testing.assert_array_equal(h_ref, st[path_ref[-1]])  # oracle self-consistency
        e = rel_err(out["h"][inst].double().cpu().numpy(), h_ref)
        assert e <= TOL, f"committed h of instance ({i},{j}): {e}"
        head = int(out["ring_head"][inst])
        assert head == head_ref
        ring_gpu = out["ring"][inst].view(torch.int16).cpu().numpy().view(np.uint16)
        ring_exp = b["ring"][i, j].copy()
        R = ring_exp.shape[0]
        for jj, m in enumerate(path_ref):
            ring_exp[(int(b["ring_head"][i, j]) + jj) % R] = b["xBC"][i, j, m]
        np.testing.assert_array_equal(ring_window(ring_gpu, head), ring_window(ring_exp, head))
    assert int(out["status"]) == 0


def test_tiny_130m_tree15_every_element():
    w = workload(0)
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(0, 0)])


def test_ragged_heads_and_node_tiles():
    # H = 6: head groups of 4 (+2 ragged) in verify, one ragged group of 8 in commit;
    # 40 nodes: node tiles 16 + 16 + 8
    w = Workload(50, "ragged", Shape(H=6), n_layers=2, batch=3, trees=(("full", 3, 3),), p_accept=0.9)
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(3) for j in range(2)])


@pytest.mark.parametrize("deep", ["1", "2"])
@pytest.mark.parametrize("spec", [("random", 16, 3, 4), ("random", 24, 3, 4), ("full", 3, 3), ("random", 64, 4, 15),
                                  ("chain", 16), ("full", 2, 5)])
def test_tree_shapes(spec, deep, tuning):
    # deep "1": two CTAs per SM with 3-4 chunks in flight; "2": one with 8 (where it fits: one
    # node tile)
    tuning("SSM_VERIFY_DEEP", deep)
    w = Workload(51, "shapes", Shape(H=8), n_layers=2, batch=2, trees=(spec,), p_accept=0.85)
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(2) for j in range(2)])


@pytest.mark.parametrize("gpc", ["2", "3"])
def test_several_head_groups_per_cta(gpc, tuning):
    # one CTA walks several head groups (the last one ragged): inputs of the next group
    # arrive while the current group's epilogue still reads its own
    tuning("SSM_VERIFY_GROUPS_PER_CTA", gpc)
    w = Workload(55, "groups", Shape(H=10), n_layers=2, batch=2, trees=(("random", 16, 3, 4),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(2) for j in range(2)])


@pytest.mark.parametrize("gpc", ["2", "3"])
def test_several_head_groups_and_node_tiles(gpc, tuning):
    # several head groups per CTA (the last one ragged) with a 40-node tree (three node
    # tiles): the next group's x conv runs inside the last tile of the current group
    tuning("SSM_VERIFY_GROUPS_PER_CTA", gpc)
    w = Workload(56, "groups x tiles", Shape(H=10), n_layers=2, batch=2, trees=(("full", 3, 3),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(2) for j in range(2)])


@pytest.mark.parametrize("g", ["2", "4"])
def test_two_and_four_head_groups(g, tuning):
    # the same small batch with 2-head and with 4-head groups (H = 10: the last group ragged
    # either way), against the oracle
    tuning("SSM_VERIFY_HEADS_PER_GROUP", g)
    w = Workload(57, "head groups", Shape(H=10), n_layers=2, batch=2, trees=(("random", 16, 3, 4),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(2) for j in range(2)])


@pytest.mark.parametrize("deep", ["1", "2"])
@pytest.mark.parametrize("g", ["2", "4"])
def test_deep_and_shallow_pipelines(deep, g, tuning):
    # the tree kernel with 3-4 state chunks in flight per CTA (1) or 8 at one CTA per SM (2),
    # 2- and 4-head groups, 3 groups per CTA (the last CTA's ragged)
    tuning("SSM_VERIFY_DEEP", deep)
    tuning("SSM_VERIFY_HEADS_PER_GROUP", g)
    tuning("SSM_VERIFY_GROUPS_PER_CTA", "3")
    w = Workload(58, "pipelines", Shape(H=14), n_layers=2, batch=2, trees=(("random", 16, 3, 4),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(2) for j in range(2)])


def test_single_node_tree():
    w = Workload(52, "root only", Shape(H=4), n_layers=3, batch=2, trees=(("chain", 1),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(2) for j in range(3)])
    assert out["path_len"].cpu().tolist() == [1, 1]


def test_2p7b_batch1_full_size_sampled():
    w = workload(2)
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(0, 0), (0, 31), (0, 63)])
    assert torch.isfinite(out["y"]).all()


def test_2p7b_batch16_full_size_sampled():
    w = workload(3)
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(0, 0), (15, 63), (7, 40), (3, 5), (12, 17)])
    assert torch.isfinite(out["y"]).all()
    # accepted paths of every sequence against the oracle (integers: all of them)
    for i in range(w.batch):
        path_ref, bonus_ref = oracle.accept(b["parent"][i], b["tok"][i], b["tgt"][i])
        assert out["path"][i, :int(out["path_len"][i])].cpu().tolist() == path_ref
        assert int(out["bonus"][i]) == bonus_ref


def test_780m_ternary40_sampled():
    w = workload(4)
    b = batch(w, seqs=[0, 21, 63], tree=0)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(0, 0), (1, 24), (2, 47)])


def test_chain_accept_and_commit_256():
    # the 256-node chain of the stress workload: accept and commit (path up to 256)
    w = workload(4)
    b = batch(w, seqs=[0, 1], layers=[0, 47], tree=1)
    d = upload_tree_batch(b, w)
    from speculative_decoding_mamba2_gb300 import ssm_accept_path, ssm_commit
    S, n, dims = d["n_seq"], d["n"], d["dims"]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    path = torch.empty((S, 256), dtype=torch.int32, device="cuda")
    plen = torch.empty(S, dtype=torch.int32, device="cuda")
    bonus = torch.empty(S, dtype=torch.int32, device="cuda")
    ssm_accept_path(S, n, 256, d["layout"], d["tok"], d["tgt"], path, plen, bonus, status)
    h, ring, head = d["h0"].clone(), d["ring"].clone(), d["ring_head"].clone()
    ssm_commit(dims, d["params"], S, n, d["layout"], 256, path, plen, d["xBC"], d["dt"], h, ring, head, status)
    torch.cuda.synchronize()
    assert int(status) == 0
    for i in range(S):
        path_ref, bonus_ref = oracle.accept(b["parent"][i], b["tok"][i], b["tgt"][i])
        assert path[i, :int(plen[i])].cpu().tolist() == path_ref and int(bonus[i]) == bonus_ref
        for j in range(2):
            h_ref, _, head_ref = oracle.commit(params_at(b["params"], j), b["parent"][i], path_ref,
                                               f64(b["xBC"][i, j]), f64(b["dt"][i, j]),
                                               b["h0"][i, j].astype(np.float64), f64(b["ring"][i, j]),
                                               int(b["ring_head"][i, j]))
            assert rel_err(h[i * 2 + j].double().cpu().numpy(), h_ref) <= TOL
            assert int(head[i * 2 + j]) == head_ref


def _chain_reference(b, i, j):
    """Oracle outputs of a chain by sequential one-token steps (pinned equal to the
    oracle's chain verify in test_oracle_pins.test_draft_chain_equals_chain_verify)."""
    prm = params_at(b["params"], j)
    h = b["h0"][i, j].astype(np.float64)
    ring = f64(b["ring"][i, j])
    head = int(b["ring_head"][i, j])
    xs, dts = f64(b["xBC"][i, j]), f64(b["dt"][i, j])
    ys = []
    for t in range(len(xs)):
        h, y, ring, _ = oracle.draft_step(prm, xs[t], dts[t], h, ring, head, t)
        ys.append(y)
    return np.stack(ys)


@pytest.mark.parametrize("n", [17, 40])
def test_chain_kernel_small(n):
    # chains deeper than the branching-tree limit take the on-chip walk
    w = Workload(56, "chain", Shape(H=5), n_layers=2, batch=2, trees=(("chain", n),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w), max_path=n)
    check_instances(b, out, [(i, j) for i in range(2) for j in range(2)])


def test_chain_kernel_longest_chain():
    # 4095 nodes, one below SSM_MAX_CHAIN_NODES: 256 chunks, the last one 15 nodes; an odd
    # head count (a CTA with one head); two layers
    from speculative_decoding_mamba2_gb300 import ssm_tree_verify, ssm_tree_verify_workspace_size
    n = 4095
    w = Workload(57, "longest chain", Shape(H=3), n_layers=2, batch=1, trees=(("chain", n),))
    b = batch(w)
    d = upload_tree_batch(b, w)
    dims, S = d["dims"], d["n_seq"]
    y = torch.full((S * 2, n, dims.d_inner), float("nan"), device="cuda")
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, d["depth"]), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm_tree_verify(dims, d["params"], S, n, d["depth"], d["layout"], d["xBC"], d["dt"], d["h0"], d["ring"],
                    d["ring_head"], y, ws, status)
    torch.cuda.synchronize()
    assert int(status) == 0
    for j in range(2):
        ref = _chain_reference(b, 0, j)
        assert rel_err(y[j].double().cpu().numpy(), ref) <= TOL, j


def test_780m_chain256_sampled():
    w = workload(4)
    b = batch(w, seqs=[0, 63], layers=[0, 47], tree=1)
    out = run_tree_step(upload_tree_batch(b, w), max_path=256, commit=False)
    for i, j in [(0, 0), (1, 1)]:
        ref = _chain_reference(b, i, j)
        assert rel_err(out["y"][i * 2 + j].double().cpu().numpy(), ref) <= TOL, (i, j)
    assert torch.isfinite(out["y"]).all()


def test_delta_zero_keeps_state_exactly():
    w = Workload(53, "dt=-inf", Shape(H=4), n_layers=1, batch=2, trees=(("random", 16, 3, 4),))
    b = batch(w)
    b["dt"][:] = 0xC61C  # bf16 -9984: softplus underflows to exactly 0
    out = run_tree_step(upload_tree_batch(b, w))
    np.testing.assert_array_equal(out["h"].cpu().numpy(), b["h0"].reshape(out["h"].shape))
    check_instances(b, out, [(0, 0), (1, 0)])


def test_verify_is_deterministic():
    w = Workload(54, "det", Shape(H=8), n_layers=2, batch=2, trees=(("random", 16, 3, 4),))
    b = batch(w)
    d = upload_tree_batch(b, w)
    a = run_tree_step(d)
    c = run_tree_step(d)
    assert torch.equal(a["y"], c["y"]) and torch.equal(a["h"], c["h"])


@pytest.mark.parametrize("ctas", [1, 2])
def test_persistent_ctas_walk_many_items(ctas, tuning):
    # the tensor-memory tree kernels with one or two persistent CTAs walking every (instance,
    # head pair) item, the instance tables reloaded at each instance boundary; a 40-node tree
    tuning("SSM_VERIFY_KERNEL", 2)
    tuning("SSM_VERIFY_CTAS", ctas)
    w = Workload(86, "multi-item plain", Shape(H=6), n_layers=3, batch=2, trees=(("full", 3, 3),))
    b = batch(w)
    out = run_tree_step(upload_tree_batch(b, w))
    check_instances(b, out, [(i, j) for i in range(2) for j in range(3)])
