"""libssmtree's C ABI on the CPU: it builds, loads, exports every symbol the
header declares, its host-only layout builder matches the oracle bit for bit,
and every device entry point rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from speculative_decoding_mamba2_gb300 import binding as B
from speculative_decoding_mamba2_gb300 import build as BLD
from synth import WORKLOADS, Shape, Workload, tree_parents

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ssm_tree.h")


@pytest.fixture(scope="module")
def L():
    BLD.build()
    return B.lib()


def declared_functions():
    src = open(HEADER).read() + open(os.path.join(os.path.dirname(HEADER), "ssm_layer.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    fns = declared_functions()
    for name in ["ssm_tree_layout_build", "ssm_tree_verify", "ssm_tree_verify_workspace_size", "ssm_accept_path",
                 "ssm_commit", "ssm_draft_step", "ssm_replay", "ssm_last_error", "ssm_version"]:
        assert name in fns


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert B.ssm_version() >= 100
    assert B.library_path().endswith("libssmtree.so")


def _oracle_records(parent):
    lay = oracle.tree_layout(parent)
    n = lay["n"]
    out = np.zeros((n, 8), np.int32)
    for v in range(n):
        ch = lay["children"][v]
        out[v] = [lay["parent"][v], lay["depth"][v], ch[0] if ch else n, len(ch), *lay["taps"][v], 0]
    return out, max(lay["depth"])


def test_layout_build_matches_oracle(L):
    trees = [[-1], [-1, 0, 0, 1, 1, 2, 3], list(range(-1, 255))]
    for cfg, tr in [(0, 0), (2, 0), (4, 0), (4, 1)]:
        w = WORKLOADS[cfg]
        trees += [tree_parents(w, s, tr) for s in range(6)]
    w = Workload(97, "layout", Shape(H=1), 1, 1, trees=(("random", 40, 4, 9),))
    trees += [tree_parents(w, s) for s in range(30)]
    for par in trees:
        got, depth = B.ssm_tree_layout_build(par)
        ref, rdepth = _oracle_records(par)
        np.testing.assert_array_equal(got[0], ref)
        assert depth == rdepth


def test_layout_build_batched_and_caps(L):
    w = WORKLOADS[3]
    par = np.stack([tree_parents(w, s) for s in range(16)])
    got, depth = B.ssm_tree_layout_build(par, max_branches=3, max_depth=4)
    assert got.shape == (16, 16, 8) and depth <= 4
    for s in range(16):
        np.testing.assert_array_equal(got[s], _oracle_records(par[s])[0])
    with pytest.raises(B.SSMError) as e:
        B.ssm_tree_layout_build(np.arange(-1, 9), max_depth=4)
    assert e.value.code == B.SSM_ERR_CAPACITY
    with pytest.raises(B.SSMError) as e:
        B.ssm_tree_layout_build([-1, 0, 0, 0, 0], max_branches=3)
    assert e.value.code == B.SSM_ERR_CAPACITY


@pytest.mark.parametrize("bad", [[0], [-1, 1], [-1, 0, 2], [-1, 0, 1, 0], [-1, -1], [5, 0]])
def test_layout_build_rejects_what_the_oracle_rejects(L, bad):
    with pytest.raises(oracle.BadTree):
        oracle.tree_layout(bad)
    with pytest.raises(B.SSMError) as e:
        B.ssm_tree_layout_build(bad)
    assert e.value.code == B.SSM_ERR_BAD_TREE
    assert "ssm_tree_layout_build" in B.ssm_last_error()


# ---------------------------------------------------------------------------
# device entry points: argument validation happens before any CUDA call
# ---------------------------------------------------------------------------
def _dims(**kw):
    d = dict(n_heads=4, head_dim=64, d_state=128, conv_width=4, n_layers=2, ring_cap=20)
    d.update(kw)
    return B.ssm_dims(**d)


def _prm(null=False):
    x = None if null else 16
    return B.ssm_params(16, 16, 16, x, 16)


FAKE = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first


def _verify(L, dims, prm, n_seq=1, n=16, depth=4, ptr=FAKE, ws_bytes=1 << 30):
    return L.ssm_tree_verify(ctypes.byref(dims) if dims is not None else None,
                             ctypes.byref(prm) if prm is not None else None,
                             n_seq, n, depth, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ctypes.c_size_t(ws_bytes),
                             None, None)


def test_verify_validation(L):
    assert _verify(L, None, _prm()) == B.SSM_ERR_INVALID_ARG
    assert _verify(L, _dims(), None) == B.SSM_ERR_INVALID_ARG
    assert _verify(L, _dims(head_dim=32), _prm()) == B.SSM_ERR_INVALID_ARG
    assert _verify(L, _dims(d_state=64), _prm()) == B.SSM_ERR_INVALID_ARG
    assert _verify(L, _dims(conv_width=3), _prm()) == B.SSM_ERR_INVALID_ARG
    assert _verify(L, _dims(ring_cap=2), _prm()) == B.SSM_ERR_INVALID_ARG
    assert _verify(L, _dims(), _prm(null=True)) == B.SSM_ERR_INVALID_ARG
    assert _verify(L, _dims(), _prm(), n=65, depth=4) == B.SSM_ERR_CAPACITY
    assert _verify(L, _dims(), _prm(), n=64, depth=16) == B.SSM_ERR_CAPACITY
    assert _verify(L, _dims(), _prm(), n=8, depth=8) == B.SSM_ERR_RANGE
    assert _verify(L, _dims(), _prm(), ptr=None) == B.SSM_ERR_INVALID_ARG
    assert "NULL" in B.ssm_last_error()
    assert _verify(L, _dims(), _prm(), n_seq=-1) == B.SSM_ERR_INVALID_ARG
    # an empty batch is a valid no-op and enqueues nothing
    assert _verify(L, _dims(), _prm(), n_seq=0, ptr=None) == B.SSM_OK
    # workspace: size query, too-small and misaligned workspaces are rejected before any CUDA call
    need = B.ssm_tree_verify_workspace_size(B.Dims(n_heads=4, n_layers=2), 1, 16, 4)
    assert need > 0 and need % 16 == 0
    assert _verify(L, _dims(), _prm(), ws_bytes=need - 16) == B.SSM_ERR_CAPACITY
    assert _verify(L, _dims(), _prm(), ptr=ctypes.c_void_p(24)) == B.SSM_ERR_INVALID_ARG
    assert B.ssm_tree_verify_workspace_size(B.Dims(n_heads=4, n_layers=2), 3, 16, 4) == 3 * need
    with pytest.raises(B.SSMError):
        B.ssm_tree_verify_workspace_size(B.Dims(n_heads=4, n_layers=2), 1, 65, 4)


def _commit_verify(L, dims, prm, n_seq=1, prev_n=16, lp=5, n=16, depth=4, ptr=FAKE, ws_bytes=1 << 30):
    return L.ssm_commit_verify(ctypes.byref(dims), ctypes.byref(prm) if prm is not None else None, n_seq, prev_n,
                               ptr, lp, ptr, ptr, ptr, ptr, n, depth, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr,
                               ctypes.c_size_t(ws_bytes), None, None)


def test_commit_verify_validation(L):
    d, p = _dims(), _prm()
    assert _commit_verify(L, d, p, n_seq=0, ptr=None) == B.SSM_OK
    assert _commit_verify(L, d, None) == B.SSM_ERR_INVALID_ARG
    assert _commit_verify(L, d, p, ptr=None) == B.SSM_ERR_INVALID_ARG
    assert _commit_verify(L, d, p, lp=0) == B.SSM_ERR_RANGE
    assert _commit_verify(L, d, p, lp=17) == B.SSM_ERR_RANGE  # paths of trees the tree kernel verifies
    assert _commit_verify(L, d, p, prev_n=0) == B.SSM_ERR_RANGE
    assert _commit_verify(L, d, p, prev_n=65) == B.SSM_ERR_RANGE
    assert _commit_verify(L, _dims(ring_cap=7), p, lp=5) == B.SSM_ERR_CAPACITY  # rows before the path kept
    assert _commit_verify(L, d, p, n=256, depth=255) == B.SSM_ERR_CAPACITY  # long chains: separate calls
    assert "chain" in B.ssm_last_error()
    assert _commit_verify(L, d, p, n=8, depth=8) == B.SSM_ERR_RANGE
    assert _commit_verify(L, d, p, ptr=ctypes.c_void_p(24)) == B.SSM_ERR_INVALID_ARG
    dims = B.Dims(n_heads=4, n_layers=2)
    need = B.ssm_commit_verify_workspace_size(dims, 1, 16, 4, 5)
    assert need % 16 == 0 and need > B.ssm_tree_verify_workspace_size(dims, 1, 16, 4)
    assert B.ssm_commit_verify_workspace_size(dims, 3, 16, 4, 5) == 3 * need
    assert _commit_verify(L, d, p, ws_bytes=need - 16) == B.SSM_ERR_CAPACITY
    with pytest.raises(B.SSMError):
        B.ssm_commit_verify_workspace_size(dims, 1, 16, 4, 17)


def test_accept_commit_draft_replay_validation(L):
    P = FAKE
    assert L.ssm_accept_path(1, 16, 0, P, P, P, P, P, P, None, None) == B.SSM_ERR_RANGE
    assert L.ssm_accept_path(1, 16, 257, P, P, P, P, P, P, None, None) == B.SSM_ERR_RANGE
    assert L.ssm_accept_path(1, 0, 5, P, P, P, P, P, P, None, None) == B.SSM_ERR_INVALID_ARG
    assert L.ssm_accept_path(1, 16, 5, P, None, P, P, P, P, None, None) == B.SSM_ERR_INVALID_ARG
    assert L.ssm_accept_path(0, 16, 5, None, None, None, None, None, None, None, None) == B.SSM_OK
    d, p = _dims(), _prm()
    assert L.ssm_commit(ctypes.byref(d), ctypes.byref(p), 1, 16, P, 0, P, P, P, P, P, P, P, None,
                        None) == B.SSM_ERR_RANGE
    assert L.ssm_commit(ctypes.byref(d), ctypes.byref(p), 1, 16, P, 5, P, P, P, P, None, P, P, None,
                        None) == B.SSM_ERR_INVALID_ARG
    dd = _dims(ring_cap=10)
    # step + 3 must stay below ring_cap so the three committed rows survive drafting
    assert L.ssm_draft_step(ctypes.byref(dd), ctypes.byref(p), 1, 7, 16, P, P, P, P, P, P, P, P, P, P, P, None,
                            None) == B.SSM_ERR_CAPACITY
    assert L.ssm_draft_step(ctypes.byref(d), ctypes.byref(p), 1, 16, 16, P, P, P, P, P, P, P, P, P, P, P, None,
                            None) == B.SSM_ERR_RANGE
    assert L.ssm_draft_step(ctypes.byref(d), ctypes.byref(p), 1, -1, 16, P, P, P, P, P, P, P, P, P, P, P, None,
                            None) == B.SSM_ERR_RANGE
    assert L.ssm_replay(ctypes.byref(d), ctypes.byref(_prm(null=True)), 1, 16, P, P, P, P, P, P, P, None,
                        None) == B.SSM_ERR_INVALID_ARG
    assert L.ssm_replay(ctypes.byref(d), ctypes.byref(p), 1, 0, P, P, P, P, P, P, P, None,
                        None) == B.SSM_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(L):
    import torch
    t = torch.zeros(4)
    with pytest.raises(ValueError):
        B._dev(t, "t", torch.float32, 4)


def _level(L, dims, prm, n_seq=1, n=16, level=0, ptr=FAKE, h=FAKE, ws=FAKE, ws_bytes=1 << 30):
    P = ptr
    return L.ssm_draft_tree_level(ctypes.byref(dims), ctypes.byref(prm), n_seq, n, level, P, P, P, h, P, P, P, P,
                                  P, P, ws, ctypes.c_size_t(ws_bytes), None, None)


def test_draft_tree_validation(L):
    d, p = _dims(), _prm()
    assert _level(L, d, p, n=0) == B.SSM_ERR_INVALID_ARG
    assert _level(L, d, p, n=65) == B.SSM_ERR_CAPACITY
    assert _level(L, d, p, level=-1) == B.SSM_ERR_RANGE
    assert _level(L, d, p, level=16) == B.SSM_ERR_RANGE
    assert _level(L, d, p, n_seq=-1) == B.SSM_ERR_INVALID_ARG
    assert _level(L, d, p, n_seq=0, ptr=None, h=None, ws=None) == B.SSM_OK  # nothing to do, no CUDA call
    assert _level(L, d, p, ptr=None) == B.SSM_ERR_INVALID_ARG
    assert _level(L, d, p, ws=None) == B.SSM_ERR_INVALID_ARG
    assert _level(L, d, p, h=ctypes.c_void_p(24)) == B.SSM_ERR_INVALID_ARG  # not 16-byte aligned
    assert _level(L, d, _prm(null=True)) == B.SSM_ERR_INVALID_ARG
    need = L.ssm_draft_tree_workspace_size(ctypes.byref(d), 1, 16)
    # C rows, e^S, path sums and the 16 path products per node and instance, each part 128-byte aligned
    assert need >= 16 * (128 + d.n_heads + d.n_heads * 64 + 16) * 4 * d.n_layers and need % 128 == 0
    assert _level(L, d, p, ws_bytes=need - 1) == B.SSM_ERR_CAPACITY
    assert L.ssm_draft_tree_workspace_size(ctypes.byref(d), 1, 65) == 0
    P = FAKE
    # commit: (dims, prm, n_seq, n, layout, max_path, path, path_len, log_d, log_B, log_x, xBC, h, ring, head)
    assert L.ssm_draft_tree_commit(ctypes.byref(d), ctypes.byref(p), 1, 16, P, 0, P, P, P, P, P, P, P, P, P, None,
                                   None) == B.SSM_ERR_RANGE
    assert L.ssm_draft_tree_commit(ctypes.byref(d), ctypes.byref(p), 1, 16, P, 257, P, P, P, P, P, P, P, P, P, None,
                                   None) == B.SSM_ERR_RANGE
    assert L.ssm_draft_tree_commit(ctypes.byref(d), ctypes.byref(p), 1, 65, P, 5, P, P, P, P, P, P, P, P, P, None,
                                   None) == B.SSM_ERR_CAPACITY
    assert L.ssm_draft_tree_commit(ctypes.byref(d), ctypes.byref(p), 1, 16, P, 5, P, None, P, P, P, P, P, P, P, None,
                                   None) == B.SSM_ERR_INVALID_ARG
    assert L.ssm_draft_tree_commit(ctypes.byref(d), ctypes.byref(p), 1, 16, P, 5, P, P, P, ctypes.c_void_p(20), P, P,
                                   P, P, P, None, None) == B.SSM_ERR_INVALID_ARG  # log_B not 16-byte aligned
    assert L.ssm_draft_tree_commit(ctypes.byref(d), ctypes.byref(_prm(null=True)), 1, 16, P, 5, P, P, P, P, P, P, P,
                                   P, P, None, None) == B.SSM_ERR_INVALID_ARG
    assert L.ssm_draft_tree_commit(ctypes.byref(d), ctypes.byref(p), 0, 16, None, 5, None, None, None, None, None,
                                   None, None, None, None, None, None) == B.SSM_OK


def test_selftest_bounded_wait_validation(L):
    assert L.ssm_selftest_bounded_wait(0, FAKE, None) == B.SSM_ERR_RANGE
    assert L.ssm_selftest_bounded_wait(1000001, FAKE, None) == B.SSM_ERR_RANGE
    assert L.ssm_selftest_bounded_wait(1000, None, None) == B.SSM_ERR_INVALID_ARG


def test_set_tuning_validation(L):
    # no CUDA call: the knobs are host-side plan overrides
    from speculative_decoding_mamba2_gb300 import SSM_ERR_INVALID_ARG, SSM_OK
    for name in (b"SSM_VERIFY_GROUPS_PER_CTA", b"SSM_VERIFY_HEADS_PER_GROUP", b"SSM_LINEAR_TCHUNK",
                 b"SSM_LINEAR_SPLITS", b"SSM_LINEAR_STAGES", b"SSM_VERIFY_KERNEL", b"SSM_VERIFY_CTAS",
                 b"SSM_VERIFY_DEEP"):
        assert L.ssm_set_tuning(name, 2) == SSM_OK
        assert L.ssm_set_tuning(name, 0) == SSM_OK
    assert L.ssm_set_tuning(b"SSM_NO_SUCH_KNOB", 1) == SSM_ERR_INVALID_ARG
    assert "unknown" in L.ssm_last_error().decode()
    assert L.ssm_set_tuning(b"SSM_LINEAR_STAGES", -1) == SSM_ERR_INVALID_ARG
    assert L.ssm_set_tuning(None, 1) == SSM_ERR_INVALID_ARG


def test_selftest_silu_validation(L):
    assert L.ssm_selftest_silu(FAKE, FAKE, -1, None) == B.SSM_ERR_RANGE
    assert L.ssm_selftest_silu(None, FAKE, 4, None) == B.SSM_ERR_INVALID_ARG
    assert L.ssm_selftest_silu(FAKE, None, 4, None) == B.SSM_ERR_INVALID_ARG
    assert L.ssm_selftest_silu(None, None, 0, None) == B.SSM_OK  # nothing to do, no CUDA call
