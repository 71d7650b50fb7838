"""Pins for the oracle's draft-tree functions (draft_tree_level, draft_tree_commit), on the
CPU, each against something other than themselves: the one-token draft step and replay
(themselves pinned in test_oracle_pins.py), tree verification and the target's commit
(pinned there by closed forms, brute force and the dual form), and a hand-derived closed
form.  Plausible mistakes planted in the two functions are caught by at least one pin."""
import math

import numpy as np
import pytest

import oracle
import oracle.ssm_oracle as so
from tests.test_oracle_pins import rand_params, rand_problem, _scalar_params, _s


def _all_levels(prm, parent, xBC, dt, h, ring, head):
    lay = oracle.tree_layout(parent)
    log, ys = {}, {}
    for d in range(max(lay["depth"]) + 1):
        y_d, rows = oracle.draft_tree_level(prm, parent, d, xBC, dt, h, ring, head, log)
        assert set(y_d) == {v for v in range(lay["n"]) if lay["depth"][v] == d}
        ys.update(y_d)
        log.update(rows)
    return np.stack([ys[v] for v in range(lay["n"])]), log


def test_draft_tree_chain_equals_draft_steps():
    # a chain drafted level by level = sixteen one-token draft steps (same y, same log rows)
    g = np.random.default_rng(31)
    H, P, N, R, head, T = 2, 3, 4, 20, 3, 16
    prm = rand_params(H, P, N, g)
    conv_dim = H * P + 2 * N
    xs = g.normal(0, 1, (T, conv_dim))
    dts = g.normal(0, 0.5, (T, H))
    h0 = g.normal(0, 0.1, (H, P, N))
    ring = g.normal(0, 1, (R, conv_dim))
    parent = np.arange(-1, T - 1)
    y_tree, log = _all_levels(prm, parent, xs, dts, h0, ring, head)
    h, r = h0, ring
    for t in range(T):
        h, y, r, row = oracle.draft_step(prm, xs[t], dts[t], h, r, head, t)
        np.testing.assert_array_equal(y_tree[t], y)
        for a, b in zip(log[t], row):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("seed", [41, 42, 43])
def test_draft_tree_levels_equal_tree_verify(seed):
    # every node's output from the level-by-level draft = verification of the whole tree
    g = np.random.default_rng(seed)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, n=16)
    y_tree, _ = _all_levels(prm, parent, xBC, dt, h0, ring, head)
    np.testing.assert_allclose(y_tree, oracle.verify(prm, parent, xBC, dt, h0, ring, head), rtol=1e-13, atol=1e-14)


def test_draft_tree_closed_form_branching():
    # H = P = N = 1, taps [0,0,0,1], decay 1/2, Δ = ln 2: root with two children, each
    # child from the root's state (not its sibling's)
    ln2 = math.log(2.0)
    pre = np.array([[1.0, 1.0, 2.0], [2.0, -1.0, 0.5], [-1.0, 3.0, 1.0]])
    prm = _scalar_params()
    y, log = _all_levels(prm, [-1, 0, 0], pre, np.zeros((3, 1)), np.ones((1, 1, 1)), np.zeros((4, 3)), 3)
    x = [_s(r[0]) for r in pre]
    B = [_s(r[1]) for r in pre]
    C = [_s(r[2]) for r in pre]
    hr = 0.5 + ln2 * x[0] * B[0]
    ha = 0.5 * hr + ln2 * x[1] * B[1]
    hb = 0.5 * hr + ln2 * x[2] * B[2]
    np.testing.assert_allclose(y[:, 0], [C[0] * hr + 0.25 * x[0], C[1] * ha + 0.25 * x[1], C[2] * hb + 0.25 * x[2]],
                               rtol=1e-15)
    for v in range(3):  # log rows: Δ = ln 2, post-conv B and x
        np.testing.assert_allclose([log[v][0][0], log[v][1][0], log[v][2][0]], [ln2, B[v], x[v]], rtol=1e-15)
    # commit of the accepted path root -> 2
    h, _, hd = oracle.draft_tree_commit(prm["A_log"], [-1, 0, 0], [0, 2], log, pre, np.ones((1, 1, 1)),
                                        np.zeros((4, 3)), 3)
    np.testing.assert_allclose(h[0, 0, 0], hb, rtol=1e-15)
    assert hd == 5


@pytest.mark.parametrize("seed", [51, 52])
def test_draft_tree_commit_equals_target_commit(seed):
    # replaying the accepted path's log = the target's selective recompute of that path
    g = np.random.default_rng(seed)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, n=16)
    _, log = _all_levels(prm, parent, xBC, dt, h0, ring, head)
    lay = oracle.tree_layout(parent)
    deepest = int(np.argmax(lay["depth"]))
    for path in ([0], lay["path"][deepest], lay["path"][len(parent) - 1]):
        h, r, hd = oracle.draft_tree_commit(prm["A_log"], parent, path, log, xBC, h0, ring, head)
        h_ref, r_ref, hd_ref = oracle.commit(prm, parent, path, xBC, dt, h0, ring, head)
        np.testing.assert_allclose(h, h_ref, rtol=1e-13, atol=1e-15)
        np.testing.assert_array_equal(r, r_ref)
        assert hd == hd_ref


def test_draft_tree_commit_on_a_chain_equals_replay():
    g = np.random.default_rng(61)
    H, P, N, R, head, T = 2, 3, 4, 20, 5, 12
    prm = rand_params(H, P, N, g)
    conv_dim = H * P + 2 * N
    xs, dts = g.normal(0, 1, (T, conv_dim)), g.normal(0, 0.5, (T, H))
    h0, ring = g.normal(0, 0.1, (H, P, N)), g.normal(0, 1, (R, conv_dim))
    parent = np.arange(-1, T - 1)
    _, log = _all_levels(prm, parent, xs, dts, h0, ring, head)
    for k in (1, 5, T):
        h, _, hd = oracle.draft_tree_commit(prm["A_log"], parent, list(range(k)), log, xs, h0, ring, head)
        h_ref, hd_ref = oracle.replay(prm["A_log"], [log[t] for t in range(T)], k, h0, head)
        np.testing.assert_array_equal(h, h_ref)
        assert hd == hd_ref


def test_draft_tree_edges():
    g = np.random.default_rng(71)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, n=9)
    lay = oracle.tree_layout(parent)
    ys, rows = oracle.draft_tree_level(prm, parent, max(lay["depth"]) + 1, xBC, dt, h0, ring, head, {})
    assert ys == {} and rows == {}  # a level below the deepest node has no nodes
    with pytest.raises(ValueError):
        oracle.draft_tree_commit(prm["A_log"], parent, [1], {}, xBC, h0, ring, head)  # not from the root
    with pytest.raises(KeyError):  # a level before its ancestors were drafted
        oracle.draft_tree_level(prm, parent, 1, xBC, dt, h0, ring, head, {})


# ---- planted mistakes ----
_orig_level = so.draft_tree_level
_orig_commit = so.draft_tree_commit


def _level_newest_first(params, parent, level, xBC, dt, h_ckpt, ring, head, log):
    lay = so.tree_layout(parent)
    H, P, N = h_ckpt.shape
    A = -np.exp(np.asarray(params["A_log"], np.float64))
    ys, rows = {}, {}
    for v in range(lay["n"]):
        if lay["depth"][v] != level:
            continue
        post = so.conv_silu(so.node_window(lay, v, xBC, ring, head), params["conv_w"], params["conv_b"])
        x, B, C = so.split_xbc(post, H, P, N)
        delta = so.softplus(dt[v] + params["dt_bias"])
        h = np.array(h_ckpt, np.float64)
        for m in lay["path"][v][:-1][::-1]:
            dm, Bm, xm = log[m]
            h = so.ssm_step(h, dm, A, xm.reshape(H, P), Bm)
        h = so.ssm_step(h, delta, A, x, B)
        ys[v] = so.ssm_out(h, C, params["D"], x).reshape(H * P)
        rows[v] = (delta, B, x.reshape(H * P))
    return ys, rows


def _level_own_update_dropped(params, parent, level, xBC, dt, h_ckpt, ring, head, log):
    ys, rows = _orig_level(params, parent, level, xBC, dt, h_ckpt, ring, head, log)
    H, P, N = h_ckpt.shape
    lay = so.tree_layout(parent)
    A = -np.exp(np.asarray(params["A_log"], np.float64))
    for v in ys:
        post = so.conv_silu(so.node_window(lay, v, xBC, ring, head), params["conv_w"], params["conv_b"])
        x, _, C = so.split_xbc(post, H, P, N)
        h = np.array(h_ckpt, np.float64)
        for m in lay["path"][v][:-1]:
            dm, Bm, xm = log[m]
            h = so.ssm_step(h, dm, A, xm.reshape(H, P), Bm)
        ys[v] = so.ssm_out(h, C, params["D"], x).reshape(H * P)
    return ys, rows


def _level_pre_conv_log(params, parent, level, xBC, dt, h_ckpt, ring, head, log):
    ys, rows = _orig_level(params, parent, level, xBC, dt, h_ckpt, ring, head, log)
    H, P, N = h_ckpt.shape
    d_inner = H * P
    return ys, {v: (r[0], np.asarray(xBC[v][d_inner:d_inner + N], np.float64), np.asarray(xBC[v][:d_inner], np.float64))
                for v, r in rows.items()}


def _commit_last_dropped(A_log, parent, path, log, xBC, h_ckpt, ring, head):
    h, r, _ = _orig_commit(A_log, parent, path[:-1] if len(path) > 1 else path, log, xBC, h_ckpt, ring, head)
    return h, r, head + len(path)


def _commit_rows_reversed(A_log, parent, path, log, xBC, h_ckpt, ring, head):
    h, _, hd = _orig_commit(A_log, parent, path, log, xBC, h_ckpt, ring, head)
    r = np.array(ring, copy=True)
    for j, m in enumerate(path[::-1]):
        r[(head + j) % ring.shape[0]] = xBC[m]
    return h, r, hd


MUTATIONS = {
    "ancestors applied newest first": ("draft_tree_level", _level_newest_first),
    "node's own update dropped": ("draft_tree_level", _level_own_update_dropped),
    "pre-conv values logged": ("draft_tree_level", _level_pre_conv_log),
    "last path node not committed": ("draft_tree_commit", _commit_last_dropped),
    "ring rows in reverse": ("draft_tree_commit", _commit_rows_reversed),
}

PINS = [test_draft_tree_chain_equals_draft_steps, lambda: test_draft_tree_levels_equal_tree_verify(41),
        test_draft_tree_closed_form_branching, lambda: test_draft_tree_commit_equals_target_commit(51),
        test_draft_tree_commit_on_a_chain_equals_replay]


def _any_pin_fails():
    for t in PINS:
        try:
            t()
        except AssertionError:
            return True
    return False


def test_unmutated_draft_tree_oracle_passes_every_pin():
    assert not _any_pin_fails()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_draft_tree_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(so, attr, fn)
    monkeypatch.setattr(oracle, attr, fn)
    with np.errstate(all="ignore"):
        assert _any_pin_fails(), f"no pin caught: {name}"
