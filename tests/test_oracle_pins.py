"""Pins for the fp64 oracle, each against something other than the oracle itself.

* softplus / SiLU against numpy.logaddexp and scipy.special.expit;
* the causal tree conv on a chain against numpy.convolve (a textbook routine);
* hand-derived closed forms for H = P = N = 1 (decay 1/2, Δ = ln 2), on a chain
  and on a branching tree, with distinct x, B, C and D so a swapped or dropped
  term changes the number;
* an independent evaluation of the whole tree by the dual (quadratic) form of
  the linear recurrence, with its own conv via numpy.convolve over each path;
* Δ -> 0 leaves the state exactly unchanged;
* tree = separate linear runs along every root-to-node path ("100%
  verification accuracy", SpecMamba page §3.2);
* accept walk against brute-force enumeration of every root-to-node path;
* replay from the (Δ, B, x) log reproduces the stored draft state (§3.1);
* commit equals the verified state of the accepted node.
"""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle
from synth import Workload, Shape, tree_parents, tree_tokens

RNG = np.random.default_rng(20261202)


# ---------------------------------------------------------------------------
# small random problems
# ---------------------------------------------------------------------------
def rand_params(H, P, N, g):
    conv_dim = H * P + 2 * N
    return dict(conv_w=g.uniform(-0.5, 0.5, (conv_dim, 4)), conv_b=g.normal(0, 0.1, conv_dim),
                dt_bias=np.log(np.expm1(np.exp(g.uniform(np.log(1e-3), np.log(0.1), H)))),
                A_log=np.log(g.uniform(1, 16, H)), D=g.normal(1, 0.3, H))


def rand_tree(g, n, max_branches=3, max_depth=4):
    w = Workload(99, "pin", Shape(H=1), 1, 1, trees=(("random", n, max_branches, max_depth),))
    # reuse the generator's tree sampler with a per-call seed
    return tree_parents(w, int(g.integers(1 << 30)))


def rand_problem(g, H=3, P=4, N=5, n=12, R=8, head=11, parent=None):
    prm = rand_params(H, P, N, g)
    parent = rand_tree(g, n) if parent is None else np.asarray(parent)
    n = len(parent)
    conv_dim = H * P + 2 * N
    xBC = g.normal(0, 1, (n, conv_dim))
    dt = g.normal(0, 0.5, (n, H))
    h0 = g.normal(0, 0.1, (H, P, N))
    ring = g.normal(0, 1, (R, conv_dim))
    return prm, parent, xBC, dt, h0, ring, head


def path_of(parent, v):
    p = [v]
    while parent[p[-1]] >= 0:
        p.append(int(parent[p[-1]]))
    return p[::-1]


# ---------------------------------------------------------------------------
# scalar maps
# ---------------------------------------------------------------------------
def test_softplus_matches_logaddexp():
    v = np.concatenate([np.linspace(-60, 30, 2001), [-7.0, -2.25, 0.0, 1e-8]])
    np.testing.assert_allclose(oracle.softplus(v), np.logaddexp(0.0, v), rtol=1e-14, atol=0)


def test_silu_matches_expit():
    v = np.linspace(-40, 40, 1601)
    np.testing.assert_allclose(oracle.silu(v), v * expit(v), rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0


# ---------------------------------------------------------------------------
# conv on a chain against numpy.convolve
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("head", [3, 9, 13])
def test_chain_conv_matches_numpy_convolve(head):
    g = np.random.default_rng(head)
    C, n, R = 7, 9, 8
    w = g.uniform(-0.5, 0.5, (C, 4))  # deliberately asymmetric taps
    b = g.normal(0, 0.2, C)
    xBC = g.normal(0, 1, (n, C))
    ring = g.normal(0, 1, (R, C))
    parent = np.arange(-1, n - 1)
    lay = oracle.tree_layout(parent)
    prior = np.stack([ring[(head - 3) % R], ring[(head - 2) % R], ring[(head - 1) % R]])
    seq = np.concatenate([prior, xBC])  # positions head-3 .. head+n-1
    for c in range(C):
        ref = np.convolve(seq[:, c], w[c][::-1], mode="valid")  # ref[t] = sum_k w[c,k] seq[t+k]
        ref = (b[c] + ref) * expit(b[c] + ref)
        got = [oracle.conv_silu(oracle.node_window(lay, v, xBC, ring, head), w, b)[c] for v in range(n)]
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------
# closed forms, H = P = N = 1
# ---------------------------------------------------------------------------
def _scalar_params(D=0.25):
    # taps [0,0,0,1], bias 0: post = SiLU(pre) for x, B and C;
    # dt_bias = 0 with dt = 0 gives Δ = ln 2; A_log = 0 gives A = -1, decay = 1/2.
    w = np.zeros((3, 4))
    w[:, 3] = 1.0
    return dict(conv_w=w, conv_b=np.zeros(3), dt_bias=np.zeros(1), A_log=np.zeros(1), D=np.array([D]))


def _s(v):
    return v / (1.0 + math.exp(-v))


def _run_scalar(parent, pre):
    prm = _scalar_params()
    xBC = np.asarray(pre, np.float64)  # rows: [x_pre, B_pre, C_pre]
    dt = np.zeros((len(parent), 1))
    h0 = np.ones((1, 1, 1))
    ring = np.zeros((4, 3))
    y, st = oracle.verify(prm, parent, xBC, dt, h0, ring, 3, return_states=True)
    return y[:, 0], st[:, 0, 0, 0]


def test_closed_form_scalar_chain():
    ln2 = math.log(2.0)
    pre = [[1.0, 1.0, 2.0], [2.0, -1.0, 0.5], [-1.0, 3.0, 1.0]]
    y, h = _run_scalar([-1, 0, 1], pre)
    x = [_s(r[0]) for r in pre]
    B = [_s(r[1]) for r in pre]
    C = [_s(r[2]) for r in pre]
    h1 = 0.5 * 1.0 + ln2 * x[0] * B[0]
    h2 = 0.5 * h1 + ln2 * x[1] * B[1]
    h3 = 0.5 * h2 + ln2 * x[2] * B[2]
    np.testing.assert_allclose(h, [h1, h2, h3], rtol=1e-15)
    np.testing.assert_allclose(y, [C[0] * h1 + 0.25 * x[0], C[1] * h2 + 0.25 * x[1], C[2] * h3 + 0.25 * x[2]],
                               rtol=1e-15)
    # hand-computed values for x = SiLU(1), SiLU(2), B = C = D = 1 (state path only)
    hh1 = 0.5 + ln2 * 0.7310585786300049
    assert abs(hh1 - 1.006731192601549) < 1e-15
    assert abs(0.5 * hh1 + ln2 * 1.7615941559557646 - 1.7244096187923894) < 1e-15


def test_closed_form_scalar_branching():
    # root with two children: each child starts from h_root, not from its sibling
    ln2 = math.log(2.0)
    pre = [[1.0, 1.0, 2.0], [2.0, -1.0, 0.5], [-1.0, 3.0, 1.0]]
    y, h = _run_scalar([-1, 0, 0], pre)
    x = [_s(r[0]) for r in pre]
    B = [_s(r[1]) for r in pre]
    C = [_s(r[2]) for r in pre]
    hr = 0.5 + ln2 * x[0] * B[0]
    ha = 0.5 * hr + ln2 * x[1] * B[1]
    hb = 0.5 * hr + ln2 * x[2] * B[2]
    np.testing.assert_allclose(h, [hr, ha, hb], rtol=1e-15)
    np.testing.assert_allclose(y, [C[0] * hr + 0.25 * x[0], C[1] * ha + 0.25 * x[1], C[2] * hb + 0.25 * x[2]],
                               rtol=1e-15)


def test_closed_form_pure_decay():
    # x = SiLU(0) = 0 removes the input term: h_v = 2^-(depth+1) * h0 exactly
    parent = [-1, 0, 0, 1, 3]
    y, h = _run_scalar(parent, [[0.0, 1.0, 1.0]] * 5)
    depth = np.array([0, 1, 1, 2, 3])
    np.testing.assert_array_equal(h, 0.5 ** (depth + 1))
    np.testing.assert_allclose(y, _s(1.0) * 0.5 ** (depth + 1), rtol=1e-15)


# ---------------------------------------------------------------------------
# independent dual-form evaluation
# ---------------------------------------------------------------------------
def dual_form(prm, parent, xBC, dt, h0, ring, head):
    """y_v = e^{S_v} C_v.h0 + sum_{m in path(v)} e^{S_v - S_m} Δ_m (C_v.B_m) x_m + D x_v,
    S_v = sum_{m in path(v)} Δ_m A; conv by numpy.convolve over ring rows + path rows."""
    H, P, N = h0.shape
    d_inner = H * P
    n = len(parent)
    R = ring.shape[0]
    A = -np.exp(prm["A_log"])
    y = np.zeros((n, H, P))
    hs = np.zeros((n, H, P, N))
    for v in range(n):
        path = path_of(parent, v)
        seq = np.concatenate([np.stack([ring[(head - 3 + i) % R] for i in range(3)]), xBC[path]])
        pre = np.stack([np.convolve(seq[:, c], prm["conv_w"][c][::-1], mode="valid")
                        for c in range(seq.shape[1])], axis=1) + prm["conv_b"]
        post = pre * expit(pre)  # [len(path)][conv_dim]
        xs = post[:, :d_inner].reshape(len(path), H, P)
        Bs = post[:, d_inner:d_inner + N]
        Cv = post[-1, d_inner + N:]
        dl = np.logaddexp(0.0, dt[path] + prm["dt_bias"])  # [len][H]
        S = np.cumsum(dl * A, axis=0)  # [len][H]
        Sv = S[-1]
        acc = np.exp(Sv)[:, None] * np.einsum("hpn,n->hp", h0, Cv)
        hv = np.exp(Sv)[:, None, None] * h0
        for j in range(len(path)):
            wgt = np.exp(Sv - S[j]) * dl[j]  # [H]
            acc += wgt[:, None] * (Cv @ Bs[j]) * xs[j]
            hv += wgt[:, None, None] * xs[j][:, :, None] * Bs[j][None, None, :]
        y[v] = acc + prm["D"][:, None] * xs[-1]
        hs[v] = hv
    return y.reshape(n, d_inner), hs


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_tree_matches_dual_form(seed):
    g = np.random.default_rng(seed)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, H=3, P=4, N=5, n=14)
    y, st = oracle.verify(prm, parent, xBC, dt, h0, ring, head, return_states=True)
    yd, hd = dual_form(prm, parent, xBC, dt, h0, ring, head)
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(st, hd, rtol=1e-12, atol=1e-13)


def test_chain_matches_dual_form_long():
    g = np.random.default_rng(7)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, H=2, P=3, N=4, parent=np.arange(-1, 40))
    y = oracle.verify(prm, parent, xBC, dt, h0, ring, head)
    yd, _ = dual_form(prm, parent, xBC, dt, h0, ring, head)
    np.testing.assert_allclose(y, yd, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def test_delta_to_zero_keeps_state():
    g = np.random.default_rng(11)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g)
    dt[:] = -1.0e4  # softplus -> exactly 0: decay 1, no input
    y, st = oracle.verify(prm, parent, xBC, dt, h0, ring, head, return_states=True)
    for v in range(len(parent)):
        np.testing.assert_array_equal(st[v], h0)
    # y = C_v.h0 + D x_v with post-conv C, x from the pinned conv
    lay = oracle.tree_layout(parent)
    H, P, N = h0.shape
    for v in range(len(parent)):
        post = oracle.conv_silu(oracle.node_window(lay, v, xBC, ring, head), prm["conv_w"], prm["conv_b"])
        x, _, C = oracle.split_xbc(post, H, P, N)
        np.testing.assert_allclose(y[v], (np.einsum("hpn,n->hp", h0, C) + prm["D"][:, None] * x).ravel(),
                                   rtol=1e-14)
    hn, _, _ = oracle.commit(prm, parent, path_of(parent, len(parent) - 1), xBC, dt, h0, ring, head)
    np.testing.assert_array_equal(hn, h0)


def test_tree_equals_separate_linear_runs():
    g = np.random.default_rng(5)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, n=16)
    y = oracle.verify(prm, parent, xBC, dt, h0, ring, head)
    for v in range(len(parent)):
        p = path_of(parent, v)
        chain = np.arange(-1, len(p) - 1)
        yc = oracle.verify(prm, chain, xBC[p], dt[p], h0, ring, head)
        np.testing.assert_allclose(y[v], yc[-1], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------------------
# accept walk against brute force
# ---------------------------------------------------------------------------
def brute_force_accept(parent, tok, tgt):
    n = len(parent)
    best = 0
    for v in range(n):
        p = path_of(parent, v)
        if all(tok[c] == tgt[u] for u, c in zip(p, p[1:])) and len(p) > len(path_of(parent, best)):
            best = v
    return path_of(parent, best), int(tgt[best])


@pytest.mark.parametrize("seed", range(40))
def test_accept_matches_brute_force(seed):
    for p_acc, spec in [(0.8, ("random", 16, 3, 4)), (0.9, ("full", 3, 3)), (0.95, ("chain", 40)),
                        (0.8, ("full", 2, 3))]:
        w = Workload(98, "acc", Shape(H=1), 1, 1, trees=(spec,), p_accept=p_acc)
        parent = tree_parents(w, seed)
        tok, tgt = tree_tokens(w, seed, parent)
        assert oracle.accept(parent, tok, tgt) == brute_force_accept(parent, tok, tgt)


def test_accept_tie_break_lowest_index():
    # two siblings carry the same draft token; the walk takes the earlier one
    parent = [-1, 0, 0, 1, 2]
    tok = [7, 5, 5, 9, 9]
    tgt = [5, 9, 9, 1, 2]
    assert oracle.accept(parent, tok, tgt) == ([0, 1, 3], 1)
    assert oracle.accept(parent, tok, [4, 0, 0, 0, 0]) == ([0], 4)


# ---------------------------------------------------------------------------
# layout
# ---------------------------------------------------------------------------
def test_layout_hand_example():
    lay = oracle.tree_layout([-1, 0, 0, 1, 1, 2, 3])
    assert lay["depth"] == [0, 1, 1, 2, 2, 2, 3]
    assert lay["children"] == [[1, 2], [3, 4], [5], [6], [], [], []]
    assert lay["path"][6] == [0, 1, 3, 6]
    assert lay["taps"][0] == [-1, -2, -3]
    assert lay["taps"][2] == [0, -1, -2]
    assert lay["taps"][3] == [1, 0, -1]
    assert lay["taps"][6] == [3, 1, 0]


@pytest.mark.parametrize("bad", [[], [0], [-1, 1], [-1, 0, 2], [-1, 0, 1, 0], [-1, -1]])
def test_layout_rejects_bad_trees(bad):
    with pytest.raises(oracle.BadTree):
        oracle.tree_layout(bad)


# ---------------------------------------------------------------------------
# commit, draft, replay
# ---------------------------------------------------------------------------
def test_commit_equals_verified_node_state_and_appends_rows():
    g = np.random.default_rng(3)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, n=16, R=9, head=7)
    _, st = oracle.verify(prm, parent, xBC, dt, h0, ring, head, return_states=True)
    for v in range(len(parent)):
        p = path_of(parent, v)
        hn, rn, hd = oracle.commit(prm, parent, p, xBC, dt, h0, ring, head)
        np.testing.assert_array_equal(hn, st[v])
        assert hd == head + len(p)
        for j, m in enumerate(p):
            np.testing.assert_array_equal(rn[(head + j) % 9], xBC[m])


def test_commit_rejects_non_paths():
    g = np.random.default_rng(4)
    prm, parent, xBC, dt, h0, ring, head = rand_problem(g, parent=[-1, 0, 0, 1])
    with pytest.raises(ValueError):
        oracle.commit(prm, parent, [0, 2, 3], xBC, dt, h0, ring, head)
    with pytest.raises(ValueError):
        oracle.commit(prm, parent, [1, 3], xBC, dt, h0, ring, head)


def _draft_run(g, steps=16, H=2, P=3, N=4, R=20, head=3):
    prm = rand_params(H, P, N, g)
    conv_dim = H * P + 2 * N
    xs = g.normal(0, 1, (steps, conv_dim))
    dts = g.normal(0, 0.5, (steps, H))
    h = g.normal(0, 0.1, (H, P, N))
    ring = g.normal(0, 1, (R, conv_dim))
    states, ys, log = [h], [], []
    r = ring
    for t in range(steps):
        h, y, r, row = oracle.draft_step(prm, xs[t], dts[t], h, r, head, t)
        states.append(h)
        ys.append(y)
        log.append(row)
    return prm, xs, dts, ring, head, states, ys, log, r


def test_replay_reproduces_draft_states():
    g = np.random.default_rng(9)
    prm, xs, dts, ring, head, states, ys, log, _ = _draft_run(g)
    for k in range(17):
        h, hd = oracle.replay(prm["A_log"], log, k, states[0], head)
        np.testing.assert_array_equal(h, states[k])
        assert hd == head + k


def test_draft_chain_equals_chain_verify():
    # sixteen one-node draft steps = one 16-node chain verified from the same state
    g = np.random.default_rng(10)
    prm, xs, dts, ring, head, states, ys, log, ring_after = _draft_run(g)
    y = oracle.verify(prm, np.arange(-1, 15), xs, dts, states[0], ring, head)
    np.testing.assert_allclose(np.stack(ys), y, rtol=1e-13, atol=1e-14)
    for t in range(16):
        np.testing.assert_array_equal(ring_after[(head + t) % 20], xs[t])
