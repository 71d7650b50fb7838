"""fp64 CPU oracle for SpecMamba-style tree verification on a Mamba2 SSM layer.

TEST INFRASTRUCTURE ONLY.  This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py`` and by
nothing else; the CUDA library and its Python binding never import, call or
link it, and it shares no code with them.  It is plain, slow and sequential on
purpose: every node is evaluated by walking its own root-to-node path from the
committed state, one recurrence step after another, in float64.

Sources (page title, then section):

* "FPGA 加速器完全拆解（二）…FlightLLM、CXL-SpecKV 与 LightMamba", section
  "为什么 Mamba 难加速": the input projection yields X, B, C, Δ, Z; X passes a
  conv1d and then the SSM, which keeps a hidden state h_t and emits Y; the SSM
  intermediates are the terms B̄X and Āh_{t-1}.  The same page's rotation
  section writes the update as Ā⊙h_{t-1} + B̄⊙X_t.  Read in the Mamba2 form:
  Ā = exp(Δ·A_h) (one scalar per head), B̄X = Δ·(x ⊗ B), Δ = softplus(dt +
  dt_bias), A_h = -exp(A_log_h), y = C·h + D·x.
* "FPGA加速Mamba推理：SpecMamba方案与优化实践":
  §1.2 draft model proposes, target model verifies in parallel;
  §2.1 a rejected draft forces the state back to the last accepted token;
  §3.1 the draft keeps only the light intermediates (Δ, A, B, X) for fast
  recovery; the target recomputes only the affected path;
  §3.2 the token tree is flattened breadth-first; a node's children are updated
  from the node's state, which is then released ("100% verification accuracy":
  the tree walk equals the separate linear runs it replaces);
  §5.2 tree_config (max_branches, max_depth).

Readings where the pages are silent (each one also listed in the design notes):
causal width-4 conv, taps oldest first, bias before SiLU, SiLU on all of
x|B|C; channel order [x | B | C]; head h owns x channels [h·P, (h+1)·P); B and C
shared by all heads (ngroups = 1); node 0 is the last committed token and is
processed with h_parent(root) = h0 and the conv ring holding the positions
before it; softplus is exact log1p(exp(v)); the greedy accept walk takes, at
each node, the first child in breadth-first order whose draft token equals the
target's token after that node; a draft tree is processed one depth level at a
time, each node from its branch state, which is the committed state followed by
its ancestors' logged (Δ, B, x) updates.

Every function here has a pin in ``tests/test_oracle_pins.py`` that checks it
against something other than itself (a library routine, a closed form, an
independent evaluation, brute force).
"""
from __future__ import annotations

import numpy as np

CONV_WIDTH = 4


class BadTree(ValueError):
    pass


# ---------------------------------------------------------------------------
# scalar maps
# ---------------------------------------------------------------------------
def softplus(v):
    """Δ = softplus(dt + dt_bias), exact, no threshold."""
    return np.log1p(np.exp(v))


def silu(v):
    return v / (1.0 + np.exp(-v))


# ---------------------------------------------------------------------------
# tree layout (breadth-first flattening with a parent[] array, §3.2)
# ---------------------------------------------------------------------------
def tree_layout(parent):
    """Validate a breadth-first parent[] and derive depth, children, paths, conv taps.

    parent[0] = -1 (the root, the last committed token); 0 <= parent[v] < v;
    breadth-first order means parent[] is non-decreasing, so each node's
    children occupy a contiguous, increasing index range.

    taps[v][d-1], d = 1..3: the source of the pre-conv row d positions before v
    on v's path: an ancestor's node index, or -(d - depth[v]) meaning ring
    position head - (d - depth[v]).
    """
    parent = [int(p) for p in np.asarray(parent).reshape(-1)]
    n = len(parent)
    if n < 1:
        raise BadTree("empty tree")
    if parent[0] != -1:
        raise BadTree("parent[0] must be -1")
    for v in range(1, n):
        if not (0 <= parent[v] < v):
            raise BadTree(f"parent[{v}]={parent[v]} is not an earlier node")
        if v >= 2 and parent[v] < parent[v - 1]:
            raise BadTree(f"parent[] not breadth-first at node {v}")
    depth = [0] * n
    children = [[] for _ in range(n)]
    for v in range(1, n):
        depth[v] = depth[parent[v]] + 1
        children[parent[v]].append(v)
    path = []
    for v in range(n):
        chain = [v]
        while parent[chain[-1]] >= 0:
            chain.append(parent[chain[-1]])
        path.append(chain[::-1])  # root first
    taps = []
    for v in range(n):
        row = []
        for d in range(1, CONV_WIDTH):
            if d <= depth[v]:
                row.append(path[v][depth[v] - d])
            else:
                row.append(-(d - depth[v]))
        taps.append(row)
    return dict(n=n, parent=parent, depth=depth, children=children, path=path, taps=taps)


# ---------------------------------------------------------------------------
# conv1d + SiLU on one node (causal, over the node's ancestor chain)
# ---------------------------------------------------------------------------
def _ring_row(ring, head, offset):
    """Ring row at absolute position head + offset (offset < 0 for committed rows)."""
    return ring[(head + offset) % ring.shape[0]]


def node_window(lay, v, xBC, ring, head):
    """The W pre-conv rows ending at node v, oldest first ([W][conv_dim])."""
    rows = []
    for d in range(CONV_WIDTH - 1, 0, -1):
        src = lay["taps"][v][d - 1]
        rows.append(xBC[src] if src >= 0 else _ring_row(ring, head, src))
    rows.append(xBC[v])
    return np.stack(rows)


def conv_silu(window, conv_w, conv_b):
    """post[c] = SiLU(b[c] + sum_k w[c][k] * window[k][c]), taps oldest first."""
    return silu(conv_b + np.einsum("ck,kc->c", conv_w, window))


def split_xbc(post, H, P, N):
    d_inner = H * P
    x = post[..., :d_inner].reshape(post.shape[:-1] + (H, P))
    B = post[..., d_inner:d_inner + N]
    C = post[..., d_inner + N:d_inner + 2 * N]
    return x, B, C


# ---------------------------------------------------------------------------
# one recurrence step and one output (Mamba2 form)
# ---------------------------------------------------------------------------
def ssm_step(h, delta, A, x, B):
    """h' = exp(Δ·A)·h + Δ·(x ⊗ B), per head.  h [H][P][N], delta/A [H], x [H][P], B [N]."""
    decay = np.exp(delta * A)
    return decay[:, None, None] * h + (delta[:, None] * x)[:, :, None] * B[None, None, :]


def ssm_out(h, C, D, x):
    """y[h][p] = sum_n C[n]·h[h][p][n] + D[h]·x[h][p]."""
    return np.einsum("hpn,n->hp", h, C) + D[:, None] * x


# ---------------------------------------------------------------------------
# the verify / accept / commit / draft / replay rows of the method
# ---------------------------------------------------------------------------
def verify(params, parent, xBC, dt, h0, ring, head, return_states=False):
    """Tree verification of one layer instance.

    params: conv_w [conv_dim][W], conv_b [conv_dim], dt_bias [H], A_log [H], D [H]
    xBC [n][conv_dim] pre-conv, dt [n][H] raw, h0 [H][P][N], ring [R][conv_dim].
    Returns y [n][H*P] (and the per-node states h_v [n][H][P][N] if asked).
    """
    H, P, N = h0.shape
    lay = tree_layout(parent)
    n = lay["n"]
    A = -np.exp(np.asarray(params["A_log"], np.float64))
    post = np.stack([conv_silu(node_window(lay, v, xBC, ring, head), params["conv_w"], params["conv_b"])
                     for v in range(n)])
    x, B, C = split_xbc(post, H, P, N)
    delta = softplus(dt + params["dt_bias"][None, :])
    y = np.empty((n, H, P))
    states = []
    for v in range(n):
        h = np.array(h0, np.float64)
        for m in lay["path"][v]:  # root .. v, sequentially
            h = ssm_step(h, delta[m], A, x[m], B[m])
        y[v] = ssm_out(h, C[v], params["D"], x[v])
        if return_states:
            states.append(h)
    y = y.reshape(n, H * P)
    return (y, np.stack(states)) if return_states else y


def accept(parent, tok, tgt):
    """Greedy accept walk: from the root, move to the first child (breadth-first
    order) whose draft token equals the target's token after the current node.
    Returns (path as node indices root..last, bonus token = tgt[last])."""
    lay = tree_layout(parent)
    cur = 0
    path = [0]
    while True:
        nxt = None
        for c in lay["children"][cur]:
            if int(tok[c]) == int(tgt[cur]):
                nxt = c
                break
        if nxt is None:
            break
        cur = nxt
        path.append(cur)
    return path, int(tgt[cur])


def commit(params, parent, path, xBC, dt, h0, ring, head):
    """Selective recompute of the accepted path only (§3.1): returns (h_new, ring_new, head_new).

    h_new is the state after the last path node; the path's pre-conv rows are
    appended to the conv ring at positions head .. head+len-1 and the head
    advances by len.
    """
    H, P, N = h0.shape
    lay = tree_layout(parent)
    path = [int(v) for v in path]
    if not path or path[0] != 0:
        raise ValueError("path must start at the root")
    for a, b in zip(path, path[1:]):
        if lay["parent"][b] != a:
            raise ValueError("path is not a root-to-node chain")
    A = -np.exp(np.asarray(params["A_log"], np.float64))
    h = np.array(h0, np.float64)
    for m in path:
        post = conv_silu(node_window(lay, m, xBC, ring, head), params["conv_w"], params["conv_b"])
        x, B, _ = split_xbc(post, H, P, N)
        delta = softplus(dt[m] + params["dt_bias"])
        h = ssm_step(h, delta, A, x, B)
    ring_new = np.array(ring, copy=True)
    R = ring.shape[0]
    for j, m in enumerate(path):
        ring_new[(head + j) % R] = xBC[m]
    return h, ring_new, head + len(path)


def draft_step(params, xBC_t, dt_t, h, ring, head, step):
    """One draft token (a one-node tree) at position head + step.

    Appends the pre-conv row to the ring at that position, updates h, returns
    (h_new, y [H*P], ring_new, log_row) with log_row = (Δ [H], B [N], x [H*P]),
    all post-conv: the light intermediates the draft keeps for recovery (§3.1).
    """
    H, P, N = h.shape
    R = ring.shape[0]
    pos = head + step
    window = np.stack([ring[(pos - 3) % R], ring[(pos - 2) % R], ring[(pos - 1) % R], xBC_t])
    ring_new = np.array(ring, copy=True)
    ring_new[pos % R] = xBC_t
    post = conv_silu(window, params["conv_w"], params["conv_b"])
    x, B, C = split_xbc(post, H, P, N)
    A = -np.exp(np.asarray(params["A_log"], np.float64))
    delta = softplus(dt_t + params["dt_bias"])
    h_new = ssm_step(np.asarray(h, np.float64), delta, A, x, B)
    y = ssm_out(h_new, C, params["D"], x).reshape(H * P)
    return h_new, y, ring_new, (delta, B, x.reshape(H * P))


def replay(A_log, log_rows, k, h_ckpt, head):
    """Recover the draft state at accepted position k from the checkpoint and the
    logged (Δ, B, x) rows, no conv and no input re-read: returns (h, head + k)."""
    H, P, N = h_ckpt.shape
    A = -np.exp(np.asarray(A_log, np.float64))
    h = np.array(h_ckpt, np.float64)
    for t in range(int(k)):
        delta, B, x = log_rows[t]
        h = ssm_step(h, np.asarray(delta), A, np.asarray(x).reshape(H, P), np.asarray(B))
    return h, head + int(k)


# ---------------------------------------------------------------------------
# draft-side tree drafting: branch states recovered from the light log
# ---------------------------------------------------------------------------
def draft_tree_level(params, parent, level, xBC, dt, h_ckpt, ring, head, log):
    """Process the nodes of depth `level` of a draft tree (the tree the target verifies next).

    The draft keeps one committed state h_ckpt and, for each node it has processed, only the
    light log row (Δ [H], B [N], x [H*P]), post-conv (SpecMamba page §3.1: the small
    intermediates recover the state).  A node's branch state is h_ckpt followed by the logged
    updates of its ancestors, root first, then the node's own update; it is never stored.
    xBC [n][conv_dim] holds the pre-conv rows of every node of depth <= level (a node's conv
    window runs over its ancestors, then the conv ring, as in verify); dt [n][H] raw.
    log: dict node -> (Δ, B, x) for every node of depth < level.
    Returns (ys, rows): dicts node -> y [H*P] and node -> (Δ, B, x) for the level's nodes.
    """
    H, P, N = h_ckpt.shape
    lay = tree_layout(parent)
    A = -np.exp(np.asarray(params["A_log"], np.float64))
    ys, rows = {}, {}
    for v in range(lay["n"]):
        if lay["depth"][v] != level:
            continue
        post = conv_silu(node_window(lay, v, xBC, ring, head), params["conv_w"], params["conv_b"])
        x, B, C = split_xbc(post, H, P, N)
        delta = softplus(dt[v] + params["dt_bias"])
        h = np.array(h_ckpt, np.float64)
        for m in lay["path"][v][:-1]:  # the ancestors' logged updates, root first
            dm, Bm, xm = log[m]
            h = ssm_step(h, np.asarray(dm), A, np.asarray(xm).reshape(H, P), np.asarray(Bm))
        h = ssm_step(h, delta, A, x, B)
        ys[v] = ssm_out(h, C, params["D"], x).reshape(H * P)
        rows[v] = (delta, B, x.reshape(H * P))
    return ys, rows


def draft_tree_commit(A_log, parent, path, log, xBC, h_ckpt, ring, head):
    """Move the draft's committed state along the path the target accepted (root..last,
    node indices): h <- the path's logged updates applied in order (no conv, no input
    re-read); the path's pre-conv rows go to ring positions head .. head+len-1 and the head
    advances by len.  Returns (h, ring_new, head_new)."""
    lay = tree_layout(parent)
    path = [int(v) for v in path]
    if not path or path[0] != 0:
        raise ValueError("path must start at the root")
    for a, b in zip(path, path[1:]):
        if lay["parent"][b] != a:
            raise ValueError("path is not a root-to-node chain")
    H, P, N = h_ckpt.shape
    A = -np.exp(np.asarray(A_log, np.float64))
    h = np.array(h_ckpt, np.float64)
    for m in path:
        dm, Bm, xm = log[m]
        h = ssm_step(h, np.asarray(dm), A, np.asarray(xm).reshape(H, P), np.asarray(Bm))
    ring_new = np.array(ring, copy=True)
    R = ring.shape[0]
    for j, m in enumerate(path):
        ring_new[(head + j) % R] = xBC[m]
    return h, ring_new, head + len(path)
