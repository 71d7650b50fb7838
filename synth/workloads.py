"""Workload presets and seeded generators.

Every random draw comes from its own ``numpy.random.Generator(PCG64(SeedSequence(
[0x5EED, workload, seq, layer, stream])))``, so any single instance can be
regenerated on its own (a sampled parity check at full size does not need the
whole batch on the host).

Value recipe (the Mamba2 shapes named by the workloads; the pages print no
worked example, so these distributions stand in for trained weights and for
the MT-Bench / GSM-8K / HumanEval prompts the SpecMamba page measures on):

* pre-conv ``xBC`` rows ~ N(0, 1) and raw ``dt`` ~ N(0, 0.5) (second argument
  read as the standard deviation), both rounded to bf16 (round-to-nearest-even);
* ``dt_bias`` = inverse softplus of u, u log-uniform on [1e-3, 0.1];
* ``A_log`` = log U[1, 16] per head, ``D`` = 1, conv weights U(-0.5, 0.5),
  conv bias 0 -- all fp32;
* committed state ``h0`` ~ N(0, 0.1) fp32; the conv ring holds the 3 positions
  before the root, ~ N(0, 1) bf16, and the ring head counts those 3 positions;
* token ids uniform in [0, 50280); sibling draft tokens are distinct; a node
  with children gets a target token equal to one child's draft token with
  probability p (child chosen uniformly), else an id that matches no child;
  a leaf gets a uniform id.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Iterable, Sequence

import numpy as np

VOCAB = 50280
SEED_ROOT = 0x5EED

# random streams (last SeedSequence word)
_ST_PARAMS = 1
_ST_STATE = 2
_ST_NODES = 3
_ST_TREE = 4
_ST_TOKENS = 5
_ST_DRAFT = 6
_ST_REPLAY = 7


@dataclass(frozen=True)
class Shape:
    """Mamba2 SSM-layer shape: H heads x P headdim, d_state N, conv width W, ngroups 1."""

    H: int
    P: int = 64
    N: int = 128
    W: int = 4

    @property
    def d_inner(self) -> int:
        return self.H * self.P

    @property
    def conv_dim(self) -> int:
        return self.d_inner + 2 * self.N


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    shape: Shape
    n_layers: int
    batch: int
    trees: tuple  # tree specs, see tree_parents()
    p_accept: float = 0.8
    draft_steps: int = 0
    ring_cap: int = 20  # rows per instance in the conv ring (>= 3 + draft_steps)

    @property
    def n_inst(self) -> int:
        return self.n_layers * self.batch

    def n_nodes(self, tree: int = 0) -> int:
        spec = self.trees[tree]
        if spec[0] == "full":
            b, d = spec[1], spec[2]
            return sum(b**i for i in range(d + 1))
        return spec[1]


WORKLOADS = {
    0: Workload(0, "tiny tree verify, Mamba2-130M layer shape, 1 layer, batch 1, 15-node full binary tree",
                Shape(H=24), n_layers=1, batch=1, trees=(("full", 2, 3),)),
    1: Workload(1, "draft chain decode, Mamba2-370M shape, 48 layers, batch 1, 16 draft steps + replay",
                Shape(H=32), n_layers=48, batch=1, trees=(), draft_steps=16),
    2: Workload(2, "target tree verify, Mamba2-2.7B shape, 64 layers, batch 1, 16-node random tree",
                Shape(H=80), n_layers=64, batch=1, trees=(("random", 16, 3, 4),)),
    3: Workload(3, "batched target verify, Mamba2-2.7B shape, 64 layers, batch 16, 16-node random trees",
                Shape(H=80), n_layers=64, batch=16, trees=(("random", 16, 3, 4),)),
    4: Workload(4, "stress, Mamba2-780M shape, 48 layers, batch 64, 40-node ternary tree + 256-node chain",
                Shape(H=48), n_layers=48, batch=64, trees=(("full", 3, 3), ("chain", 256)),
                p_accept=0.9, draft_steps=16),
    5: Workload(5, "draft tree, Mamba2-370M shape, 48 layers, batch 1, 16-node random tree drafted level by level",
                Shape(H=32), n_layers=48, batch=1, trees=(("random", 16, 3, 4),)),
}


def workload(index: int) -> Workload:
    return WORKLOADS[int(index)]


def _rng(w: Workload, seq: int, layer: int, stream: int, extra: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence([SEED_ROOT, w.index, int(seq), int(layer), stream, int(extra)])
    return np.random.Generator(np.random.PCG64(ss))


# ---------------------------------------------------------------------------
# bf16 bit patterns (inputs are generated in fp32 and rounded once; both sides
# then read the identical 16-bit patterns)
# ---------------------------------------------------------------------------
def to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16, nearest-even; returns uint16 bit patterns.  In 32-bit
    arithmetic: for every finite or infinite input the sum stays below 2^32 (the largest
    finite pattern 0xFF7FFFFF plus 0x8000 is 0xFF807FFF)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    u = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# per-layer parameters (shared by every sequence)
# ---------------------------------------------------------------------------
def layer_params(w: Workload, layers: Iterable[int] | None = None) -> dict:
    layers = list(range(w.n_layers)) if layers is None else [int(l) for l in layers]
    s = w.shape
    conv_w = np.empty((len(layers), s.conv_dim, s.W), np.float32)
    conv_b = np.zeros((len(layers), s.conv_dim), np.float32)
    dt_bias = np.empty((len(layers), s.H), np.float32)
    A_log = np.empty((len(layers), s.H), np.float32)
    D = np.ones((len(layers), s.H), np.float32)
    for i, l in enumerate(layers):
        g = _rng(w, 0, l, _ST_PARAMS)
        conv_w[i] = g.uniform(-0.5, 0.5, size=(s.conv_dim, s.W))
        u = np.exp(g.uniform(np.log(1e-3), np.log(0.1), size=s.H))
        dt_bias[i] = np.log(np.expm1(u))  # inverse of softplus, so softplus(dt_bias) = u
        A_log[i] = np.log(g.uniform(1.0, 16.0, size=s.H))
    return dict(conv_w=conv_w, conv_b=conv_b, dt_bias=dt_bias, A_log=A_log, D=D)


# ---------------------------------------------------------------------------
# trees and tokens
# ---------------------------------------------------------------------------
def _full_tree(branching: int, depth: int) -> np.ndarray:
    parent = [-1]
    level = [0]
    for _ in range(depth):
        nxt = []
        for u in level:
            for _ in range(branching):
                parent.append(u)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.asarray(parent, np.int32)


def _random_tree(g: np.random.Generator, n: int, max_branches: int, max_depth: int) -> np.ndarray:
    par, depth, nchild = [-1], [0], [0]
    for i in range(1, n):
        cands = [u for u in range(i) if depth[u] < max_depth and nchild[u] < max_branches]
        u = cands[int(g.integers(len(cands)))]
        par.append(u)
        depth.append(depth[u] + 1)
        nchild[u] += 1
        nchild.append(0)
    # relabel breadth-first: by (depth, new id of parent, creation order)
    new = {0: 0}
    order = [0]
    for d in range(1, max(depth) + 1):
        lvl = sorted((i for i in range(n) if depth[i] == d), key=lambda i: (new[par[i]], i))
        for i in lvl:
            new[i] = len(order)
            order.append(i)
    out = np.empty(n, np.int32)
    for old in order:
        out[new[old]] = -1 if par[old] < 0 else new[par[old]]
    return out


def tree_parents(w: Workload, seq: int, tree: int = 0) -> np.ndarray:
    """parent[] of one sequence's draft tree, breadth-first, parent[0] = -1."""
    spec = w.trees[tree]
    if spec[0] == "full":
        return _full_tree(spec[1], spec[2])
    if spec[0] == "chain":
        return np.arange(-1, spec[1] - 1, dtype=np.int32)
    if spec[0] == "random":
        return _random_tree(_rng(w, seq, 0, _ST_TREE, tree), spec[1], spec[2], spec[3])
    raise ValueError(spec)


def tree_tokens(w: Workload, seq: int, parent: Sequence[int], tree: int = 0):
    """(tok, tgt): draft token of every node and the target's greedy token after every node."""
    g = _rng(w, seq, 0, _ST_TOKENS, tree)
    n = len(parent)
    children = [[] for _ in range(n)]
    for v in range(1, n):
        children[int(parent[v])].append(v)
    tok = np.zeros(n, np.int32)
    tok[0] = g.integers(VOCAB)
    for u in range(n):
        used = set()
        for c in children[u]:
            t = int(g.integers(VOCAB))
            while t in used:
                t = int(g.integers(VOCAB))
            used.add(t)
            tok[c] = t
    tgt = np.zeros(n, np.int32)
    for u in range(n):
        ch = children[u]
        if ch and g.random() < w.p_accept:
            tgt[u] = tok[ch[int(g.integers(len(ch)))]]
        else:
            avoid = {int(tok[c]) for c in ch}
            t = int(g.integers(VOCAB))
            while t in avoid:
                t = int(g.integers(VOCAB))
            tgt[u] = t
    return tok, tgt


# ---------------------------------------------------------------------------
# per-instance tensors
# ---------------------------------------------------------------------------
def instance_state(w: Workload, seq: int, layer: int):
    """(h0 fp32 [H][P][N], ring bf16-bits [ring_cap][conv_dim], ring_head)."""
    s = w.shape
    g = _rng(w, seq, layer, _ST_STATE)
    h0 = g.standard_normal((s.H, s.P, s.N), dtype=np.float32)
    h0 *= np.float32(0.1)
    ring = np.zeros((w.ring_cap, s.conv_dim), np.uint16)
    ring[:3] = to_bf16_bits(g.standard_normal((3, s.conv_dim), dtype=np.float32))
    return h0, ring, 3


def node_inputs(w: Workload, seq: int, layer: int, n_nodes: int, tree: int = 0):
    """(xBC bf16-bits [n][conv_dim] pre-conv, dt bf16-bits [n][H] raw)."""
    s = w.shape
    g = _rng(w, seq, layer, _ST_NODES, tree)
    xbc = to_bf16_bits(g.standard_normal((n_nodes, s.conv_dim), dtype=np.float32))
    dt = g.standard_normal((n_nodes, s.H), dtype=np.float32)
    dt *= np.float32(0.5)
    return xbc, to_bf16_bits(dt)


def draft_inputs(w: Workload, seq: int, layer: int, steps: int | None = None):
    """(xBC bf16-bits [steps][conv_dim], dt bf16-bits [steps][H]) for the draft's chain."""
    s = w.shape
    steps = w.draft_steps if steps is None else steps
    g = _rng(w, seq, layer, _ST_DRAFT)
    xbc = to_bf16_bits(g.standard_normal((steps, s.conv_dim), dtype=np.float32))
    dt = g.standard_normal((steps, s.H), dtype=np.float32)
    dt *= np.float32(0.5)
    return xbc, to_bf16_bits(dt)


def replay_k(w: Workload, seq: int) -> int:
    """Accepted draft position k in [0, draft_steps] for one sequence."""
    return int(_rng(w, seq, 0, _ST_REPLAY).integers(0, w.draft_steps + 1))


# ---------------------------------------------------------------------------
# stacked batches (instance = seq * n_layers + layer, sequence-major)
# ---------------------------------------------------------------------------
def batch(w: Workload, seqs: Sequence[int] | None = None, layers: Sequence[int] | None = None,
          tree: int = 0) -> dict:
    """All tensors of a tree-verify step for the chosen sequences x layers."""
    seqs = list(range(w.batch)) if seqs is None else [int(x) for x in seqs]
    layers = list(range(w.n_layers)) if layers is None else [int(x) for x in layers]
    s = w.shape
    n = w.n_nodes(tree)
    S, L = len(seqs), len(layers)
    out = dict(
        seqs=np.asarray(seqs, np.int32), layers=np.asarray(layers, np.int32), n_nodes=n,
        parent=np.empty((S, n), np.int32), tok=np.empty((S, n), np.int32), tgt=np.empty((S, n), np.int32),
        xBC=np.empty((S, L, n, s.conv_dim), np.uint16), dt=np.empty((S, L, n, s.H), np.uint16),
        h0=np.empty((S, L, s.H, s.P, s.N), np.float32),
        ring=np.empty((S, L, w.ring_cap, s.conv_dim), np.uint16), ring_head=np.empty((S, L), np.int32),
    )
    for i, q in enumerate(seqs):
        par = tree_parents(w, q, tree)
        out["parent"][i] = par
        out["tok"][i], out["tgt"][i] = tree_tokens(w, q, par, tree)
        for j, l in enumerate(layers):
            out["h0"][i, j], out["ring"][i, j], out["ring_head"][i, j] = instance_state(w, q, l)
            out["xBC"][i, j], out["dt"][i, j] = node_inputs(w, q, l, n, tree)
    out["params"] = layer_params(w, layers)
    return out


def _fill_part(args):
    """Worker of batch_parallel: generate sequences seqs[lo:hi] into the shared arrays."""
    from multiprocessing import shared_memory
    w, seqs, layers, tree, lo, hi, specs, with_state = args
    blocks = {k: shared_memory.SharedMemory(name=name) for k, (name, _, _) in specs.items()}
    try:
        arr = {k: np.ndarray(shape, dtype, buffer=blocks[k].buf) for k, (_, shape, dtype) in specs.items()}
        small = []
        for i in range(lo, hi):
            q = seqs[i]
            par = tree_parents(w, q, tree)
            tok, tgt = tree_tokens(w, q, par, tree)
            small.append((par, tok, tgt))
            for j, l in enumerate(layers):
                if with_state:
                    arr["h0"][i, j], arr["ring"][i, j], arr["ring_head"][i, j] = instance_state(w, q, l)
                arr["xBC"][i, j], arr["dt"][i, j] = node_inputs(w, q, l, len(par), tree)
        del arr
        return lo, small
    finally:
        for b in blocks.values():
            b.close()


def batch_parallel(w: Workload, seqs: Sequence[int] | None = None, layers: Sequence[int] | None = None,
                   tree: int = 0, workers: int | None = None, with_state: bool = True) -> dict:
    """batch() with the sequences generated by a spawn pool of `workers` processes that
    write straight into shared memory; every instance comes from its own seeded
    streams, so the result is identical to batch().  with_state=False leaves out h0,
    ring and ring_head (a second tree of the same instances reuses the first's)."""
    import multiprocessing as mp
    import os
    from concurrent.futures import ProcessPoolExecutor
    from multiprocessing import shared_memory
    seqs = list(range(w.batch)) if seqs is None else [int(x) for x in seqs]
    layers = list(range(w.n_layers)) if layers is None else [int(x) for x in layers]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    workers = max(1, min(workers or cores, len(seqs)))
    s = w.shape
    n = w.n_nodes(tree)
    S, L = len(seqs), len(layers)
    shapes = {"xBC": ((S, L, n, s.conv_dim), np.uint16), "dt": ((S, L, n, s.H), np.uint16)}
    if with_state:
        shapes.update({"h0": ((S, L, s.H, s.P, s.N), np.float32), "ring": ((S, L, w.ring_cap, s.conv_dim), np.uint16),
                       "ring_head": ((S, L), np.int32)})
    blocks = {k: shared_memory.SharedMemory(create=True, size=max(1, int(np.prod(sh)) * np.dtype(dt).itemsize))
              for k, (sh, dt) in shapes.items()}
    try:
        specs = {k: (blocks[k].name, sh, dt) for k, (sh, dt) in shapes.items()}
        if with_state:  # ring rows past the three generated ones start at zero, as in batch()
            np.ndarray(shapes["ring"][0], np.uint16, buffer=blocks["ring"].buf).fill(0)
        per = (S + workers - 1) // workers
        tasks = [(w, seqs, layers, tree, lo, min(S, lo + per), specs, with_state) for lo in range(0, S, per)]
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            with ProcessPoolExecutor(len(tasks), mp_context=mp.get_context("spawn")) as ex:
                parts = list(ex.map(_fill_part, tasks))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k)
                else:
                    os.environ[k] = v
        out = dict(seqs=np.asarray(seqs, np.int32), layers=np.asarray(layers, np.int32), n_nodes=n,
                   parent=np.empty((S, n), np.int32), tok=np.empty((S, n), np.int32), tgt=np.empty((S, n), np.int32))
        for lo, small in parts:
            for k, (par, tok, tgt) in enumerate(small):
                out["parent"][lo + k], out["tok"][lo + k], out["tgt"][lo + k] = par, tok, tgt
        for k, (sh, dt) in shapes.items():
            out[k] = np.ndarray(sh, dt, buffer=blocks[k].buf).copy()
    finally:
        for b in blocks.values():
            b.close()
            b.unlink()
    out["params"] = layer_params(w, layers)
    return out


def draft_batch(w: Workload, seqs: Sequence[int] | None = None, layers: Sequence[int] | None = None,
                steps: int | None = None) -> dict:
    """All tensors of a draft round (chain of draft steps, then replay) for seqs x layers."""
    seqs = list(range(w.batch)) if seqs is None else [int(x) for x in seqs]
    layers = list(range(w.n_layers)) if layers is None else [int(x) for x in layers]
    steps = w.draft_steps if steps is None else steps
    s = w.shape
    S, L = len(seqs), len(layers)
    out = dict(
        seqs=np.asarray(seqs, np.int32), layers=np.asarray(layers, np.int32), steps=steps,
        xBC=np.empty((steps, S, L, s.conv_dim), np.uint16), dt=np.empty((steps, S, L, s.H), np.uint16),
        h0=np.empty((S, L, s.H, s.P, s.N), np.float32),
        ring=np.empty((S, L, w.ring_cap, s.conv_dim), np.uint16), ring_head=np.empty((S, L), np.int32),
        k=np.asarray([replay_k(w, q) for q in seqs], np.int32),
    )
    for i, q in enumerate(seqs):
        for j, l in enumerate(layers):
            out["h0"][i, j], out["ring"][i, j], out["ring_head"][i, j] = instance_state(w, q, l)
            xb, d = draft_inputs(w, q, l, steps)
            out["xBC"][:, i, j] = xb
            out["dt"][:, i, j] = d
    out["params"] = layer_params(w, layers)
    return out
