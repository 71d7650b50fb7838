"""The seeded input module: bf16 rounding, determinism, tree shapes."""
import numpy as np
import torch

import oracle
from synth import (WORKLOADS, bf16_bits_to_f32, instance_state, node_inputs, to_bf16_bits, tree_parents,
                   tree_tokens, workload)


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    a = np.concatenate([g.standard_normal(100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 3.0e38, 1e-40, 1.00390625, 1.01171875], np.float32)])
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(to_bf16_bits(a), ref)
    np.testing.assert_array_equal(bf16_bits_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_instances_are_deterministic_and_independent():
    w = workload(2)
    a = node_inputs(w, 0, 5, 16)
    b = node_inputs(w, 0, 5, 16)
    c = node_inputs(w, 0, 6, 16)
    np.testing.assert_array_equal(a[0], b[0])
    assert not np.array_equal(a[0], c[0])
    h, ring, head = instance_state(w, 0, 5)
    assert h.shape == (80, 64, 128) and ring.shape == (w.ring_cap, 5376) and head == 3
    assert np.all(ring[3:] == 0)


def test_tree_shapes():
    assert WORKLOADS[0].n_nodes() == 15 and WORKLOADS[4].n_nodes(0) == 40 and WORKLOADS[4].n_nodes(1) == 256
    for cfg, tree in [(0, 0), (2, 0), (3, 0), (4, 0), (4, 1)]:
        w = workload(cfg)
        for seq in range(min(w.batch, 8)):
            par = tree_parents(w, seq, tree)
            lay = oracle.tree_layout(par)  # breadth-first, valid
            assert len(par) == w.n_nodes(tree)
            if w.trees[tree][0] == "random":
                assert max(lay["depth"]) <= w.trees[tree][3]
                assert max(len(c) for c in lay["children"]) <= w.trees[tree][2]
            tok, tgt = tree_tokens(w, seq, par, tree)
            for ch in lay["children"]:
                assert len({int(tok[c]) for c in ch}) == len(ch)  # distinct siblings


def test_acceptance_rate_is_near_p():
    w = workload(3)
    hits = tot = 0
    for seq in range(200):
        par = tree_parents(w, seq)
        tok, tgt = tree_tokens(w, seq, par)
        lay = oracle.tree_layout(par)
        for u, ch in enumerate(lay["children"]):
            if ch:
                tot += 1
                hits += int(any(tok[c] == tgt[u] for c in ch))
    assert abs(hits / tot - 0.8) < 0.05


def test_batch_parallel_is_batch():
    # the pool generator writes the same seeded streams into shared memory: identical arrays
    from synth import batch, batch_parallel, workload
    w = workload(4)
    a = batch_parallel(w, seqs=[0, 7, 63], layers=[0, 47], workers=2)
    b = batch(w, seqs=[0, 7, 63], layers=[0, 47])
    for k in ("parent", "tok", "tgt", "xBC", "dt", "h0", "ring", "ring_head"):
        assert np.array_equal(a[k], b[k]), k
    c = batch_parallel(w, seqs=[5, 6], layers=[3], tree=1, workers=2, with_state=False)
    d = batch(w, seqs=[5, 6], layers=[3], tree=1)
    assert "h0" not in c
    for k in ("parent", "tok", "tgt", "xBC", "dt"):
        assert np.array_equal(c[k], d[k]), k
