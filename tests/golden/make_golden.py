"""Writes tests/golden/oracle_tiny.json: a tiny tree-verify / accept / commit /
draft / replay case evaluated by the fp64 oracle.  It is a regression fixture
(the pages print no worked example): it freezes the oracle's current answers so
a later change to the oracle's arithmetic shows up as a diff.  Inputs come from
numpy's default_rng(2026); outputs come from oracle/ only.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402

H, P, N, R = 2, 3, 4, 8
PARENT = [-1, 0, 0, 1, 1, 2, 3]


def case():
    g = np.random.default_rng(2026)
    conv_dim = H * P + 2 * N
    prm = dict(conv_w=g.uniform(-0.5, 0.5, (conv_dim, 4)), conv_b=g.normal(0, 0.1, conv_dim),
               dt_bias=g.uniform(-6.9, -2.25, H), A_log=np.log(g.uniform(1, 16, H)), D=g.normal(1, 0.3, H))
    n = len(PARENT)
    inp = dict(xBC=g.normal(0, 1, (n, conv_dim)), dt=g.normal(0, 0.5, (n, H)), h0=g.normal(0, 0.1, (H, P, N)),
               ring=g.normal(0, 1, (R, conv_dim)), head=5, tok=[11, 3, 4, 8, 9, 1, 6], tgt=[4, 7, 1, 6, 2, 3, 5],
               draft_x=g.normal(0, 1, (4, conv_dim)), draft_dt=g.normal(0, 0.5, (4, H)))
    return prm, inp


def evaluate(prm, inp):
    y, st = oracle.verify(prm, PARENT, inp["xBC"], inp["dt"], inp["h0"], inp["ring"], inp["head"],
                          return_states=True)
    path, bonus = oracle.accept(PARENT, inp["tok"], inp["tgt"])
    hc, rc, hd = oracle.commit(prm, PARENT, path, inp["xBC"], inp["dt"], inp["h0"], inp["ring"], inp["head"])
    h, ring, log, ys = inp["h0"], inp["ring"], [], []
    for t in range(4):
        h, yt, ring, row = oracle.draft_step(prm, inp["draft_x"][t], inp["draft_dt"][t], h, ring, inp["head"], t)
        log.append(row)
        ys.append(yt)
    hr, hh = oracle.replay(prm["A_log"], log, 2, inp["h0"], inp["head"])
    return dict(y=y, path=path, bonus=bonus, h_commit=hc, head_commit=hd, draft_y=np.stack(ys), h_replay2=hr)


def _lists(d):
    return {k: (v.tolist() if isinstance(v, np.ndarray) else v) for k, v in d.items()}


if __name__ == "__main__":
    prm, inp = case()
    out = dict(parent=PARENT, shape=[H, P, N, R], params=_lists(prm), inputs=_lists(inp),
               expected=_lists(evaluate(prm, inp)))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)
