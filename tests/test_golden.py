"""The oracle still gives the answers frozen in tests/golden/oracle_tiny.json."""
import json
import os

import numpy as np

from tests.golden.make_golden import evaluate

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_tiny.json")


def test_oracle_matches_frozen_fixture():
    with open(HERE) as f:
        g = json.load(f)
    prm = {k: np.asarray(v) for k, v in g["params"].items()}
    inp = {k: (np.asarray(v) if isinstance(v, list) else v) for k, v in g["inputs"].items()}
    got = evaluate(prm, inp)
    for k, v in g["expected"].items():
        if isinstance(v, list) and k != "path":
            np.testing.assert_allclose(got[k], np.asarray(v), rtol=1e-13, atol=1e-15, err_msg=k)
        else:
            assert got[k] == v, k
