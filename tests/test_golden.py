"""The oracle reproduces its stored regression fixture bit for bit."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_fixture(oracle):
    sys.path.insert(0, os.path.join(HERE, "golden"))
    import make_golden
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        fx = json.load(f)
    got = make_golden.compute()
    for k, v in got.items():
        want = np.array([float.fromhex(h) for h in fx[k]]).reshape(fx[k + "_shape"])
        assert np.array_equal(np.asarray(v), want), k
