"""The oracle reproduces its frozen fixtures in tests/golden/ (drift guard)."""

import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_frozen_fixtures():
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        data = json.load(f)
    assert len(data["cases"]) >= 4
    for c in data["cases"]:
        G = np.array([float(v) for v in c["input"]]).reshape(c["H"], c["W"])
        want = np.array([float(v) for v in c["output"]]).reshape(c["H"], c["W"])
        got = oracle.tiled_ns(G, c["T"], c["K"], tuple(c["coeffs"]), c["norm"], c["eps"])
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-13, err_msg=c["name"])
