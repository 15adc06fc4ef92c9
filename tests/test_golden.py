"""The oracle reproduces its stored regression fixture (see tests/golden/README.md)."""
import json
import os

import numpy as np

import oracle
import rvq_inputs as ri

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny_regression.json")


def test_oracle_matches_regression_fixture():
    g = json.load(open(GOLDEN))
    w = ri.WORKLOAD_BY_NAME["tiny"]
    W = ri.make_weights(w, with_bias=True)
    x = ri.make_x(w, W, rows=np.array(g["rows"]))
    r = oracle.reconstruct(W, x)
    assert r["codes"].tolist() == g["codes"]
    np.testing.assert_allclose(r["gap"], np.array(g["gap"]), rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(r["x_hat"][0, :8], g["x_hat_row0_first8"], rtol=1e-13)
