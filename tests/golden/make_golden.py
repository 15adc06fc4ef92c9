"""Writes oracle_tiny_regression.json: the float64 oracle's codes and relative
gaps for the first 24 frames of the 250-frame, D=256, Q=8, K=1024, d=64
workload (with small biases).  It calls only oracle/ and the input generator.
omnivoice.cpp ARCHITECTURE.md and moss-tts.cpp AGENTS.md print no worked
numeric RVQ example, so this fixture pins the oracle against unintended change
(and across CPU architectures), not against a printed example.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import rvq_inputs as ri  # noqa: E402


def main():
    w = ri.WORKLOAD_BY_NAME["tiny"]
    W = ri.make_weights(w, with_bias=True)
    x = ri.make_x(w, W, rows=np.arange(24))
    r = oracle.reconstruct(W, x)
    out = {
        "workload": w.describe() + " with_bias=True bias_scale=0.1",
        "rows": list(range(24)),
        "codes": r["codes"].tolist(),
        "gap": [[float(f"{g:.12e}") for g in row] for row in r["gap"]],
        "x_hat_row0_first8": [float(f"{v:.15e}") for v in r["x_hat"][0, :8]],
    }
    with open(os.path.join(HERE, "oracle_tiny_regression.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
