"""Comparison rules between the CUDA path and the float64 oracle.

Codes (near-tie rule): walk each frame's stages in order.  Where the oracle's
relative gap (d2 - d1) / d2 between its best and second-best squared distance
exceeds `thresh` (1e-5), the codes must be equal.  Where the gap is at most
`thresh` the decision is a near-tie that float32 arithmetic may break either
way: if the codes differ, the frame has diverged and its later stages (whose
residuals now differ) are not compared.

Floats: max |gpu - oracle| <= tol * RMS, with RMS over the whole input x of
the workload (or over the oracle's y for decode-only work).
"""

from __future__ import annotations

import numpy as np

GAP_THRESH = 1e-5
FLOAT_TOL = 1e-4


def compare_codes(gpu: np.ndarray, ref: np.ndarray, gap: np.ndarray, thresh: float = GAP_THRESH) -> dict:
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert gpu.shape == ref.shape == gap.shape, (gpu.shape, ref.shape, gap.shape)
    N, Q = ref.shape
    eq = gpu == ref
    clear = gap > thresh
    fails = []
    excluded = 0
    diverged = 0
    near_ties = int((~clear).sum())
    for n in np.nonzero(~eq.all(axis=1))[0]:
        for q in range(Q):
            if eq[n, q]:
                continue
            if clear[n, q]:
                fails.append((int(n), int(q), int(gpu[n, q]), int(ref[n, q]), float(gap[n, q])))
            else:
                diverged += 1
                excluded += Q - q - 1
            break
    return {"n_fail": len(fails), "fails": fails[:20], "n_diverged_frames": diverged,
            "n_excluded_stages": excluded, "n_near_ties": near_ties, "n_stages": N * Q,
            "n_equal": int(eq.sum())}


def max_abs_rel_to_rms(a: np.ndarray, b: np.ndarray, rms: float) -> float:
    return float(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)).max() / rms)


def rms(a: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a)))
