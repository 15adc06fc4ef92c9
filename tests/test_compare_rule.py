"""The near-tie comparison rule itself (host logic, no GPU)."""
import numpy as np

from rvq_compare import compare_codes


def test_clear_mismatch_fails_and_near_tie_diverges():
    ref = np.array([[1, 2, 3, 4], [5, 6, 7, 8], [1, 1, 1, 1]])
    gap = np.array([[0.1, 0.1, 0.1, 0.1], [0.1, 1e-6, 0.1, 0.1], [0.1, 0.1, 0.0, 0.2]])
    gpu = ref.copy()
    gpu[1, 1] = 9      # near tie at stage 1: frame diverges, stages 2 and 3 excluded
    gpu[1, 3] = 0      # ...so this later mismatch is not counted
    gpu[2, 2] = 4      # exact tie (gap 0) broken differently: diverged
    r = compare_codes(gpu, ref, gap)
    assert r["n_fail"] == 0 and r["n_diverged_frames"] == 2 and r["n_excluded_stages"] == 3
    gpu[0, 2] = 0      # a clear decision that differs
    r = compare_codes(gpu, ref, gap)
    assert r["n_fail"] == 1 and r["fails"][0][:2] == (0, 2)


def test_equal_codes_pass():
    ref = np.arange(12).reshape(3, 4)
    r = compare_codes(ref.copy(), ref, np.zeros((3, 4)))
    assert r["n_fail"] == 0 and r["n_equal"] == 12 and r["n_near_ties"] == 12
