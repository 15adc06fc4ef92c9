"""Pins for the float64 CPU oracle, from closed forms, invariants, exact brute
force and library routines -- never from the oracle itself.

The oracle follows the residual loop and the decode graph of omnivoice.cpp
ARCHITECTURE.md, section "RVQ codec".  Each test below is chosen so that a
plausible slip in it fails: a transposed projection (planted recovery), a
flipped residual update (balanced-ternary digits), a wrong metric (nearest
neighbour against scipy), a wrong tie rule (duplicate rows and exact integer
instances), a dropped bias (bias tests), a wrong prefix (n_q tests).
"""

import itertools
from fractions import Fraction

import numpy as np
import pytest
from scipy.spatial.distance import cdist

import oracle
import rvq_inputs as ri


def _weights(w_in, codebook, w_out, b_in=None, b_out=None):
    f = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float32)
    return {"w_in": f(w_in), "codebook": f(codebook), "w_out": f(w_out), "b_in": f(b_in), "b_out": f(b_out)}


# ---------------------------------------------------------------------------
# closed form: balanced-ternary digit extraction
# ---------------------------------------------------------------------------

def test_balanced_ternary_digits_closed_form():
    """Stage q's codebook holds {-1,0,1}^2 * 3^(Q-1-q) in a 2-d code space that
    every stage projects onto the same two directions of a 4-d frame.  Greedy
    nearest-codeword RVQ must then return the balanced-ternary digits of the
    two coordinates, and the final residual is the part of x orthogonal to
    the code space.  Every value is exact in float32 and float64."""
    Q, d, D = 6, 2, 4
    U = np.array([[1, 1], [1, -1], [1, 1], [1, -1]], dtype=np.float64)   # orthogonal columns, |u|^2 = 4
    w_out = np.stack([U] * Q)                 # [Q][D][d]
    w_in = np.stack([U.T / 4.0] * Q)          # [Q][d][D]; w_in @ w_out = I
    digits = list(itertools.product((-1, 0, 1), repeat=2))    # k = 3*(a+1) + (b+1)
    cb = np.stack([np.array(digits, dtype=np.float64) * 3 ** (Q - 1 - q) for q in range(Q)])
    rng = np.random.default_rng(1)
    N = 300
    t = rng.integers(-1, 2, size=(N, Q, 2))
    v = (t * (3.0 ** (Q - 1 - np.arange(Q)))[None, :, None]).sum(axis=1)   # [N][2]
    x_perp = rng.integers(-4, 5, size=(N, 1)) * np.array([[0.5, 0.5, -0.5, -0.5]])
    x = v @ U.T + x_perp
    res = oracle.encode(_weights(w_in, cb, w_out), x)
    want = 3 * (t[:, :, 0] + 1) + (t[:, :, 1] + 1)
    assert np.array_equal(res["codes"], want)
    assert np.array_equal(res["residual"], x_perp)
    # decode of the digits rebuilds the in-space part exactly
    y, bad = oracle.decode(_weights(w_in, cb, w_out), want)
    assert bad == 0 and np.array_equal(y, v @ U.T)


def test_gap_and_distance_closed_form():
    """d = 1, codebook {0, 1, 3}, projected value 0.375: distances are
    0.140625, 0.390625, 6.890625, so code 0 and gap (d2-d1)/d2 = 0.64."""
    w_in = np.array([[[1.0]]])
    w_out = np.array([[[1.0]]])
    cb = np.array([[[0.0], [1.0], [3.0]]])
    res = oracle.encode(_weights(w_in, cb, w_out), np.array([[0.375]]))
    assert res["codes"][0, 0] == 0
    assert res["best_dist"][0, 0] == 0.140625
    assert res["gap"][0, 0] == pytest.approx(0.25 / 0.390625, rel=1e-15)
    assert res["residual"][0, 0] == 0.375
    # an exact tie: value 0.5 is equidistant from 0 and 1; lowest index wins, gap 0
    res = oracle.encode(_weights(w_in, cb, w_out), np.array([[0.5]]))
    assert res["codes"][0, 0] == 0 and res["gap"][0, 0] == 0.0


# ---------------------------------------------------------------------------
# planted codes with orthogonal projections
# ---------------------------------------------------------------------------

def _orthogonal(D, seed):
    rng = np.random.default_rng(seed)
    q, r = np.linalg.qr(rng.standard_normal((D, D)))
    return q * np.sign(np.diag(r))[None, :]


@pytest.mark.parametrize("with_bias", [False, True])
def test_planted_recovery_exact(with_bias):
    """W_out[q] = column block q of an orthogonal matrix, W_in[q] = W_out[q]^T,
    x = sum_q (W_out[q] C[q, c_q] + b_out[q]) with b_out in the orthogonal
    complement: then e_q = C[q, c_q] and the encoder must return c exactly,
    leave a (numerically) zero residual, and decode(c) must rebuild x."""
    D, Q, d, K, N = 256, 4, 32, 64, 200
    O = _orthogonal(D, 3)
    w_out = np.stack([O[:, q * d:(q + 1) * d] for q in range(Q)])
    w_in = np.transpose(w_out, (0, 2, 1)).copy()
    rng = np.random.default_rng(4)
    cb = rng.standard_normal((Q, K, d))
    b_out = np.stack([0.5 * O[:, Q * d + q] for q in range(Q)]) if with_bias else None
    W = _weights(w_in, cb, w_out, None, b_out)
    c = rng.integers(0, K, size=(N, Q))
    w64 = {k: (None if v is None else v.astype(np.float64)) for k, v in W.items()}
    x = np.zeros((N, D))
    for q in range(Q):
        x += w64["codebook"][q][c[:, q]] @ w64["w_out"][q].T
        if with_bias:
            x += w64["b_out"][q][None, :]
    x32 = x.astype(np.float32)
    res = oracle.encode(W, x32)
    assert np.array_equal(res["codes"], c)
    assert np.abs(res["residual"]).max() < 1e-5
    y, bad = oracle.decode(W, c)
    assert bad == 0
    assert np.abs(y - x).max() < 1e-12 * max(1.0, np.abs(x).max())


def test_planted_recovery_with_noise():
    """sigma = 0.05 noise is far below the codeword spacing (about 8 in 32-d),
    so recovery stays exact and the final residual is the noise's
    component outside... within the code space's complement bound."""
    D, Q, d, K, N = 256, 8, 32, 128, 300
    O = _orthogonal(D, 5)
    w_out = np.stack([O[:, q * d:(q + 1) * d] for q in range(Q)])
    w_in = np.transpose(w_out, (0, 2, 1)).copy()
    rng = np.random.default_rng(6)
    cb = rng.standard_normal((Q, K, d))
    W = _weights(w_in, cb, w_out)
    c = rng.integers(0, K, size=(N, Q))
    x = sum(W["codebook"][q].astype(np.float64)[c[:, q]] @ W["w_out"][q].astype(np.float64).T for q in range(Q))
    x = x + 0.05 * rng.standard_normal((N, D))
    res = oracle.encode(W, x.astype(np.float32))
    assert np.array_equal(res["codes"], c)


# ---------------------------------------------------------------------------
# special case: one stage with identity projections is nearest-neighbour search
# ---------------------------------------------------------------------------

def test_single_stage_identity_is_nearest_neighbour():
    rng = np.random.default_rng(7)
    D = d = 16
    K, N = 200, 500
    cb = rng.standard_normal((1, K, d)).astype(np.float32)
    x = rng.standard_normal((N, D)).astype(np.float32)
    eye = np.eye(D, dtype=np.float32)[None]
    res = oracle.encode(_weights(eye, cb, eye), x)
    dist = cdist(x.astype(np.float64), cb[0].astype(np.float64), "sqeuclidean")
    assert np.array_equal(res["codes"][:, 0], np.argmin(dist, axis=1))
    np.testing.assert_allclose(res["best_dist"][:, 0], dist.min(axis=1), rtol=1e-13)
    np.testing.assert_array_equal(res["residual"], x.astype(np.float64) - cb[0][res["codes"][:, 0]])


# ---------------------------------------------------------------------------
# exact brute force on tiny integer instances (ties included)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_integer_instances_argmin_certificate(seed):
    """Small integer weights keep every float64 operation exact.  For each
    frame the residual chain is rebuilt with Python integers from the oracle's
    codes, and each stage's code is checked against every entry: no entry is
    closer, and no lower-index entry is as close (lowest index wins ties).
    The reported gap must be the exact rational (d2 - d1) / d2."""
    rng = np.random.default_rng(100 + seed)
    D, d, K, Q, N = 5, 3, 6, 3, 60
    w_in = rng.integers(-2, 3, size=(Q, d, D))
    w_out = rng.integers(-2, 3, size=(Q, D, d))
    cb = rng.integers(-3, 4, size=(Q, K, d))
    b_in = rng.integers(-2, 3, size=(Q, d))
    b_out = rng.integers(-2, 3, size=(Q, D))
    x = rng.integers(-5, 6, size=(N, D))
    W = _weights(w_in, cb, w_out, b_in, b_out)
    res = oracle.encode(W, x)
    n_ties = 0
    for n in range(N):
        r = [int(v) for v in x[n]]
        for q in range(Q):
            e = [sum(int(w_in[q, j, i]) * r[i] for i in range(D)) + int(b_in[q, j]) for j in range(d)]
            dist = [sum((e[j] - int(cb[q, k, j])) ** 2 for j in range(d)) for k in range(K)]
            code = int(res["codes"][n, q])
            assert all(dist[code] <= dk for dk in dist)
            assert all(dist[code] < dist[k] for k in range(code))
            d1 = dist[code]
            d2 = min(dist[k] for k in range(K) if k != code)
            n_ties += d1 == d2
            want_gap = Fraction(d2 - d1, d2) if d2 > 0 else Fraction(0)
            assert res["gap"][n, q] == pytest.approx(float(want_gap), abs=1e-15)
            assert res["best_dist"][n, q] == d1
            out = [sum(int(w_out[q, i, j]) * int(cb[q, code, j]) for j in range(d)) + int(b_out[q, i]) for i in range(D)]
            r = [r[i] - out[i] for i in range(D)]
        assert [float(v) for v in r] == list(res["residual"][n])
    assert n_ties > 0  # the instances do exercise the tie rule


def test_duplicate_rows_take_lowest_index():
    rng = np.random.default_rng(9)
    K, d = 32, 8
    cb = rng.standard_normal((1, K, d)).astype(np.float32)
    x = rng.standard_normal((50, d)).astype(np.float32)
    eye = np.eye(d, dtype=np.float32)[None]
    base = oracle.encode(_weights(eye, cb, eye), x)["codes"][:, 0]
    # copy each frame's winner to a higher index and to a lower index
    for n in range(5):
        win = base[n]
        cb2 = cb.copy()
        hi = (win + 7) % K
        cb2[0, hi] = cb[0, win]
        r = oracle.encode(_weights(eye, cb2, eye), x[n:n + 1])
        assert r["codes"][0, 0] == min(win, hi) and r["gap"][0, 0] == 0.0


# ---------------------------------------------------------------------------
# decode: linearity, stage additivity, biases, bad codes
# ---------------------------------------------------------------------------

def _random_weights(D=48, d=8, K=40, Q=5, seed=11, bias=True):
    rng = np.random.default_rng(seed)
    return _weights(rng.standard_normal((Q, d, D)) / np.sqrt(D), rng.standard_normal((Q, K, d)),
                    rng.standard_normal((Q, D, d)) / np.sqrt(d),
                    0.1 * rng.standard_normal((Q, d)) if bias else None,
                    0.1 * rng.standard_normal((Q, D)) if bias else None)


def _stage(W, q):
    return {k: (None if v is None else v[q:q + 1]) for k, v in W.items()}


def test_decode_is_sum_of_single_stage_decodes():
    W = _random_weights()
    rng = np.random.default_rng(12)
    c = rng.integers(0, 40, size=(30, 5)).astype(np.int32)
    y, _ = oracle.decode(W, c)
    parts = sum(oracle.decode(_stage(W, q), c[:, q:q + 1])[0] for q in range(5))
    np.testing.assert_allclose(y, parts, rtol=0, atol=1e-13)
    # single stage closed form: w_out[q] @ codebook[q][c] + b_out[q]
    y0 = oracle.decode(_stage(W, 2), c[:, 2:3])[0]
    want = W["codebook"][2].astype(np.float64)[c[:, 2]] @ W["w_out"][2].astype(np.float64).T + W["b_out"][2]
    np.testing.assert_allclose(y0, want, rtol=1e-14, atol=1e-14)


def test_decode_scaling_bias_and_prefix():
    W = _random_weights()
    W0 = dict(W, b_in=None, b_out=None)
    rng = np.random.default_rng(13)
    c = rng.integers(0, 40, size=(30, 5)).astype(np.int32)
    y0, _ = oracle.decode(W0, c)
    W2 = dict(W0, w_out=W0["w_out"] * 2)
    assert np.array_equal(oracle.decode(W2, c)[0], 2 * y0)
    yb, _ = oracle.decode(W, c)
    np.testing.assert_allclose(yb - y0, np.broadcast_to(W["b_out"].astype(np.float64).sum(0), y0.shape), atol=1e-13)
    y3, _ = oracle.decode(W, c[:, :3], 3)
    y4, _ = oracle.decode(W, c[:, :4], 4)
    np.testing.assert_allclose(y4 - y3, oracle.decode(_stage(W, 3), c[:, 3:4])[0], atol=1e-13)


def test_decode_counts_and_skips_bad_codes():
    W = _random_weights()
    c = np.array([[1, 2, 3, 4, 5], [-1, 2, 40, 4, 1 << 30]], dtype=np.int32)
    y, bad = oracle.decode(W, c)
    assert bad == 3
    keep = oracle.decode(_stage(W, 1), c[1:, 1:2])[0] + oracle.decode(_stage(W, 3), c[1:, 3:4])[0]
    np.testing.assert_allclose(y[1:], keep, atol=1e-13)


# ---------------------------------------------------------------------------
# encode invariants
# ---------------------------------------------------------------------------

def test_greedy_prefix_property():
    w = ri.WORKLOADS[0]
    W = ri.make_weights(w, with_bias=True)
    x = ri.make_x(w, W, rows=np.arange(64))
    full = oracle.encode(W, x)
    for k in (1, 3, 7):
        part = oracle.encode(W, x, n_q=k)
        assert np.array_equal(part["codes"], full["codes"][:, :k])
        assert np.array_equal(part["gap"], full["gap"][:, :k])


def test_reconstruct_consistency():
    w = ri.WORKLOADS[0]
    W = ri.make_weights(w, with_bias=True)
    x = ri.make_x(w, W, rows=np.arange(64))
    r = oracle.reconstruct(W, x)
    err = np.abs(r["x_hat"] - (x.astype(np.float64) - r["residual"])).max()
    assert err <= 1e-12 * np.abs(x).max()


def test_batch_and_thread_invariance():
    w = ri.WORKLOADS[0]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)
    a = oracle.encode(W, x, threads=1)
    b = oracle.encode(W, x, threads=7)
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["residual"], b["residual"])
    for n in (0, 131, 249):
        s = oracle.encode(W, x[n:n + 1])
        assert np.array_equal(s["codes"][0], a["codes"][n])
        assert np.array_equal(s["gap"][0], a["gap"][n])


def test_input_bias_is_a_codebook_shift():
    """||e + b - c||^2 = ||e - (c - b)||^2: one stage with bias b_in equals one
    stage without it over the codebook shifted by -b_in (integers: exact)."""
    rng = np.random.default_rng(15)
    D, d, K = 12, 4, 25
    w_in = rng.integers(-2, 3, size=(1, d, D))
    w_out = rng.integers(-2, 3, size=(1, D, d))
    cb = rng.integers(-6, 7, size=(1, K, d))
    b = rng.integers(-3, 4, size=(1, d))
    x = rng.integers(-4, 5, size=(80, D))
    a = oracle.encode(_weights(w_in, cb, w_out, b_in=b), x)
    s = oracle.encode(_weights(w_in, cb - b[:, None, :], w_out), x)
    assert np.array_equal(a["codes"], s["codes"])
    assert np.array_equal(a["best_dist"], s["best_dist"])


def test_rejects_bad_arguments():
    W = _random_weights()
    with pytest.raises(ValueError):
        oracle.encode(W, np.zeros((2, 48), np.float32), n_q=6)
    with pytest.raises(ValueError):
        oracle.encode(W, np.zeros((2, 48), np.float32), n_q=0)


# ---------------------------------------------------------------------------
# the normalised ("cosine") metric of moss-tts.cpp AGENTS.md, gotcha 9:
# projection and codewords L2-normalised (eps 1e-12) before the argmin; the
# residual update and decode use the stored codeword
# ---------------------------------------------------------------------------

def _eye_weights(codebook, Q=1):
    cb = np.asarray(codebook, dtype=np.float64)
    if cb.ndim == 2:
        cb = cb[None]
    Q, K, d = cb.shape
    eye = np.stack([np.eye(d)] * Q)
    return _weights(eye, cb, eye)


def test_cosine_closed_form_2d():
    """e = (3, 4) normalises to (0.6, 0.8); the codebook {(1, 0), (0, 2), (0, 0)}
    normalises to {(1, 0), (0, 1), (0, 0)}.  Squared distances 0.8, 0.4, 1.0:
    code 1, best distance 0.4, gap (0.8 - 0.4) / 0.8 = 0.5, and the residual
    subtracts the stored codeword (0, 2), leaving (3, 2)."""
    W = _eye_weights([[1.0, 0.0], [0.0, 2.0], [0.0, 0.0]])
    res = oracle.encode(W, np.array([[3.0, 4.0]]), metric="cosine")
    assert res["codes"].tolist() == [[1]]
    assert abs(res["best_dist"][0, 0] - 0.4) <= 1e-15
    assert abs(res["gap"][0, 0] - 0.5) <= 1e-15
    assert np.array_equal(res["residual"], np.array([[3.0, 2.0]]))
    # the plain metric on the same frame: distances 20, 13, 25 -> code 1 as
    # well, best distance 13 (a mix-up of the two metrics shows in best_dist)
    res0 = oracle.encode(W, np.array([[3.0, 4.0]]))
    assert res0["codes"].tolist() == [[1]] and res0["best_dist"][0, 0] == 13.0


def test_cosine_eps_clamps_small_vectors():
    """A projection of norm t = 1e-13 < eps is divided by eps, not by its norm:
    (t, 0) -> (t/eps, 0) ~ (0.1, 0), squared distance to (1, 0) = (1 - t/eps)^2
    ~ 0.81 and to (0, 1) = (t/eps)^2 + 1; a zero codeword stays zero (distance
    (t/eps)^2 ~ 0.01).  t is the float32 value the oracle receives."""
    t = float(np.float32(1e-13))
    u = t / 1e-12
    W = _eye_weights([[1.0, 0.0], [0.0, 1.0]])
    res = oracle.encode(W, np.array([[t, 0.0]]), metric="cosine")
    assert res["codes"].tolist() == [[0]]
    assert abs(res["best_dist"][0, 0] - (1.0 - u) ** 2) <= 1e-15
    assert abs(u - 0.1) < 1e-8
    W0 = _eye_weights([[1.0, 0.0], [0.0, 0.0]])
    res = oracle.encode(W0, np.array([[t, 0.0]]), metric="cosine")
    assert res["codes"].tolist() == [[1]]
    assert abs(res["best_dist"][0, 0] - u * u) <= 1e-15


def test_cosine_single_stage_is_scipy_cosine_neighbour():
    """One stage with identity projections: the argmin of ||e/|e| - c/|c|||^2
    = 2 - 2 cos(e, c) is the nearest codeword under scipy's cosine distance,
    and the best squared distance is twice that distance."""
    rng = np.random.default_rng(11)
    d, K, N = 8, 200, 400
    cb = rng.standard_normal((K, d)).astype(np.float32).astype(np.float64)   # the values the oracle receives
    x = rng.standard_normal((N, d)).astype(np.float32).astype(np.float64)
    res = oracle.encode(_eye_weights(cb), x, metric="cosine")
    cd = cdist(x, cb, metric="cosine")
    srt = np.sort(cd, axis=1)
    clear = (srt[:, 1] - srt[:, 0]) > 1e-9
    assert clear.mean() > 0.99
    assert np.array_equal(res["codes"][clear, 0], np.argmin(cd, axis=1)[clear])
    assert np.allclose(res["best_dist"][:, 0], 2.0 * srt[:, 0], rtol=0, atol=1e-12)


def test_cosine_scale_invariance_of_one_stage():
    """With one stage and no input bias, scaling the frames by a positive
    factor or the codewords by positive factors changes no code."""
    rng = np.random.default_rng(12)
    Q, d, D, K, N = 1, 8, 24, 64, 300
    w_in = rng.standard_normal((Q, d, D)) / np.sqrt(D)
    w_out = rng.standard_normal((Q, D, d)) / np.sqrt(d)
    cb = rng.standard_normal((Q, K, d))
    x = rng.standard_normal((N, D))
    base = oracle.encode(_weights(w_in, cb, w_out), x, metric="cosine")["codes"]
    scaled_x = oracle.encode(_weights(w_in, cb, w_out), 8.0 * x, metric="cosine")["codes"]
    f = np.exp2(rng.integers(-3, 4, size=(Q, K, 1))).astype(np.float64)   # powers of two: exact
    scaled_cb = oracle.encode(_weights(w_in, cb * f, w_out), x, metric="cosine")["codes"]
    assert np.array_equal(base, scaled_x)
    assert np.array_equal(base, scaled_cb)
    # the plain metric is not scale invariant on the same data
    assert not np.array_equal(oracle.encode(_weights(w_in, cb * f, w_out), x)["codes"], base)


def test_cosine_planted_recovery_exact():
    """Stages project onto orthogonal 8-d blocks of a 32-d frame; x = sum_q
    w_out[q] c_q with codewords of varied lengths.  The normalised argmin
    must return every planted code, the residual (stored codewords
    subtracted) must vanish, and decode must rebuild x."""
    rng = np.random.default_rng(13)
    Q, d, K, N = 4, 8, 32, 200
    D = Q * d
    basis = np.linalg.qr(rng.standard_normal((D, D)))[0]
    w_out = np.stack([basis[:, q * d:(q + 1) * d] for q in range(Q)])       # [Q][D][d]
    w_in = np.transpose(w_out, (0, 2, 1))                                  # orthonormal: w_in[q] w_out[s] = delta
    cb = rng.standard_normal((Q, K, d)) * rng.uniform(0.5, 3.0, size=(Q, K, 1))
    c = rng.integers(0, K, size=(N, Q))
    x = sum(cb[q, c[:, q]] @ w_out[q].T for q in range(Q))
    W = _weights(w_in, cb, w_out)
    res = oracle.encode(W, x, metric="cosine")
    assert np.array_equal(res["codes"], c)
    assert np.abs(res["residual"]).max() < 1e-5   # float32 weights: exact up to their rounding
    y, _ = oracle.decode(W, res["codes"])
    assert np.abs(y - x).max() < 1e-5


# ---------------------------------------------------------------------------
# the Linear layers around the quantizer (omnivoice.cpp ARCHITECTURE.md,
# "Audio tokenizer"): fc before the residual loop, fc2 after the decoded sum.
# Integer weights and frames keep every product exact in float32 and float64.
# ---------------------------------------------------------------------------

def _int_rvq(rng, Q, d, D, K):
    w_in = rng.integers(-2, 3, size=(Q, d, D)).astype(np.float64)
    w_out = rng.integers(-2, 3, size=(Q, D, d)).astype(np.float64)
    cb = rng.integers(-4, 5, size=(Q, K, d)).astype(np.float64)
    return w_in, cb, w_out


def test_fc_maps_frames_before_the_loop():
    """With fc (a non-square, non-symmetric integer D x D_in matrix plus an
    integer bias) the codes, distances and final residual equal those of the
    plain loop run on fc(x) = fc_w x + fc_b, computed exactly here."""
    rng = np.random.default_rng(21)
    Q, d, D, D_in, K, N = 3, 3, 5, 7, 9, 200
    w_in, cb, w_out = _int_rvq(rng, Q, d, D, K)
    fc_w = rng.integers(-3, 4, size=(D, D_in)).astype(np.float64)
    fc_b = rng.integers(-5, 6, size=(D,)).astype(np.float64)
    x = rng.integers(-4, 5, size=(N, D_in)).astype(np.float64)
    xp = (x.astype(np.int64) @ fc_w.astype(np.int64).T + fc_b.astype(np.int64)).astype(np.float64)
    W = _weights(w_in, cb, w_out)
    Wfc = dict(W, fc_w=np.float32(fc_w), fc_b=np.float32(fc_b))
    a = oracle.encode(Wfc, x)
    b = oracle.encode(W, xp)
    assert np.array_equal(a["codes"], b["codes"])
    assert np.array_equal(a["best_dist"], b["best_dist"])
    assert np.array_equal(a["residual"], b["residual"])
    # and fc changes the result (the test is not vacuous)
    assert not np.array_equal(oracle.encode(W, x[:, :D])["codes"], a["codes"])


def test_fc2_maps_the_decoded_sum():
    """decode with fc2 = fc2_w (sum of the stage outputs) + fc2_b, the bias
    once (three stages), against fc2 applied exactly to the plain decode."""
    rng = np.random.default_rng(22)
    Q, d, D, D_out, K, N = 3, 2, 6, 4, 7, 150
    w_in, cb, w_out = _int_rvq(rng, Q, d, D, K)
    b_out = rng.integers(-3, 4, size=(Q, D)).astype(np.float64)
    fc2_w = rng.integers(-3, 4, size=(D_out, D)).astype(np.float64)
    fc2_b = rng.integers(-5, 6, size=(D_out,)).astype(np.float64)
    codes = rng.integers(0, K, size=(N, Q)).astype(np.int32)
    W = _weights(w_in, cb, w_out, b_out=b_out)
    y, bad = oracle.decode(W, codes)
    y2, bad2 = oracle.decode(dict(W, fc2_w=np.float32(fc2_w), fc2_b=np.float32(fc2_b)), codes)
    want = (y.astype(np.int64) @ fc2_w.astype(np.int64).T + fc2_b.astype(np.int64)).astype(np.float64)
    assert bad == bad2 == 0
    assert y2.shape == (N, D_out)
    assert np.array_equal(y2, want)
