"""The seeded input generator: published splitmix64 values, backend agreement,
row independence and the workload distributions."""

import math

import numpy as np
import pytest
import torch

import rvq_inputs as ri


def test_splitmix64_published_sequence():
    # SplitMix64 seeded with 0 produces these first three words (the values
    # printed with Vigna's reference implementation, splitmix64.c).
    got = [int(v) for v in ri.words_np(0, np.arange(3, dtype=np.uint64))]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_numpy_and_torch_words_bit_identical():
    key = ri.stream_key(12345, ri.T_X)
    idx = np.arange(0, 200000, 7, dtype=np.uint64)
    a = ri.words_np(key, idx).view(np.int64)
    b = ri.words_torch(key, torch.from_numpy(idx.astype(np.int64))).numpy()
    assert np.array_equal(a, b)
    ca = ri.codes_np(key, idx, 1024)
    cb = ri.codes_torch(key, torch.from_numpy(idx.astype(np.int64)), 1024).numpy()
    assert np.array_equal(ca, cb)
    assert ca.min() >= 0 and ca.max() < 1024
    # K = 1024: multiply-shift equals the top ten bits of the word
    assert np.array_equal(ca, (ri.words_np(key, idx) >> np.uint64(54)).astype(np.int32))


def test_gaussians_agree_and_look_normal():
    key = ri.stream_key(7, ri.T_W_IN)
    idx = np.arange(400000, dtype=np.uint64)
    g = ri.gaussian_np(key, idx)
    gt = ri.gaussian_torch(key, torch.from_numpy(idx.astype(np.int64))).numpy()
    assert np.abs(g - gt).max() < 1e-12
    assert abs(g.mean()) < 0.01 and abs(g.std() - 1.0) < 0.01
    # fourth moment of N(0,1) is 3
    assert abs((g ** 4).mean() - 3.0) < 0.1


def test_rows_regenerate_independently():
    w = ri.WORKLOADS[1]
    W = ri.make_weights(w)
    rows = np.array([0, 5, 777, 11999])
    full = ri.make_x(w, W, rows=np.arange(0, 1000))
    part = ri.make_x(w, W, rows=rows[:3])
    assert np.array_equal(full[rows[:3]], part)
    c_all = ri.make_codes(w, np.arange(12000))
    assert np.array_equal(c_all[rows], ri.make_codes(w, rows))


def test_workload_shapes_and_scales():
    for w in ri.WORKLOADS:
        W = ri.make_weights(w)
        assert W["w_in"].shape == (w.Q, w.d, w.D)
        assert W["codebook"].shape == (w.Q, w.K, w.d)
        assert W["w_out"].shape == (w.Q, w.D, w.d)
        assert abs(W["w_in"].std() * math.sqrt(w.D) - 1.0) < 0.02
        assert abs(W["w_out"].std() * math.sqrt(w.d) - 1.0) < 0.02
        for q in (0, w.Q - 1):
            assert abs(W["codebook"][q].std() / (w.cb_decay ** q) - 1.0) < 0.02
    assert ri.WORKLOAD_BY_NAME["large_batch"].N == 192000
    assert ri.WORKLOAD_BY_NAME["moss_deep"].Q == 32


def test_torch_planted_frames_match_numpy():
    w = ri.WORKLOADS[4]
    W = ri.make_weights(w)
    x_np = ri.make_x(w, W, rows=np.arange(64))
    small = ri.Workload("probe", 1, 64, w.D, w.Q, w.K, w.d, "planted", sigma=w.sigma, seed=w.seed)
    x_t = ri.make_x_torch(small, ri.weights_to_torch(W, "cpu"), "cpu")
    # the float64 sums may differ in the last bit before rounding to float32
    assert np.abs(x_t.numpy() - x_np).max() <= 1e-6 * np.abs(x_np).max()


def test_decode_workload_has_no_frames():
    with pytest.raises(ValueError):
        ri.make_x(ri.WORKLOADS[2], ri.make_weights(ri.WORKLOADS[2]))
