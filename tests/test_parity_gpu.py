"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Codes follow the near-tie rule of rvq_compare; decoded and reconstructed
frames must lie within 1e-4 * RMS of the oracle's decode of the same codes.
Small workloads are compared on every frame; the full-size workloads run on
the GPU at full size (the benchmark's launch configuration) and are compared
on sampled frames, which the oracle computes frame by frame.
"""

import numpy as np
import pytest
import torch

import oracle
import rvq_inputs as ri
from rvq_compare import FLOAT_TOL, compare_codes, max_abs_rel_to_rms, rms

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import residual_vector_quantisation_gb300 as rq  # noqa: E402
from residual_vector_quantisation_gb300 import build as rqb  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rqb.build_library()
    rq.load_library()


def make_rvq(W, metric="l2"):
    t = ri.weights_to_torch(W, DEV)
    return rq.RVQ(t["w_in"], t["codebook"], t["w_out"], t["b_in"], t["b_out"], device=DEV, metric=metric,
                  fc_w=t.get("fc_w"), fc_b=t.get("fc_b"), fc2_w=t.get("fc2_w"), fc2_b=t.get("fc2_b"))


def check_encode(W, x, codes_gpu, rows=None, n_q=None, x_rms=None, x_hat_gpu=None, label="", metric="l2"):
    """Oracle-encode x[rows]; compare codes (near-tie rule) and x_hat."""
    rows = np.arange(x.shape[0]) if rows is None else rows
    xs = x[rows]
    ref = oracle.encode(W, xs, n_q, want_residual=False, metric=metric)
    cg = codes_gpu[rows]
    res = compare_codes(cg, ref["codes"], ref["gap"])
    assert res["n_fail"] == 0, f"{label}: code mismatches at clear decisions: {res}"
    # decode tolerance: oracle decode of the GPU's codes
    if x_hat_gpu is not None:
        y_ref, _ = oracle.decode(W, cg, cg.shape[1])
        r = x_rms if x_rms is not None else rms(x)
        err = max_abs_rel_to_rms(x_hat_gpu[rows], y_ref, r)
        assert err <= FLOAT_TOL, f"{label}: x_hat error {err:.3e} * RMS"
    return res


def run_small(W, x, n_q=None, label="", metric="l2"):
    rvq = make_rvq(W, metric)
    xt = torch.from_numpy(x).to(DEV)
    codes, x_hat = rvq.reconstruct(xt, n_q)
    codes_e = rvq.encode(xt, n_q)
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    assert np.array_equal(c, codes_e.cpu().numpy()), "encode and reconstruct disagree"
    res = check_encode(W, x, c, n_q=n_q, x_hat_gpu=x_hat.cpu().numpy(), label=label, metric=metric)
    # decode through the decode entry point too
    y = rvq.decode(codes).cpu().numpy()
    assert np.array_equal(y, x_hat.cpu().numpy())
    return res, c


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def test_tiny_workload_every_frame():
    w = ri.WORKLOAD_BY_NAME["tiny"]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)
    res, _ = run_small(W, x, label="tiny")
    assert res["n_equal"] >= 0.99 * res["n_stages"]


def test_omnivoice_workload_every_frame():
    w = ri.WORKLOAD_BY_NAME["omnivoice"]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)
    res, c = run_small(W, x, label="omnivoice")
    assert res["n_equal"] >= 0.99 * res["n_stages"]


def test_decode_only_workload_sampled():
    w = ri.WORKLOAD_BY_NAME["decode_only"]
    W = ri.make_weights(w)
    codes = ri.make_codes(w)
    rvq = make_rvq(W)
    ct = torch.from_numpy(codes).to(DEV)
    bad = torch.zeros(1, dtype=torch.int64, device=DEV)
    y = rvq.decode(ct, bad_codes=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0
    rows = np.random.default_rng(0).choice(w.N, 4096, replace=False)
    rows = np.concatenate([rows, [0, w.N - 1]])
    y_ref, _ = oracle.decode(W, codes[rows])
    yg = y[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    err = max_abs_rel_to_rms(yg, y_ref, rms(y_ref))
    assert err <= FLOAT_TOL, f"decode error {err:.3e} * RMS(y)"


def test_moss_deep_workload_sampled():
    w = ri.WORKLOAD_BY_NAME["moss_deep"]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)
    rvq = make_rvq(W)
    xt = torch.from_numpy(x).to(DEV)
    codes, x_hat = rvq.reconstruct(xt)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(1).choice(w.N, 2500, replace=False))
    res = check_encode(W, x, codes.cpu().numpy(), rows=rows, x_rms=rms(x), x_hat_gpu=x_hat.cpu().numpy(),
                       label="moss_deep")
    assert res["n_equal"] >= 0.97 * res["n_stages"]


def test_k4096_q10_workload_sampled():
    """Ten books of 4096 codewords: 32 distance chunks per stage and 45 G
    tables; 2000 sampled frames (including both ends) checked on the oracle."""
    w = ri.WORKLOAD_BY_NAME["k4096_q10"]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)
    rvq = make_rvq(W)
    xt = torch.from_numpy(x).to(DEV)
    codes, x_hat = rvq.reconstruct(xt)
    torch.cuda.synchronize()
    rows = np.sort(np.concatenate([np.random.default_rng(3).choice(w.N - 2, 1998, replace=False) + 1, [0, w.N - 1]]))
    res = check_encode(W, x, codes.cpu().numpy(), rows=rows, x_rms=rms(x), x_hat_gpu=x_hat.cpu().numpy(),
                       label="k4096_q10")
    assert res["n_equal"] >= 0.97 * res["n_stages"]


def test_large_batch_workload_full_size_sampled():
    """192 000 frames encoded and decoded on the GPU exactly as the benchmark
    does; 3000 sampled frames (including both ends) checked on the oracle."""
    w = ri.WORKLOAD_BY_NAME["large_batch"]
    W = ri.make_weights(w)
    Wt = ri.weights_to_torch(W, DEV)
    xt = ri.make_x_torch(w, Wt, DEV)
    rvq = make_rvq(W)
    codes = rvq.encode(xt)
    y = rvq.decode(codes)
    torch.cuda.synchronize()
    rows = np.sort(np.concatenate([np.random.default_rng(2).choice(w.N - 2, 2998, replace=False) + 1, [0, w.N - 1]]))
    ridx = torch.from_numpy(rows).to(DEV)
    x_s = xt[ridx].cpu().numpy()
    x_rms = float(torch.sqrt(torch.mean(xt.double() ** 2)).item())
    ref = oracle.encode(W, x_s, want_residual=False)
    cg = codes[ridx].cpu().numpy()
    res = compare_codes(cg, ref["codes"], ref["gap"])
    assert res["n_fail"] == 0, res
    y_ref, _ = oracle.decode(W, cg)
    err = max_abs_rel_to_rms(y[ridx].cpu().numpy(), y_ref, x_rms)
    assert err <= FLOAT_TOL, err


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def _small_weights(D=64, K=256, Q=4, seed=3, bias=False, decay=1.0, d=64):
    w = ri.Workload("edge", 1, 1, D, Q, K, d, "gauss", cb_decay=decay, seed=seed)
    return w, ri.make_weights(w, with_bias=bias, bias_scale=0.3)


@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 127, 129, 333])
@pytest.mark.parametrize("threshold", [0, None])
def test_ragged_frame_counts(N, threshold):
    """threshold 0: the tile kernels even for a single frame; None: the default
    split (small calls on the streaming kernel)."""
    w, W = _small_weights(D=128, K=256, Q=3, seed=10 + N)
    x = np.random.default_rng(N).standard_normal((N, 128)).astype(np.float32)
    prev = rq.rvq_set_stream_max_frames(-1 if threshold is None else threshold)
    try:
        run_small(W, x, label=f"N={N}")
    finally:
        rq.rvq_set_stream_max_frames(prev)


@pytest.mark.parametrize("D,K,Q", [(16, 128, 1), (48, 128, 2), (256, 384, 5), (2048, 256, 2),
                                   (64, 1152, 2), (96, 256, 20)])
def test_other_shapes(D, K, Q):
    w, W = _small_weights(D=D, K=K, Q=Q, seed=D + K + Q)
    x = np.random.default_rng(D).standard_normal((300, D)).astype(np.float32)
    run_small(W, x, label=f"D={D} K={K} Q={Q}")


@pytest.mark.parametrize("cta_rounds,extra,K,metric", [(1, 37, 256, "l2"), (3, 11, 512, "l2"), (1, 37, 384, "l2"),
                                                      (1, 37, 256, "cosine")])
def test_pair_and_split_items_mixed(cta_rounds, extra, K, metric):
    """Tile counts just above a multiple of the SM count: some CTAs get a
    second tile in an item and the rest a lone tile, which is split between
    the CTA's two pipelines when a stage has an even number of 128-codeword
    chunks (K = 256, 512) and run by one pipeline otherwise (K = 384).
    Every frame is checked."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = (cta_rounds * sms + extra) * 128 - 50
    w, W = _small_weights(D=64, K=K, Q=3, seed=K + extra)
    x = np.random.default_rng(K).standard_normal((N, 64)).astype(np.float32)
    run_small(W, x, label=f"tiles={cta_rounds}x{sms}+{extra} K={K} {metric}", metric=metric)


@pytest.mark.parametrize("K,Q,N,metric", [(4096, 3, 1, "l2"), (4096, 3, 1000, "l2"), (2048, 4, 4000, "cosine"),
                                          (4096, 2, 4900, "l2"), (1024, 5, 700, "l2"), (512, 3, 130, "cosine"),
                                          (1024, 3, 9000, "l2")])
def test_tiles_on_clusters(K, Q, N, metric):
    """Calls that fit one wave of 2-CTA clusters (and have a multiple of four
    128-codeword chunks a stage: K = 512 .. 4096) run each 128-frame tile on a
    cluster pair splitting every stage's codebook chunks and exchanging
    per-frame minima through distributed shared memory.  The tile kernels are
    forced (threshold 0); every frame is checked."""
    prev = rq.rvq_set_stream_max_frames(0)
    try:
        w, W = _small_weights(D=96, K=K, Q=Q, seed=K + N, bias=True)
        x = np.random.default_rng(K + N).standard_normal((N, 96)).astype(np.float32)
        run_small(W, x, label=f"K={K} Q={Q} N={N} {metric}", metric=metric)
    finally:
        rq.rvq_set_stream_max_frames(prev)


@pytest.mark.parametrize("K,Q,N,metric,d", [(512, 20, 3000, "l2", 64), (768, 20, 3000, "l2", 64),
                                            (768, 13, 2000, "cosine", 64), (1024, 17, 155 * 128 - 40, "l2", 64),
                                            (1024, 20, 3000, "cosine", 8), (512, 13, 160 * 128 - 7, "l2", 8)])
def test_deep_stacks_in_stage_blocks(K, Q, N, metric, d):
    """Stacks deeper than six stages whose terms outnumber a pipeline's
    chunks run as several search launches over blocks of stages, the terms of
    earlier blocks subtracted from the projections in between: on CTA pairs
    (K = 512), split items (K = 768; d = 8 at 3000 frames) and items of two
    (d = 64) or three (d = 8) tiles when the tiles outnumber the SMs, in
    blocks (d = 64: 20 = 5 + 5 + 5 + 5, 13 = 4 + 4 + 5, 17 = 5 + 6 + 6; d = 8:
    20 = 10 + 10 on split tiles, 13 = 3 + 3 + 3 + 4 on tiles of their own).
    The tile kernels are forced; every frame is checked."""
    prev = rq.rvq_set_stream_max_frames(0)
    try:
        w, W = _small_weights(D=64, K=K, Q=Q, seed=K + Q, bias=True, decay=0.9, d=d)
        x = np.random.default_rng(K + N).standard_normal((N, 64)).astype(np.float32)
        run_small(W, x, label=f"K={K} Q={Q} N={N} {metric}", metric=metric)
    finally:
        rq.rvq_set_stream_max_frames(prev)


@pytest.mark.parametrize("K,Q,d,prefixes", [(768, 13, 64, (8, 6)), (1024, 20, 8, (12, 10))])
def test_stage_blocks_keep_the_unblocked_sums(K, Q, d, prefixes):
    """The terms of earlier stage blocks are subtracted from P0 in the order
    the search continues in, so a blocked call reproduces the sums of an
    unblocked one bit for bit: the codes of every prefix depth equal the first
    stages of the full depth exactly, whether the prefix call is blocked the
    same way (d = 64: 13 = 4 + 4 + 5 and 8 = 4 + 4; d = 8: 20 = 10 + 10 and
    12 in one block) or not at all (d = 64, 6 stages; d = 8, the first 10)."""
    prev = rq.rvq_set_stream_max_frames(0)
    try:
        w, W = _small_weights(D=64, K=K, Q=Q, seed=K + Q + d, bias=True, decay=0.9, d=d)
        x = np.random.default_rng(Q).standard_normal((2000, 64)).astype(np.float32)
        rvq = make_rvq(W)
        xt = torch.from_numpy(x).to(DEV)
        full = rvq.encode(xt).cpu().numpy()
        for n_q in prefixes:
            part = rvq.encode(xt, n_q).cpu().numpy()
            assert np.array_equal(part, full[:, :n_q]), f"prefix {n_q} of {Q}"
        check_encode(W, x, full, label=f"K={K} Q={Q} d={d}")
    finally:
        rq.rvq_set_stream_max_frames(prev)


def test_prefix_depths_on_full_width_projection_items():
    """12 000 frames project as 256-frame x 256-column items, whose epilogue
    two crews of warps share (the first tile's steps and the second's); prefix
    depths of 3 and 5 stages leave the last column block part-filled (192 and
    320 columns): the codes equal the first stages of the full depth, and
    sampled frames of the full depth match the oracle."""
    w, W = _small_weights(D=1024, K=1024, Q=8, seed=31, bias=True)
    x = np.random.default_rng(31).standard_normal((12000, 1024)).astype(np.float32)
    rvq = make_rvq(W)
    xt = torch.from_numpy(x).to(DEV)
    full = rvq.encode(xt).cpu().numpy()
    for n_q in (3, 5):
        part = rvq.encode(xt, n_q).cpu().numpy()
        assert np.array_equal(part, full[:, :n_q]), f"prefix {n_q}"
    rows = np.concatenate([np.random.default_rng(1).choice(12000, 400, replace=False), [0, 255, 256, 11999]])
    check_encode(W, x, full, rows=rows, label="full-width items")


def test_biases_and_prefix_depths():
    w, W = _small_weights(D=256, K=512, Q=6, bias=True)
    x = np.random.default_rng(5).standard_normal((500, 256)).astype(np.float32)
    _, full = run_small(W, x, label="bias full")
    for n_q in (1, 2, 5):
        _, c = run_small(W, x, n_q=n_q, label=f"bias n_q={n_q}")
        assert np.array_equal(c, full[:, :n_q]), "prefix property"


def test_exact_ties_take_lowest_index():
    """Duplicated codebook rows give bit-identical distances; the lower index
    must win.  Frames sit right on duplicated entries."""
    D, K, Q = 64, 256, 2
    w, W = _small_weights(D=D, K=K, Q=Q, seed=77)
    W["w_in"] = np.stack([np.eye(64, dtype=np.float32)] * Q)
    W["w_out"] = np.stack([np.eye(64, dtype=np.float32)] * Q)
    rng = np.random.default_rng(8)
    for q in range(Q):
        for lo, hi in ((3, 200), (17, 18), (100, 255)):
            W["codebook"][q, hi] = W["codebook"][q, lo]
    picks = np.array([3, 200, 17, 18, 100, 255] * 20)
    x = W["codebook"][0][picks] + 0.01 * rng.standard_normal((len(picks), D)).astype(np.float32)
    x = x.astype(np.float32)
    rvq = make_rvq(W)
    codes = rvq.encode(torch.from_numpy(x).to(DEV)).cpu().numpy()
    ref = oracle.encode(W, x)
    assert np.array_equal(codes[:, 0], ref["codes"][:, 0])
    assert set(codes[:, 0].tolist()) <= {3, 17, 100}


def test_small_scratch_chunks_agree_bitwise():
    w = ri.WORKLOAD_BY_NAME["tiny"]
    W = ri.make_weights(w)
    x = torch.from_numpy(ri.make_x(w, W)).to(DEV)
    rvq = make_rvq(W)
    c_big = rvq.encode(x)
    small = torch.empty(rq.rvq_encode_min_scratch_bytes(rvq.dims, 8), dtype=torch.uint8, device=DEV)
    c_small = torch.empty_like(c_big)
    rq.rvq_encode(rvq.dims, rvq.tables, x, 8, c_small, small)
    torch.cuda.synchronize()
    assert torch.equal(c_big, c_small)


def test_decode_counts_bad_codes():
    w, W = _small_weights(D=64, K=128, Q=3)
    rvq = make_rvq(W)
    codes = np.array([[1, 2, 3], [-1, 5, 128], [127, 1 << 30, 0]], dtype=np.int32)
    bad = torch.zeros(1, dtype=torch.int64, device=DEV)
    y = rvq.decode(torch.from_numpy(codes).to(DEV), bad_codes=bad).cpu().numpy()
    assert int(bad.item()) == 3
    assert rq.rvq_read_error_count(bad) == 3  # the same counter through the C ABI reader
    y_ref, n_bad = oracle.decode(W, codes)
    assert n_bad == 3
    assert max_abs_rel_to_rms(y, y_ref, 1.0) <= 1e-5


def test_empty_batch_and_determinism():
    w = ri.WORKLOAD_BY_NAME["tiny"]
    W = ri.make_weights(w)
    rvq = make_rvq(W)
    empty = torch.empty((0, w.D), dtype=torch.float32, device=DEV)
    assert rvq.encode(empty).shape == (0, 8)
    x = torch.from_numpy(ri.make_x(w, W)).to(DEV)
    a = rvq.reconstruct(x)
    b = rvq.reconstruct(x)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_invalid_arguments_raise():
    w, W = _small_weights()
    rvq = make_rvq(W)
    x = torch.zeros((4, 64), device=DEV)
    with pytest.raises(rq.RVQError):
        rvq.encode(x, n_q=5)
    with pytest.raises(ValueError):
        rvq.encode(torch.zeros((4, 65), device=DEV))


# ---------------------------------------------------------------------------
# the normalised ("cosine") metric and the 8-dim code space
# ---------------------------------------------------------------------------

def test_moss_lfq_workload_every_frame():
    """32 books of 1024 entries in an 8-dim code space, argmin between
    L2-normalised vectors: all 12 000 frames checked on the oracle."""
    w = ri.WORKLOAD_BY_NAME["moss_lfq"]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)
    res, _ = run_small(W, x, label="moss_lfq", metric="cosine")
    assert res["n_equal"] >= 0.97 * res["n_stages"]


@pytest.mark.parametrize("D,K,Q,metric", [(16, 128, 1, "l2"), (64, 256, 3, "cosine"), (96, 384, 5, "l2"),
                                          (256, 1024, 8, "cosine"), (48, 640, 2, "cosine"),
                                          (128, 128, 4, "cosine"), (64, 1024, 40, "l2")])
def test_small_code_space_shapes(D, K, Q, metric):
    """d = 8: chunk counts 1 to 8 (split three ways across a CTA's pipelines,
    some of which then scan nothing), both metrics, up to 40 stages."""
    w, W = _small_weights(D=D, K=K, Q=Q, seed=D + K + Q, d=8)
    x = np.random.default_rng(D + Q).standard_normal((300, D)).astype(np.float32)
    run_small(W, x, label=f"d=8 D={D} K={K} Q={Q} {metric}", metric=metric)


@pytest.mark.parametrize("metric", ["l2", "cosine"])
def test_small_code_space_three_tile_items(metric):
    """d = 8 with more tiles than SMs: items of three tiles, one per
    pipeline, the last items with tiles past the end."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = (3 * sms + 5) * 128 - 77
    w, W = _small_weights(D=64, K=256, Q=4, seed=91, d=8)
    x = np.random.default_rng(91).standard_normal((N, 64)).astype(np.float32)
    run_small(W, x, label=f"d=8 three-tile items {metric}", metric=metric)


@pytest.mark.parametrize("d", [8, 64])
def test_cosine_biases_prefix_and_scale(d):
    """Both biases, prefix depths, and the eps floor: frames scaled down to
    norm ~1e-14 give projections below 1e-12, where the query is divided by
    eps instead of by its norm."""
    w, W = _small_weights(D=128, K=512, Q=5, bias=True, seed=31, d=d)
    rng = np.random.default_rng(32)
    x = rng.standard_normal((400, 128)).astype(np.float32)
    _, full = run_small(W, x, label=f"cosine d={d} bias", metric="cosine")
    for n_q in (1, 3):
        _, c = run_small(W, x, n_q=n_q, label=f"cosine d={d} n_q={n_q}", metric="cosine")
        assert np.array_equal(c, full[:, :n_q]), "prefix property"
    # the reconstruction of such frames is a sum of stored codewords, O(1)
    # against frames of ~1e-14: its tolerance is taken on the oracle's
    # reconstruction, as for decode-only inputs
    W0 = dict(W, b_in=None, b_out=None)
    tiny = (x[:200] * 1e-14).astype(np.float32)
    rvq = make_rvq(W0, "cosine")
    codes, x_hat = rvq.reconstruct(torch.from_numpy(tiny).to(DEV))
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    y_ref, _ = oracle.decode(W0, c)
    check_encode(W0, tiny, c, x_rms=rms(y_ref), x_hat_gpu=x_hat.cpu().numpy(), label=f"cosine d={d} tiny frames",
                 metric="cosine")


def test_cosine_d64_workload_shapes():
    """d = 64 with the normalised metric: a two-tile launch and a split one."""
    for N, K in ((150 * 128 + 40, 1024), (300, 256)):
        w, W = _small_weights(D=256, K=K, Q=4, seed=N % 97, d=64)
        x = np.random.default_rng(N).standard_normal((N, 256)).astype(np.float32)
        run_small(W, x, label=f"cosine d=64 N={N} K={K}", metric="cosine")


# ---------------------------------------------------------------------------
# the codec's Linear layers folded into the tables (fc before, fc2 after)
# ---------------------------------------------------------------------------

def _with_fc(W, D, D_in, D_out, seed):
    rng = np.random.default_rng(seed)
    W = dict(W)
    if D_in:
        W["fc_w"] = (rng.standard_normal((D, D_in)) / np.sqrt(D_in)).astype(np.float32)
        W["fc_b"] = (0.1 * rng.standard_normal(D)).astype(np.float32)
    if D_out:
        W["fc2_w"] = (rng.standard_normal((D_out, D)) / np.sqrt(D)).astype(np.float32)
        W["fc2_b"] = (0.1 * rng.standard_normal(D_out)).astype(np.float32)
    return W


@pytest.mark.parametrize("D,D_in,D_out,d,metric", [(128, 96, 64, 64, "l2"), (128, 256, 0, 64, "cosine"),
                                                   (96, 0, 32, 8, "cosine"), (64, 64, 64, 8, "l2")])
def test_fc_and_fc2_folded(D, D_in, D_out, d, metric):
    """fc (D_in -> D) folded into the projections and fc2 (D -> D_out) into the
    decode table, against the oracle applying both explicitly in float64."""
    w, W = _small_weights(D=D, K=256, Q=4, seed=D + D_in + D_out + d, d=d)
    W = _with_fc(W, D, D_in, D_out, seed=d + D_in)
    x = np.random.default_rng(D_in + 1).standard_normal((700, D_in or D)).astype(np.float32)
    rvq = make_rvq(W, metric)
    codes, x_hat = rvq.reconstruct(torch.from_numpy(x).to(DEV))
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    y_ref, _ = oracle.decode(W, c)
    assert x_hat.shape == (700, D_out or D)
    check_encode(W, x, c, x_rms=rms(y_ref), x_hat_gpu=x_hat.cpu().numpy(), label=f"fc {D_in}->{D}->{D_out}",
                 metric=metric)


def test_omnivoice_fc_workload_sampled():
    """The OmniVoice codec shape with fc 1024 -> 1024 and fc2 1024 -> 256:
    2000 sampled frames checked on the oracle."""
    w = ri.WORKLOAD_BY_NAME["omnivoice_fc"]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)
    rvq = make_rvq(W, w.metric)
    codes, x_hat = rvq.reconstruct(torch.from_numpy(x).to(DEV))
    torch.cuda.synchronize()
    rows = np.sort(np.concatenate([np.random.default_rng(4).choice(w.N - 2, 1998, replace=False) + 1, [0, w.N - 1]]))
    c = codes.cpu().numpy()
    y_ref, _ = oracle.decode(W, c[rows])
    res = check_encode(W, x, c, rows=rows, x_rms=rms(y_ref), x_hat_gpu=x_hat.cpu().numpy(), label="omnivoice_fc")
    assert res["n_equal"] >= 0.97 * res["n_stages"]
