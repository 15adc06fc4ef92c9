"""The small-batch (streaming) encode kernel against the float64 oracle.

Calls of at most rvq_set_stream_max_frames frames run on the cluster kernel
(each 16-frame group on one cluster of min(8, K/128) CTAs that exchange their
best keys through distributed shared memory).  These tests raise the
threshold so that every call of the shapes below takes it, compare every
frame with the oracle under the near-tie rule, and check the reconstruction
through decode.  Shapes cover every cluster size (K = 128 .. 1024), the wide
slices (K = 2048, 4096), both metrics, d = 8 and 64, biases, prefix depths,
stage counts that are not multiples of the cluster size, ragged frame counts
(1, 2, 7, 16, 17, 33, 64, 300) and the workload shapes.
"""

import contextlib
import subprocess

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
ALL = 1 << 40  # threshold that sends every call to the streaming kernel


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rqb.build_library()
    rq.load_library()
    prev = rq.rvq_set_stream_max_frames(-1)
    yield
    rq.rvq_set_stream_max_frames(prev)


@contextlib.contextmanager
def stream_max(frames):
    prev = rq.rvq_set_stream_max_frames(frames)
    try:
        yield
    finally:
        rq.rvq_set_stream_max_frames(prev)


def make_rvq(W, metric="l2"):
    t = ri.weights_to_torch(W, DEV)
    return rq.RVQ(t["w_in"], t["codebook"], t["w_out"], t["b_in"], t["b_out"], device=DEV, metric=metric,
                  fc_w=t.get("fc_w"), fc_b=t.get("fc_b"), fc2_w=t.get("fc2_w"), fc2_b=t.get("fc2_b"))


def device_status(rvq):
    """The status word at the head of the encode scratch (0: no device wait gave up)."""
    return int(rvq._scratch[:4].view(torch.int32).item())


def weights(D, K, Q, d, seed, bias=True, decay=1.0):
    w = ri.Workload("stream", 1, 1, D, Q, K, d, "gauss", cb_decay=decay, seed=seed)
    return ri.make_weights(w, with_bias=bias, bias_scale=0.3)


def check(W, x, n_q=None, metric="l2", label="", threshold=ALL):
    """Encode + reconstruct on the streaming kernel; every frame against the oracle."""
    rvq = make_rvq(W, metric)
    xt = torch.from_numpy(x).to(DEV)
    with stream_max(threshold):
        codes, x_hat = rvq.reconstruct(xt, n_q)
        torch.cuda.synchronize()
        assert device_status(rvq) == 0, f"{label}: device status word set"
        codes_e = rvq.encode(xt, n_q)
    torch.cuda.synchronize()
    assert device_status(rvq) == 0, f"{label}: device status word set"
    c = codes.cpu().numpy()
    assert np.array_equal(c, codes_e.cpu().numpy()), f"{label}: encode and reconstruct disagree"
    ref = oracle.encode(W, x, n_q, want_residual=False, metric=metric)
    res = compare_codes(c, ref["codes"], ref["gap"])
    assert res["n_fail"] == 0, f"{label}: code mismatches at clear decisions: {res}"
    y_ref, _ = oracle.decode(W, c, c.shape[1])
    err = max_abs_rel_to_rms(x_hat.cpu().numpy(), y_ref, max(rms(y_ref), 1e-30))
    assert err <= FLOAT_TOL, f"{label}: x_hat error {err:.3e} * RMS"
    return res, c


@pytest.mark.parametrize("N", [1, 2, 3, 5, 7, 9, 10, 15, 16, 17, 33, 64])
@pytest.mark.parametrize("K", [128, 256, 512, 1024])
def test_cluster_sizes_and_ragged_counts(N, K):
    """Cluster sizes 1, 2, 4, 8 (K/128 CTAs up to 8) and frame counts that leave
    the last 16-frame group partly empty."""
    D, Q = 128, 5
    W = weights(D, K, Q, 64, seed=K + N)
    x = np.random.default_rng(N * 7 + K).standard_normal((N, D)).astype(np.float32)
    check(W, x, label=f"N={N} K={K}")


@pytest.mark.parametrize("K,Q", [(2048, 3), (4096, 10), (1152, 2), (2176, 3), (3968, 2)])
def test_wide_slices(K, Q):
    """256 and 512 codewords per CTA (one thread per codeword; the second with
    two codewords a thread and one slice buffer instead of two), and slices of
    144, 272 and 496 codewords (K/8 not a multiple of 128: some threads idle)."""
    D = 256
    W = weights(D, K, Q, 64, seed=K)
    x = np.random.default_rng(K).standard_normal((40, D)).astype(np.float32)
    check(W, x, label=f"K={K}")


@pytest.mark.parametrize("d,K,Q,metric", [(64, 1024, 8, "cosine"), (64, 256, 11, "cosine"), (8, 1024, 32, "cosine"),
                                          (8, 128, 3, "l2"), (8, 512, 9, "l2"), (8, 1024, 12, "cosine")])
def test_metrics_and_code_dims(d, K, Q, metric):
    D = 96
    W = weights(D, K, Q, d, seed=d * K + Q, decay=0.8)
    x = np.random.default_rng(Q).standard_normal((37, D)).astype(np.float32)
    check(W, x, metric=metric, label=f"d={d} K={K} Q={Q} {metric}")


def test_prefix_depths_and_stage_counts():
    """n_q below Q (the partial-depth encode) gives the prefix of the full codes;
    stage counts 1 .. 13 against a cluster of 8."""
    D, K, Q = 192, 1024, 13
    W = weights(D, K, Q, 64, seed=99)
    x = np.random.default_rng(3).standard_normal((20, D)).astype(np.float32)
    _, full = check(W, x, label="full depth")
    for n_q in (1, 2, 7, 8, 9):
        _, c = check(W, x, n_q=n_q, label=f"n_q={n_q}")
        assert np.array_equal(c, full[:, :n_q]), "prefix property"


def test_many_groups():
    """300 frames: 19 clusters of 8 CTAs, some waiting for a free GPC."""
    D, K, Q = 256, 1024, 8
    W = weights(D, K, Q, 64, seed=5)
    x = np.random.default_rng(5).standard_normal((300, D)).astype(np.float32)
    check(W, x, label="300 frames")


@pytest.mark.parametrize("N", [33, 513, 1000, 2500])
@pytest.mark.parametrize("d,K,Q,metric", [(64, 1024, 8, "l2"), (64, 4096, 3, "l2"), (64, 1024, 32, "l2"),
                                          (8, 1024, 12, "cosine"), (64, 256, 5, "cosine"), (64, 1152, 4, "l2")])
def test_several_groups_per_cluster(N, d, K, Q, metric):
    """Calls of hundreds to thousands of frames: each cluster takes several
    16-frame groups (as many as put the call in about one wave of clusters,
    up to 8, fewer where shared memory runs out: 32 stages, K = 4096), the
    last cluster ragged; 2500 frames take two waves."""
    D = 128
    W = weights(D, K, Q, d, seed=N + K + Q, decay=0.9)
    x = np.random.default_rng(N + d).standard_normal((N, D)).astype(np.float32)
    check(W, x, metric=metric, label=f"N={N} d={d} K={K} Q={Q} {metric}")


def test_plan_of_a_call():
    """rvq_stream_plan: one group per cluster up to 16 frames (group sizes 1, 2,
    4, 8, 16 by the call's size); beyond, the fewest groups per cluster (up to
    8) that put the call in one wave, so that the cluster count falls as the
    groups per cluster rise; the clusters cover every frame; calls above the
    threshold or of shapes without the streaming tables take the tile path."""
    dims = rq._dims(1024, 64, 1024, 8)
    with stream_max(ALL):
        for n, nf in ((1, 1), (2, 2), (3, 4), (5, 8), (9, 16), (16, 16)):
            p = rq.rvq_stream_plan(dims, 8, n)
            assert p == {"stream": 1, "cluster_ctas": 8, "group_frames": nf, "groups_per_cluster": 1,
                         "clusters": 1, "slice_buffers": 2}, (n, p)
        one_wave = None
        for n in range(17, 16 * 8 * 40, 37):
            p = rq.rvq_stream_plan(dims, 8, n)
            G, c = p["groups_per_cluster"], p["clusters"]
            assert p["stream"] == 1 and p["group_frames"] == 16 and 1 <= G <= 8
            assert c * 16 * G >= n > (c - 1) * 16 * G, (n, p)
            if G < 8:  # G - 1 groups would need more clusters than this G's
                assert -(-n // (16 * (G - 1) if G > 1 else 1)) > c or G == 1, (n, p)
                one_wave = c if one_wave is None else max(one_wave, c)
        assert one_wave is not None and one_wave >= 2
        # a deep stack of wide slices: shared memory caps the groups per cluster
        deep = rq.rvq_stream_plan(rq._dims(768, 64, 4096, 32), 32, 4096)
        assert deep["stream"] == 1 and 1 <= deep["groups_per_cluster"] < 8 and deep["slice_buffers"] >= 1
    with stream_max(100):
        assert rq.rvq_stream_plan(dims, 8, 101)["stream"] == 0
        assert rq.rvq_stream_plan(dims, 8, 100)["stream"] == 1
    assert rq.rvq_stream_plan(rq._dims(256, 64, 8192, 4), 4, 16)["stream"] == 0


@pytest.mark.parametrize("name", ["tiny", "omnivoice", "moss_deep", "k4096_q10", "moss_lfq", "omnivoice_fc"])
def test_workload_shapes_small_batches(name):
    """The first frames of each workload, in calls of 1, 16 and 48 frames."""
    w = ri.WORKLOAD_BY_NAME[name]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)[:48]
    for n in (1, 16, 48):
        check(W, np.ascontiguousarray(x[:n]), metric=w.metric, label=f"{name} n={n}")


def test_planted_codes_recovered():
    """Frames built as sums of the stage outputs of chosen codes, with
    well-separated codebooks and no noise, give back those codes."""
    w = ri.WORKLOAD_BY_NAME["omnivoice"]
    W = ri.make_weights(w)
    rng = np.random.default_rng(11)
    codes = rng.integers(0, w.K, size=(16, w.Q)).astype(np.int32)
    x, _ = oracle.decode(W, codes)
    rvq = make_rvq(W)
    with stream_max(ALL):
        got = rvq.encode(torch.from_numpy(x.astype(np.float32)).to(DEV)).cpu().numpy()
    ref = oracle.encode(W, x.astype(np.float32), want_residual=False)
    res = compare_codes(got, ref["codes"], ref["gap"])
    assert res["n_fail"] == 0, res


def test_exact_ties_take_lowest_index():
    """Duplicated codewords in different slices (different CTAs of the cluster)
    and in the same slice: the lower index wins."""
    D, K, Q = 64, 1024, 2
    W = weights(D, K, Q, 64, seed=77, bias=False)
    W["w_in"] = np.stack([np.eye(64, dtype=np.float32)] * Q)
    W["w_out"] = np.stack([np.eye(64, dtype=np.float32)] * Q)
    for q in range(Q):
        for lo, hi in ((3, 900), (17, 18), (300, 1023), (130, 260)):
            W["codebook"][q, hi] = W["codebook"][q, lo]
    picks = np.array([3, 900, 17, 18, 300, 1023, 130, 260] * 2)
    rng = np.random.default_rng(8)
    x = (W["codebook"][0][picks] + 0.01 * rng.standard_normal((len(picks), D))).astype(np.float32)
    rvq = make_rvq(W)
    with stream_max(ALL):
        codes = rvq.encode(torch.from_numpy(x).to(DEV)).cpu().numpy()
    ref = oracle.encode(W, x)
    assert np.array_equal(codes[:, 0], ref["codes"][:, 0])
    assert set(codes[:, 0].tolist()) <= {3, 17, 300, 130}


def test_tile_and_stream_paths_agree():
    """Both paths on the same frames: each passes the oracle rule, and they give
    the same code wherever the oracle's decision is clear."""
    w = ri.WORKLOAD_BY_NAME["omnivoice"]
    W = ri.make_weights(w)
    x = ri.make_x(w, W)[:64]
    rvq = make_rvq(W)
    xt = torch.from_numpy(x).to(DEV)
    with stream_max(0):
        c_tile = rvq.encode(xt).cpu().numpy()
    with stream_max(ALL):
        c_stream = rvq.encode(xt).cpu().numpy()
    ref = oracle.encode(W, x, want_residual=False)
    for c in (c_tile, c_stream):
        assert compare_codes(c, ref["codes"], ref["gap"])["n_fail"] == 0
    assert (c_tile == c_stream).mean() >= 0.99


def test_static_entry_point_and_determinism():
    """rvq_encode_static on small batches takes the same kernel; repeated calls
    give identical codes."""
    w = ri.WORKLOAD_BY_NAME["omnivoice"]
    W = ri.make_weights(w)
    x = torch.from_numpy(ri.make_x(w, W)[:24]).to(DEV)
    rvq = make_rvq(W)
    with stream_max(ALL):
        a = rvq.encode(x)
        b = torch.empty_like(a)
        rq.rvq_encode_static(rvq.dims, rvq.tables, x, w.Q, b)
        c = rvq.encode(x)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


def test_unsupported_shapes_fall_back():
    """Shapes the streaming kernel does not take (d = 64 with K > 4096; more
    stages than its shared memory holds) run on the tile kernels; 64 stages
    with K = 256 (30 owned per CTA) still fit."""
    for D, K, Q in ((64, 8192, 2), (64, 128, 60), (64, 256, 64)):
        W = weights(D, K, Q, 64, seed=K + Q)
        x = np.random.default_rng(K).standard_normal((10, D)).astype(np.float32)
        check(W, x, label=f"fallback K={K} Q={Q}")


def test_small_calls_are_planned_on_the_cluster_kernels():
    """rvq_stream_plan, which the encode launcher follows, sends an 8-frame
    omnivoice call to the cluster kernels (one 8-frame group on one cluster of
    8 CTAs, K/128 = 8 codebook slices) and, with the threshold at 0, to the
    tile kernels; the library holds the cluster kernel, k_stream_search; and
    the call gives the same codes under both thresholds (distinct kernels, same
    argmins) with the status word clear."""
    w = ri.WORKLOAD_BY_NAME["omnivoice"]
    W = ri.make_weights(w)
    rvq = make_rvq(W)
    with stream_max(ALL):
        plan = rq.rvq_stream_plan(rvq.dims, w.Q, 8)
    assert plan == {"stream": 1, "cluster_ctas": 8, "group_frames": 8, "groups_per_cluster": 1, "clusters": 1,
                    "slice_buffers": plan["slice_buffers"]}
    assert plan["slice_buffers"] >= 2
    with stream_max(0):
        assert rq.rvq_stream_plan(rvq.dims, w.Q, 8)["stream"] == 0
    syms = subprocess.run(["nm", "-C", rqb.LIB], capture_output=True, text=True, check=True).stdout
    assert "k_stream_search" in syms and "k_search_tc" in syms
    x = torch.from_numpy(ri.make_x(w, W)[:8]).to(DEV)
    ref = oracle.encode(W, x.cpu().numpy(), want_residual=False)
    for threshold in (ALL, 0):
        with stream_max(threshold):
            codes = rvq.encode(x)
            torch.cuda.synchronize()
        assert device_status(rvq) == 0
        assert rq.rvq_read_status(rvq._scratch) == 0
        res = compare_codes(codes.cpu().numpy(), ref["codes"], ref["gap"])
        assert res["n_fail"] == 0, (threshold, res)


@pytest.mark.parametrize("threshold", [ALL, 0])
def test_encode_replayed_from_a_cuda_graph(threshold):
    """The realtime pattern: one encode of a 16-frame buffer captured into a CUDA
    graph, then replayed for each new group of frames copied into that buffer.
    Every replay gives the eager call's codes (small-batch kernels with a
    programmatic dependent launch, or the tile kernels with threshold 0)."""
    w = ri.WORKLOAD_BY_NAME["omnivoice"]
    W = ri.make_weights(w)
    frames = torch.from_numpy(ri.make_x(w, W)[:48]).to(DEV)
    rvq = make_rvq(W)
    x = frames[:16].clone()
    codes = torch.empty((16, w.Q), dtype=torch.int32, device=DEV)
    with stream_max(threshold):
        scratch = rvq.scratch_for(16, w.Q)
        rq.rvq_encode(rvq.dims, rvq.tables, x, w.Q, codes, scratch)  # first call: kernel attributes set
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
            rq.rvq_encode(rvq.dims, rvq.tables, x, w.Q, codes, scratch)
        for g0 in (0, 16, 32):
            x.copy_(frames[g0:g0 + 16])
            codes.fill_(-1)
            graph.replay()
            eager = rvq.encode(frames[g0:g0 + 16].clone())
            torch.cuda.synchronize()
            assert torch.equal(codes, eager), f"replay of frames {g0}.."
            assert device_status(rvq) == 0
