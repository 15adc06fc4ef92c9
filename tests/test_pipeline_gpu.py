"""The host-memory pipeline (rvq_pipeline_*): frames in pinned host memory go
through chunked copies overlapped with encode + decode; the results must be
identical to the device-buffer entry points on the same frames."""

import numpy as np
import pytest
import torch

import rvq_inputs as ri

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import residual_vector_quantisation_gb300 as rq  # noqa: E402
from residual_vector_quantisation_gb300 import build as rqb  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def rvq():
    rqb.build_library()
    rq.load_library()
    w = ri.WORKLOAD_BY_NAME["tiny"]
    W = ri.weights_to_torch(ri.make_weights(w, with_bias=True), DEV)
    return rq.RVQ(W["w_in"], W["codebook"], W["w_out"], W["b_in"], W["b_out"], device=DEV)


@pytest.mark.parametrize("n,chunk,n_q", [(250, 100, 8), (1000, 128, 8), (77, 256, 3), (4097, 640, 5)])
def test_pipeline_matches_device_path(rvq, n, chunk, n_q):
    x = torch.from_numpy(np.random.default_rng(n).standard_normal((n, rvq.D)).astype(np.float32))
    x_host = x.pin_memory()
    pipe = rq.RVQPipeline(rvq, n_q=n_q, chunk_frames=chunk)
    codes_h, x_hat_h = pipe.reconstruct(x_host)
    # the device path on the same chunks (a chunk of up to rvq_set_stream_max_frames
    # frames runs on the small-batch kernels, a larger one on the tile kernels)
    parts = [rvq.reconstruct(x[c0:c0 + chunk].to(DEV), n_q=n_q) for c0 in range(0, n, chunk)]
    codes_d = torch.cat([c for c, _ in parts])
    x_hat_d = torch.cat([y for _, y in parts])
    torch.cuda.synchronize()
    assert torch.equal(codes_h, codes_d.cpu())
    assert torch.equal(x_hat_h, x_hat_d.cpu())
    # codes only, and a second call on the same pipeline
    codes2, none = pipe.reconstruct(x_host, want_x_hat=False)
    assert none is None and torch.equal(codes2, codes_h)
    pipe.close()


@pytest.mark.parametrize("threshold", [0, 1 << 40])
def test_pipeline_on_each_encode_path(rvq, threshold):
    """Chunks of 300 frames on the tile kernels (threshold 0) and on the
    small-batch kernels: the same codes as the device path on those chunks."""
    prev = rq.rvq_set_stream_max_frames(threshold)
    try:
        n, chunk = 900, 300
        x = torch.from_numpy(np.random.default_rng(7).standard_normal((n, rvq.D)).astype(np.float32))
        pipe = rq.RVQPipeline(rvq, chunk_frames=chunk)
        codes_h, _ = pipe.reconstruct(x.pin_memory(), want_x_hat=False)
        codes_d = torch.cat([rvq.encode(x[c0:c0 + chunk].to(DEV)) for c0 in range(0, n, chunk)])
        torch.cuda.synchronize()
        assert torch.equal(codes_h, codes_d.cpu())
        pipe.close()
    finally:
        rq.rvq_set_stream_max_frames(prev)


def test_pipeline_rejects_bad_arguments(rvq):
    with pytest.raises(ValueError):
        rq.RVQPipeline(rvq, n_q=rvq.Q + 1)
    pipe = rq.RVQPipeline(rvq, chunk_frames=64)
    with pytest.raises(ValueError):
        pipe.reconstruct(torch.zeros((4, rvq.D), device=DEV))  # device tensor is not a host buffer
    pipe.close()


def test_pipeline_cancel_between_chunks(rvq):
    """The cancel callback is polled before each chunk (omnivoice.cpp
    ARCHITECTURE.md, "Public API"): stopping after the first chunk returns
    RVQ_ERR_CANCELLED with that chunk's outputs written in full and the later
    frames' outputs untouched; with the callback removed the pipeline runs to
    the end again."""
    n, chunk = 1000, 256
    x = torch.from_numpy(np.random.default_rng(11).standard_normal((n, rvq.D)).astype(np.float32)).pin_memory()
    pipe = rq.RVQPipeline(rvq, chunk_frames=chunk)
    want, _ = pipe.reconstruct(x, want_x_hat=False)
    polls = []
    pipe.set_cancel(lambda: polls.append(1) or len(polls) > 1)
    codes = torch.full((n, rvq.Q), -7, dtype=torch.int32).pin_memory()
    with pytest.raises(rq.RVQError) as err:
        pipe.reconstruct(x, codes_host=codes, want_x_hat=False)
    assert err.value.status == rq.RVQ_ERR_CANCELLED
    assert len(polls) == 2
    assert torch.equal(codes[:chunk], want[:chunk])
    assert bool((codes[chunk:] == -7).all())
    pipe.set_cancel(None)
    again, _ = pipe.reconstruct(x, want_x_hat=False)
    assert torch.equal(again, want)
    pipe.close()
