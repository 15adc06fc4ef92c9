"""rvq_encode_static: encode for callers that cannot allocate device memory.

A caller such as a real-time audio callback, or an application whose device
memory all belongs to its own pool, may not call cudaMalloc when it encodes.
rvq_encode_static uses a fixed scratch array inside the library instead of a
caller-provided scratch buffer.  These tests call it through the C ABI and
check that its codes equal rvq_encode's on two calls in a row (the second call
must not be disturbed by what the first left in the shared array), that the
second call changes the device's free memory not at all, that a call too
large for the array is refused before anything runs, that the status word of
the last call can be read back (rvq_read_status with no scratch), and that the
codes follow the float64 oracle on the 8-dim cosine code space and on
4096-entry codebooks too.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import oracle
import rvq_inputs as ri
from rvq_compare import compare_codes

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import residual_vector_quantisation_gb300 as rq  # noqa: E402
from residual_vector_quantisation_gb300 import build as rqb  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def prepared():
    rqb.build_library()
    rq.load_library()
    w = ri.WORKLOAD_BY_NAME["omnivoice"]
    W = ri.weights_to_torch(ri.make_weights(w, with_bias=True), DEV)
    rvq = rq.RVQ(W["w_in"], W["codebook"], W["w_out"], W["b_in"], W["b_out"], device=DEV)
    x = torch.from_numpy(ri.make_x(w, ri.make_weights(w), rows=np.arange(3000))).to(DEV)
    return rvq, x


def test_static_scratch_matches_rvq_encode_on_two_calls(prepared):
    rvq, x = prepared
    n_q = rvq.Q
    # two different batches, the second smaller than the first so that stale
    # rows of the first call remain in the shared array
    batches = [x[:3000].contiguous(), x[1000:2333].contiguous()]
    want = [rvq.encode(b) for b in batches]
    got = [torch.full((b.shape[0], n_q), -7, dtype=torch.int32, device=DEV) for b in batches]
    torch.cuda.synchronize()
    rq.rvq_encode_static(rvq.dims, rvq.tables, batches[0], n_q, got[0])
    torch.cuda.synchronize()
    free_after_first = torch.cuda.mem_get_info(DEV)[0]
    rq.rvq_encode_static(rvq.dims, rvq.tables, batches[1], n_q, got[1])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(DEV)[0] == free_after_first
    for g, w_ in zip(got, want):
        # same kernels and arithmetic as rvq_encode: the codes agree exactly
        assert torch.equal(g, w_)
    assert rq.rvq_read_status(None) == 0  # the library's own status word: no device wait gave up


def test_static_scratch_prefix_depth(prepared):
    rvq, x = prepared
    b = x[:500].contiguous()
    got = torch.empty((500, 3), dtype=torch.int32, device=DEV)
    rq.rvq_encode_static(rvq.dims, rvq.tables, b, 3, got)
    assert torch.equal(got, rvq.encode(b, n_q=3))


def test_static_scratch_refuses_calls_that_do_not_fit(prepared):
    rvq, _ = prepared
    row = rvq.Q * rvq.d * 4
    n_max = (rq.RVQ_STATIC_SCRATCH_BYTES - 256) // row  # a 256-byte status header, then the projections
    big = torch.zeros((n_max + 1, rvq.D), dtype=torch.float32, device=DEV)
    codes = torch.empty((n_max + 1, rvq.Q), dtype=torch.int32, device=DEV)
    with pytest.raises(rq.RVQError) as err:
        rq.rvq_encode_static(rvq.dims, rvq.tables, big, rvq.Q, codes)
    assert err.value.status == -3  # RVQ_ERR_WORKSPACE
    # exactly at the limit is accepted
    rq.rvq_encode_static(rvq.dims, rvq.tables, big[:n_max].contiguous(), rvq.Q, codes[:n_max])
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,n", [("moss_lfq", 700), ("k4096_q10", 300)])
def test_static_scratch_other_shapes_against_oracle(name, n):
    """The 8-dim cosine code space (moss_lfq, its own search kernel) and
    4096-entry codebooks (k4096_q10): equal to rvq_encode, and the codes follow
    the oracle under the relative-gap rule, on two calls in a row."""
    rqb.build_library()
    w = ri.WORKLOAD_BY_NAME[name]
    Wn = ri.make_weights(w)
    W = ri.weights_to_torch(Wn, DEV)
    rvq = rq.RVQ(W["w_in"], W["codebook"], W["w_out"], device=DEV, metric=w.metric)
    xn = ri.make_x(w, Wn, rows=np.arange(n))
    x = torch.from_numpy(xn).to(DEV)
    ref = oracle.encode(Wn, xn, want_residual=False, metric=w.metric)
    for part in (slice(0, n), slice(n // 3, n)):
        xs = x[part].contiguous()
        got = torch.full((xs.shape[0], w.Q), -7, dtype=torch.int32, device=DEV)
        rq.rvq_encode_static(rvq.dims, rvq.tables, xs, w.Q, got)
        want = rvq.encode(xs)
        torch.cuda.synchronize()
        assert rq.rvq_read_status(None) == 0
        assert torch.equal(got, want)
        res = compare_codes(got.cpu().numpy(), ref["codes"][part], ref["gap"][part])
        assert res["n_fail"] == 0, res
