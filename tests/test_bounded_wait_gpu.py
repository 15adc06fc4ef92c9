"""A device wait that runs out reports a status instead of hanging.

Every mbarrier wait in the library is bounded (rvq::ptx::mbar_wait).  This
test builds a kernel, with a short poll limit, that waits on a barrier nothing
ever arrives at, and checks that it gives up, sets the timeout status (5),
returns, and that the next kernel on the same context runs normally; and a
2-CTA cluster kernel doing the same with the cluster-scope waits of the
small-batch kernels, whose CTAs must still meet at their closing barrier.  No GPU
fault or hang is involved."""

import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from residual_vector_quantisation_gb300 import build as rqb  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounded_wait_times_out_and_context_survives(tmp_path):
    so = tmp_path / "libselftest.so"
    subprocess.run([rqb.nvcc(), *rqb.ARCH, "-O2", "-std=c++17", "-DRVQ_SPIN_LIMIT=4096u", "-Xcompiler", "-fPIC",
                    "-shared", "-I", rqb.CSRC, os.path.join(HERE, "gpu_selftest", "bounded_wait.cu"), "-o", str(so)],
                   check=True)
    lib = ctypes.CDLL(str(so))
    lib.selftest_bounded_wait.argtypes = [ctypes.c_void_p] * 3
    lib.selftest_bounded_wait.restype = ctypes.c_int
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    clk = torch.zeros(2, dtype=torch.int64, device="cuda")
    after = torch.zeros(32, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    rc = lib.selftest_bounded_wait(ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(clk.data_ptr()),
                                   ctypes.c_void_p(after.data_ptr()))
    assert rc == 0
    assert int(status[0].item()) == 5
    assert int(clk[0].item()) > 0
    # the cluster kernel: both CTAs' cluster-scope waits gave up, and both
    # reached the closing cluster barrier
    assert int(status[1].item()) == 2
    assert int(clk[1].item()) > 0
    assert torch.equal(after.cpu(), torch.arange(1000, 1032, dtype=torch.int32))
    # and torch's own kernels still run on this context
    assert float((torch.ones(1024, device="cuda") * 2).sum().item()) == 2048.0
    # the word the timed-out kernel left is what the library's status query
    # reports for a scratch buffer holding it: RVQ_ERR_TIMEOUT
    import residual_vector_quantisation_gb300 as rq
    rqb.build_library()
    scratch = torch.zeros(64, dtype=torch.int32, device="cuda")
    scratch[0] = status[0]
    assert rq.rvq_read_status(scratch) == rq.RVQ_ERR_TIMEOUT
    scratch[0] = 6  # a kernel that refused its launch shape
    assert rq.rvq_read_status(scratch) == rq.RVQ_ERR_INTERNAL
    scratch[0] = 0
    assert rq.rvq_read_status(scratch) == 0
