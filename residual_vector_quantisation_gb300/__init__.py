"""Residual vector quantisation (RVQ) encode and decode on one GB300 GPU.

A thin ctypes binding over the C ABI of include/rvq.h (librvq.so, built for
sm_103a by residual_vector_quantisation_gb300.build).  The functions below
carry the C names and only marshal arguments: torch tensors become device
pointers and the current CUDA stream.  Every step of encode and decode runs in
the library's CUDA kernels; there is no CPU path.  Loading fails loudly when
the library has not been built.

    from residual_vector_quantisation_gb300 import RVQ
    rvq = RVQ(w_in, codebook, w_out, b_in=None, b_out=None)   # cuda float32 tensors
    codes = rvq.encode(x)            # [N][n_q] int32
    y = rvq.decode(codes)            # [N][D] float32
    codes, x_hat = rvq.reconstruct(x)
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "RVQError", "load_library", "library_path", "rvq_dims", "rvq_weights",
    "rvq_dims_supported", "rvq_tables_bytes", "rvq_prepare", "rvq_encode_scratch_bytes",
    "rvq_encode_min_scratch_bytes", "rvq_encode", "rvq_decode", "rvq_reconstruct",
    "rvq_status_string", "rvq_version", "rvq_encode_static", "RVQ_STATIC_SCRATCH_BYTES", "RVQ",
    "EXPORTED_SYMBOLS", "rvq_pipeline_workspace_bytes", "rvq_pipeline_create", "rvq_pipeline_destroy",
    "rvq_pipeline_reconstruct", "RVQPipeline", "rvq_set_stream_max_frames", "rvq_stream_plan",
    "rvq_read_status", "rvq_read_error_count", "rvq_pipeline_set_cancel", "RVQ_CANCEL_FN",
]

RVQ_OK = 0
STATUS_NAMES = {0: "RVQ_OK", -1: "RVQ_ERR_INVALID_ARG", -2: "RVQ_ERR_UNSUPPORTED",
                -3: "RVQ_ERR_WORKSPACE", -4: "RVQ_ERR_CUDA", -5: "RVQ_ERR_TIMEOUT",
                -6: "RVQ_ERR_CANCELLED", -7: "RVQ_ERR_INTERNAL"}
RVQ_ERR_TIMEOUT = -5
RVQ_ERR_CANCELLED = -6
RVQ_ERR_INTERNAL = -7

EXPORTED_SYMBOLS = [
    "rvq_dims_supported", "rvq_tables_bytes", "rvq_prepare", "rvq_encode_scratch_bytes",
    "rvq_encode_min_scratch_bytes", "rvq_encode", "rvq_decode", "rvq_reconstruct",
    "rvq_status_string", "rvq_version", "rvq_encode_static", "rvq_pipeline_workspace_bytes",
    "rvq_pipeline_create", "rvq_pipeline_destroy", "rvq_pipeline_reconstruct", "rvq_set_stream_max_frames",
    "rvq_stream_plan", "rvq_read_status", "rvq_read_error_count", "rvq_pipeline_set_cancel",
]

# int (*rvq_cancel_fn)(void *user)
RVQ_CANCEL_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p)

RVQ_STATIC_SCRATCH_BYTES = 16 << 20  # include/rvq.h


class RVQError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} returned {STATUS_NAMES.get(status, status)}")


RVQ_METRIC_L2 = 0       # include/rvq.h
RVQ_METRIC_COSINE = 1
METRICS = {"l2": RVQ_METRIC_L2, "cosine": RVQ_METRIC_COSINE}


class rvq_dims(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int32), ("d", ctypes.c_int32), ("K", ctypes.c_int32), ("Q", ctypes.c_int32),
                ("metric", ctypes.c_int32), ("D_in", ctypes.c_int32), ("D_out", ctypes.c_int32)]


class rvq_weights(ctypes.Structure):
    _fields_ = [("w_in", ctypes.c_void_p), ("b_in", ctypes.c_void_p), ("codebook", ctypes.c_void_p),
                ("w_out", ctypes.c_void_p), ("b_out", ctypes.c_void_p), ("fc_w", ctypes.c_void_p),
                ("fc_b", ctypes.c_void_p), ("fc2_w", ctypes.c_void_p), ("fc2_b", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(path: Optional[str] = None):
    """Load librvq.so.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"RVQ CUDA library not built ({p} missing); run "
                           "`python -m residual_vector_quantisation_gb300.build` first")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "rvq_dims_supported": ([rvq_dims], ctypes.c_int),
        "rvq_tables_bytes": ([rvq_dims], sz),
        "rvq_prepare": ([rvq_dims, ctypes.POINTER(rvq_weights), vp, sz, vp], ctypes.c_int),
        "rvq_encode_scratch_bytes": ([rvq_dims, i64, i32], sz),
        "rvq_encode_min_scratch_bytes": ([rvq_dims, i32], sz),
        "rvq_encode": ([rvq_dims, vp, vp, i64, i32, vp, vp, sz, vp], ctypes.c_int),
        "rvq_decode": ([rvq_dims, vp, vp, i64, i32, vp, vp, vp], ctypes.c_int),
        "rvq_reconstruct": ([rvq_dims, vp, vp, i64, i32, vp, vp, vp, sz, vp], ctypes.c_int),
        "rvq_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "rvq_version": ([], ctypes.c_char_p),
        "rvq_encode_static": ([rvq_dims, vp, vp, i64, i32, vp, vp], ctypes.c_int),
        "rvq_pipeline_workspace_bytes": ([rvq_dims, i32, i64], sz),
        "rvq_pipeline_create": ([rvq_dims, i32, i64, vp, sz, ctypes.POINTER(vp)], ctypes.c_int),
        "rvq_pipeline_destroy": ([vp], ctypes.c_int),
        "rvq_pipeline_reconstruct": ([vp, vp, vp, i64, vp, vp], ctypes.c_int),
        "rvq_set_stream_max_frames": ([i64], i64),
        "rvq_stream_plan": ([rvq_dims, i32, i64, ctypes.POINTER(i64)], ctypes.c_int),
        "rvq_read_status": ([vp, vp], ctypes.c_int),
        "rvq_read_error_count": ([vp, ctypes.POINTER(i64), vp], ctypes.c_int),
        "rvq_pipeline_set_cancel": ([vp, RVQ_CANCEL_FN, vp], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


# ---------------------------------------------------------------------------
# argument marshalling
# ---------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("RVQ buffers must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("RVQ buffers must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(name: str, status: int):
    if status != RVQ_OK:
        raise RVQError(name, status)


def _dims(D: int, d: int, K: int, Q: int, metric: int = RVQ_METRIC_L2, D_in: int = 0, D_out: int = 0) -> rvq_dims:
    return rvq_dims(int(D), int(d), int(K), int(Q), int(metric), int(D_in), int(D_out))


def rvq_dims_supported(dims: rvq_dims) -> int:
    return load_library().rvq_dims_supported(dims)


def rvq_tables_bytes(dims: rvq_dims) -> int:
    return load_library().rvq_tables_bytes(dims)


def rvq_encode_scratch_bytes(dims: rvq_dims, n_frames: int, n_q: int) -> int:
    return load_library().rvq_encode_scratch_bytes(dims, int(n_frames), int(n_q))


def rvq_encode_min_scratch_bytes(dims: rvq_dims, n_q: int) -> int:
    return load_library().rvq_encode_min_scratch_bytes(dims, int(n_q))


def rvq_prepare(dims: rvq_dims, w_in, codebook, w_out, b_in, b_out, tables: torch.Tensor, stream=None,
                fc_w=None, fc_b=None, fc2_w=None, fc2_b=None) -> None:
    w = rvq_weights(_ptr(w_in), _ptr(b_in), _ptr(codebook), _ptr(w_out), _ptr(b_out), _ptr(fc_w), _ptr(fc_b),
                    _ptr(fc2_w), _ptr(fc2_b))
    _check("rvq_prepare", load_library().rvq_prepare(dims, ctypes.byref(w), _ptr(tables),
                                                     tables.numel() * tables.element_size(), _stream(stream)))


def rvq_encode(dims: rvq_dims, tables, x, n_q: int, codes, scratch, stream=None) -> None:
    n = x.shape[0]
    _check("rvq_encode", load_library().rvq_encode(dims, _ptr(tables), _ptr(x), n, int(n_q), _ptr(codes),
                                                   _ptr(scratch), scratch.numel() * scratch.element_size(),
                                                   _stream(stream)))


def rvq_decode(dims: rvq_dims, tables, codes, n_q: int, y, bad_codes=None, stream=None) -> None:
    n = codes.shape[0]
    _check("rvq_decode", load_library().rvq_decode(dims, _ptr(tables), _ptr(codes), n, int(n_q), _ptr(y),
                                                   _ptr(bad_codes), _stream(stream)))


def rvq_reconstruct(dims: rvq_dims, tables, x, n_q: int, codes, x_hat, scratch, stream=None) -> None:
    n = x.shape[0]
    _check("rvq_reconstruct", load_library().rvq_reconstruct(dims, _ptr(tables), _ptr(x), n, int(n_q), _ptr(codes),
                                                             _ptr(x_hat), _ptr(scratch),
                                                             scratch.numel() * scratch.element_size(),
                                                             _stream(stream)))


def rvq_encode_static(dims: rvq_dims, tables, x, n_q: int, codes, stream=None) -> None:
    """Encode with the library's own fixed scratch (no scratch argument; see rvq.h)."""
    n = x.shape[0]
    _check("rvq_encode_static", load_library().rvq_encode_static(dims, _ptr(tables), _ptr(x), n, int(n_q),
                                                                 _ptr(codes), _stream(stream)))


def rvq_pipeline_workspace_bytes(dims: rvq_dims, n_q: int, chunk_frames: int) -> int:
    return load_library().rvq_pipeline_workspace_bytes(dims, int(n_q), int(chunk_frames))


def rvq_pipeline_create(dims: rvq_dims, n_q: int, chunk_frames: int, workspace: torch.Tensor) -> ctypes.c_void_p:
    out = ctypes.c_void_p()
    _check("rvq_pipeline_create", load_library().rvq_pipeline_create(
        dims, int(n_q), int(chunk_frames), _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(out)))
    return out


def rvq_pipeline_destroy(pipeline) -> None:
    _check("rvq_pipeline_destroy", load_library().rvq_pipeline_destroy(pipeline))


def _host_ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("host buffers must be contiguous CPU tensors")
    return ctypes.c_void_p(t.data_ptr())


def rvq_pipeline_reconstruct(pipeline, tables, x_host, codes_host, x_hat_host=None) -> None:
    _check("rvq_pipeline_reconstruct", load_library().rvq_pipeline_reconstruct(
        pipeline, _ptr(tables), _host_ptr(x_host), x_host.shape[0], _host_ptr(codes_host), _host_ptr(x_hat_host)))


def rvq_read_status(scratch: Optional[torch.Tensor] = None, stream=None) -> int:
    """Synchronise `stream` and return the status (an rvq_status value, not
    raised) that the encode last enqueued with `scratch` left in its status
    word; scratch=None reads the library's own scratch (rvq_encode_static)."""
    return int(load_library().rvq_read_status(_ptr(scratch), _stream(stream)))


def rvq_read_error_count(bad_codes: torch.Tensor, stream=None) -> int:
    """Synchronise `stream` and return rvq_decode's bad-code counter."""
    out = ctypes.c_int64(0)
    _check("rvq_read_error_count", load_library().rvq_read_error_count(_ptr(bad_codes), ctypes.byref(out),
                                                                       _stream(stream)))
    return int(out.value)


def rvq_pipeline_set_cancel(pipeline, fn, user=None) -> None:
    """fn: an RVQ_CANCEL_FN (the caller keeps it alive) or None to remove."""
    _check("rvq_pipeline_set_cancel", load_library().rvq_pipeline_set_cancel(
        pipeline, fn if fn is not None else RVQ_CANCEL_FN(), user))


def rvq_status_string(status: int) -> str:
    return load_library().rvq_status_string(int(status)).decode()


def rvq_version() -> str:
    return load_library().rvq_version().decode()


def rvq_set_stream_max_frames(max_frames: int) -> int:
    """Threshold (frames per call) of the small-batch kernel; returns the previous one."""
    return int(load_library().rvq_set_stream_max_frames(int(max_frames)))


def rvq_stream_plan(dims: rvq_dims, n_q: int, n_frames: int) -> dict:
    """How one call of n_frames frames would run on the current device."""
    out = (ctypes.c_int64 * 6)()
    _check("rvq_stream_plan", load_library().rvq_stream_plan(dims, int(n_q), int(n_frames), out))
    keys = ("stream", "cluster_ctas", "group_frames", "groups_per_cluster", "clusters", "slice_buffers")
    return {k: int(v) for k, v in zip(keys, out)}


# ---------------------------------------------------------------------------
# convenience object: owns the tables and a scratch buffer (torch allocations)
# ---------------------------------------------------------------------------

class RVQ:
    """Prepared RVQ weights on one CUDA device.

    w_in [Q][d][D], codebook [Q][K][d], w_out [Q][D][d], b_in [Q][d] or None,
    b_out [Q][D] or None; float32 tensors (moved to `device` if needed).
    metric: "l2" (squared L2) or "cosine" (both sides L2-normalised before the
    argmin, as RVQ_METRIC_COSINE in include/rvq.h).
    fc_w [D][D_in], fc_b [D] (optional): a Linear layer applied to each frame
    before the quantizer; fc2_w [D_out][D], fc2_b [D_out] (optional): one
    applied to the decoded sum.  Both are folded into the tables.
    """

    def __init__(self, w_in, codebook, w_out, b_in=None, b_out=None, device=None, stream=None,
                 metric: str = "l2", fc_w=None, fc_b=None, fc2_w=None, fc2_b=None):
        device = torch.device(device) if device is not None else (w_in.device if w_in.is_cuda else torch.device("cuda"))
        f = lambda t: None if t is None else t.to(device=device, dtype=torch.float32).contiguous()
        w_in, codebook, w_out, b_in, b_out = map(f, (w_in, codebook, w_out, b_in, b_out))
        fc_w, fc_b, fc2_w, fc2_b = map(f, (fc_w, fc_b, fc2_w, fc2_b))
        Q, d, D = w_in.shape
        K = codebook.shape[1]
        self.D, self.d, self.K, self.Q = D, d, K, Q
        self.D_in = fc_w.shape[1] if fc_w is not None else D
        self.D_out = fc2_w.shape[0] if fc2_w is not None else D
        self.device = device
        self.metric = metric
        self.dims = _dims(D, d, K, Q, METRICS[metric], self.D_in, self.D_out)
        status = rvq_dims_supported(self.dims)
        _check("rvq_dims_supported", status)
        nbytes = rvq_tables_bytes(self.dims)
        self.tables = torch.empty(nbytes, dtype=torch.uint8, device=device)
        with torch.cuda.device(device):
            rvq_prepare(self.dims, w_in, codebook, w_out, b_in, b_out, self.tables, stream, fc_w, fc_b, fc2_w, fc2_b)
        self._scratch = None

    def scratch_for(self, n_frames: int, n_q: int) -> torch.Tensor:
        need = max(rvq_encode_scratch_bytes(self.dims, n_frames, n_q), 16)
        if self._scratch is None or self._scratch.numel() < need:
            self._scratch = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._scratch

    def _frames(self, x):
        if x.dim() != 2 or x.shape[1] != self.D_in:
            raise ValueError(f"x must be [N][{self.D_in}]")
        return x.to(device=self.device, dtype=torch.float32).contiguous()

    def encode(self, x, n_q: Optional[int] = None, codes=None, stream=None):
        n_q = self.Q if n_q is None else int(n_q)
        x = self._frames(x)
        if codes is None:
            codes = torch.empty((x.shape[0], n_q), dtype=torch.int32, device=self.device)
        rvq_encode(self.dims, self.tables, x, n_q, codes, self.scratch_for(x.shape[0], n_q), stream)
        return codes

    def decode(self, codes, n_q: Optional[int] = None, y=None, bad_codes=None, stream=None):
        codes = codes.to(device=self.device, dtype=torch.int32).contiguous()
        n_q = codes.shape[1] if n_q is None else int(n_q)
        if y is None:
            y = torch.empty((codes.shape[0], self.D_out), dtype=torch.float32, device=self.device)
        rvq_decode(self.dims, self.tables, codes, n_q, y, bad_codes, stream)
        return y

    def reconstruct(self, x, n_q: Optional[int] = None, codes=None, x_hat=None, stream=None):
        n_q = self.Q if n_q is None else int(n_q)
        x = self._frames(x)
        n = x.shape[0]
        if codes is None:
            codes = torch.empty((n, n_q), dtype=torch.int32, device=self.device)
        if x_hat is None:
            x_hat = torch.empty((n, self.D_out), dtype=torch.float32, device=self.device)
        rvq_reconstruct(self.dims, self.tables, x, n_q, codes, x_hat, self.scratch_for(n, n_q), stream)
        return codes, x_hat


class RVQPipeline:
    """Encode + decode of frames held in host memory, copies overlapped with compute.

    Wraps rvq_pipeline_*: the device workspace is a torch allocation owned by
    this object.  Pinned host tensors give full copy bandwidth.
    """

    def __init__(self, rvq: "RVQ", n_q: Optional[int] = None, chunk_frames: int = 38912):
        self.rvq = rvq
        self.n_q = rvq.Q if n_q is None else int(n_q)
        nbytes = rvq_pipeline_workspace_bytes(rvq.dims, self.n_q, chunk_frames)
        if nbytes == 0:
            raise ValueError("unsupported pipeline arguments")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=rvq.device)
        with torch.cuda.device(rvq.device):
            self.handle = rvq_pipeline_create(rvq.dims, self.n_q, chunk_frames, self.workspace)

    def reconstruct(self, x_host: torch.Tensor, codes_host: Optional[torch.Tensor] = None,
                    x_hat_host: Optional[torch.Tensor] = None, want_x_hat: bool = True):
        n = x_host.shape[0]
        if codes_host is None:
            codes_host = torch.empty((n, self.n_q), dtype=torch.int32, pin_memory=True)
        if x_hat_host is None and want_x_hat:
            x_hat_host = torch.empty((n, self.rvq.D_out), dtype=torch.float32, pin_memory=True)
        with torch.cuda.device(self.rvq.device):
            rvq_pipeline_reconstruct(self.handle, self.rvq.tables, x_host, codes_host, x_hat_host)
        return codes_host, x_hat_host

    def set_cancel(self, should_stop=None):
        """should_stop() -> bool is polled before each chunk; None removes it."""
        self._cancel = None if should_stop is None else RVQ_CANCEL_FN(lambda _user: 1 if should_stop() else 0)
        rvq_pipeline_set_cancel(self.handle, self._cancel)

    def close(self):
        if getattr(self, "handle", None) is not None:
            rvq_pipeline_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
