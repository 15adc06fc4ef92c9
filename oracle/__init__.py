"""ctypes wrapper over the float64 C++ RVQ oracle (rvq_oracle.cpp).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may use it; the CUDA path never does.  Nothing here imports the
CUDA package, and the CUDA package imports nothing from here.

Functions
---------
encode(weights, x, n_q, threads=0, metric="l2") -> dict(codes, gap, best_dist, residual)
    The residual loop of omnivoice.cpp ARCHITECTURE.md, "RVQ codec", in float64.
    metric="cosine": the quantizer of moss-tts.cpp AGENTS.md, gotcha 9 -- the
    projection and every codeword are L2-normalised (eps 1e-12) before the
    argmin; the residual update and decode use the stored codeword.
decode(weights, codes, n_q, threads=0) -> (y float64 [N][D], n_bad)
    The accumulated decode graph of the same section, in float64.
reconstruct(weights, x, n_q) -> dict(codes, ..., x_hat)
    decode(encode(x)).

`weights` is a dict of float32 numpy arrays: w_in [Q][d][D], codebook [Q][K][d],
w_out [Q][D][d], and optionally b_in [Q][d] and b_out [Q][D] (None = zero).
Optionally the Linear layers around the quantizer (omnivoice.cpp
ARCHITECTURE.md, "Audio tokenizer"): fc_w [D][D_in] with fc_b [D] maps each
frame before the residual loop (x is then [N][D_in]); fc2_w [D_out][D] with
fc2_b [D_out] maps the decoded sum (decode then returns [N][D_out]).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rvq_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "librvq_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (IEEE float64, no contraction into FMA)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = ctypes.c_void_p
            lib.rvq_oracle_encode.argtypes = [ctypes.c_int] * 4 + [f] * 6 + [ctypes.c_int64, ctypes.c_int] + [f] * 4 + [ctypes.c_int]
            lib.rvq_oracle_encode.restype = ctypes.c_int
            lib.rvq_oracle_encode_metric.argtypes = ([ctypes.c_int] * 4 + [f] * 6 + [ctypes.c_int64, ctypes.c_int]
                                                     + [f] * 4 + [ctypes.c_int, ctypes.c_int])
            lib.rvq_oracle_encode_metric.restype = ctypes.c_int
            lib.rvq_oracle_encode_ex.argtypes = ([ctypes.c_int] * 5 + [f] * 8 + [ctypes.c_int64, ctypes.c_int]
                                                 + [f] * 4 + [ctypes.c_int, ctypes.c_int])
            lib.rvq_oracle_encode_ex.restype = ctypes.c_int
            lib.rvq_oracle_decode_ex.argtypes = ([ctypes.c_int] * 5 + [f] * 6 + [ctypes.c_int64, ctypes.c_int, f, f,
                                                                                ctypes.c_int])
            lib.rvq_oracle_decode_ex.restype = ctypes.c_int
            lib.rvq_oracle_decode.argtypes = [ctypes.c_int] * 4 + [f] * 4 + [ctypes.c_int64, ctypes.c_int, f, f, ctypes.c_int]
            lib.rvq_oracle_decode.restype = ctypes.c_int
            lib.rvq_oracle_version.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _dims(weights):
    Q, d, D = weights["w_in"].shape
    K = weights["codebook"].shape[1]
    assert weights["codebook"].shape == (Q, K, d)
    assert weights["w_out"].shape == (Q, D, d)
    if weights.get("b_in") is not None:
        assert weights["b_in"].shape == (Q, d)
    if weights.get("b_out") is not None:
        assert weights["b_out"].shape == (Q, D)
    return D, d, K, Q


def _fc_dims(weights, D):
    """(D_in, D_out): the widths before fc and after fc2 (D where absent)."""
    D_in, D_out = D, D
    if weights.get("fc_w") is not None:
        assert weights["fc_w"].shape[0] == D
        D_in = weights["fc_w"].shape[1]
        if weights.get("fc_b") is not None:
            assert weights["fc_b"].shape == (D,)
    if weights.get("fc2_w") is not None:
        assert weights["fc2_w"].shape[1] == D
        D_out = weights["fc2_w"].shape[0]
        if weights.get("fc2_b") is not None:
            assert weights["fc2_b"].shape == (D_out,)
    return D_in, D_out


METRICS = {"l2": 0, "cosine": 1}


def encode(weights: dict, x: np.ndarray, n_q: int | None = None, threads: int = 0,
           want_residual: bool = True, metric: str = "l2") -> dict:
    lib = _load()
    m = METRICS[metric]
    D, d, K, Q = _dims(weights)
    D_in, _ = _fc_dims(weights, D)
    n_q = Q if n_q is None else int(n_q)
    x = _f32(x)
    N = x.shape[0]
    assert x.shape == (N, D_in)
    w = {k: _f32(weights.get(k)) for k in ("w_in", "b_in", "codebook", "w_out", "b_out")}
    codes = np.empty((N, n_q), dtype=np.int32)
    gap = np.empty((N, n_q), dtype=np.float64)
    best = np.empty((N, n_q), dtype=np.float64)
    resid = np.empty((N, D), dtype=np.float64) if want_residual else None
    if weights.get("fc_w") is not None:
        fc_w, fc_b = _f32(weights["fc_w"]), _f32(weights.get("fc_b"))
        rc = lib.rvq_oracle_encode_ex(D_in, D, d, K, Q, _ptr(w["w_in"]), _ptr(w["b_in"]), _ptr(w["codebook"]),
                                      _ptr(w["w_out"]), _ptr(w["b_out"]), _ptr(fc_w), _ptr(fc_b), _ptr(x), N, n_q,
                                      _ptr(codes), _ptr(gap), _ptr(best), _ptr(resid), m, int(threads))
    elif m == 0:
        rc = lib.rvq_oracle_encode(D, d, K, Q, _ptr(w["w_in"]), _ptr(w["b_in"]), _ptr(w["codebook"]),
                                   _ptr(w["w_out"]), _ptr(w["b_out"]), _ptr(x), N, n_q, _ptr(codes),
                                   _ptr(gap), _ptr(best), _ptr(resid), int(threads))
    else:
        rc = lib.rvq_oracle_encode_metric(D, d, K, Q, _ptr(w["w_in"]), _ptr(w["b_in"]), _ptr(w["codebook"]),
                                          _ptr(w["w_out"]), _ptr(w["b_out"]), _ptr(x), N, n_q, _ptr(codes),
                                          _ptr(gap), _ptr(best), _ptr(resid), m, int(threads))
    if rc != 0:
        raise ValueError("rvq_oracle_encode rejected its arguments")
    return {"codes": codes, "gap": gap, "best_dist": best, "residual": resid}


def decode(weights: dict, codes: np.ndarray, n_q: int | None = None, threads: int = 0):
    lib = _load()
    D, d, K, Q = _dims(weights)
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    N = codes.shape[0]
    n_q = codes.shape[1] if n_q is None else int(n_q)
    assert codes.shape == (N, n_q)
    w = {k: _f32(weights.get(k)) for k in ("codebook", "w_out", "b_out", "fc2_w", "fc2_b")}
    _, D_out = _fc_dims(weights, D)
    y = np.empty((N, D_out), dtype=np.float64)
    n_bad = ctypes.c_int64(0)
    if w["fc2_w"] is not None:
        rc = lib.rvq_oracle_decode_ex(D, D_out, d, K, Q, _ptr(w["codebook"]), _ptr(w["w_out"]), _ptr(w["b_out"]),
                                      _ptr(w["fc2_w"]), _ptr(w["fc2_b"]), _ptr(codes), N, n_q, _ptr(y),
                                      ctypes.addressof(n_bad), int(threads))
    else:
        rc = lib.rvq_oracle_decode(D, d, K, Q, _ptr(w["codebook"]), _ptr(w["w_out"]), _ptr(w["b_out"]),
                                   _ptr(codes), N, n_q, _ptr(y), ctypes.addressof(n_bad), int(threads))
    if rc != 0:
        raise ValueError("rvq_oracle_decode rejected its arguments")
    return y, int(n_bad.value)


def reconstruct(weights: dict, x: np.ndarray, n_q: int | None = None, threads: int = 0,
                metric: str = "l2") -> dict:
    enc = encode(weights, x, n_q, threads, metric=metric)
    y, _ = decode(weights, enc["codes"], enc["codes"].shape[1], threads)
    enc["x_hat"] = y
    return enc


def version() -> str:
    return _load().rvq_oracle_version().decode()
