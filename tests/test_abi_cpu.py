"""The C ABI without a GPU: the library builds, exports exactly the symbols
include/rvq.h declares, and every entry point's early-return path works."""

import ctypes
import os
import re
import subprocess

import pytest

import residual_vector_quantisation_gb300 as rq
from residual_vector_quantisation_gb300 import build as rqb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rvq.h")


@pytest.fixture(scope="module")
def lib_path():
    return rqb.build_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"RVQ_API\s+[^;]*?\b(rvq_\w+)\s*\(", text, flags=re.S)))


def test_header_declarations_match_binding():
    assert declared_symbols() == sorted(rq.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines() if " T " in line})
    public = [s for s in exported if s.startswith("rvq_")]
    assert public == declared_symbols()
    # nothing but the rvq_ prefix is exported from our code (-fvisibility=hidden)
    ours = [s for s in exported if not s.startswith(("_", "rvq_"))]
    assert not [s for s in ours if "rvq" in s.lower()]
    lib = ctypes.CDLL(lib_path)
    for name in declared_symbols():
        assert hasattr(lib, name)


def test_early_return_paths(lib_path):
    lib = rq.load_library()
    ok = rq.rvq_dims(1024, 64, 1024, 8)
    assert lib.rvq_dims_supported(ok) == 0
    assert lib.rvq_dims_supported(rq.rvq_dims(1000, 64, 1024, 8)) == -2   # D % 16
    assert lib.rvq_dims_supported(rq.rvq_dims(1024, 64, 1000, 8)) == -2   # K % 128
    assert lib.rvq_dims_supported(rq.rvq_dims(1024, 64, 1024, 65)) == -2  # Q > 64
    assert lib.rvq_dims_supported(rq.rvq_dims(1024, 64, -1, 8)) == -1
    # the 8-dim code space (K <= 1024) and the normalised metric
    assert lib.rvq_dims_supported(rq.rvq_dims(768, 8, 1024, 32, rq.RVQ_METRIC_COSINE)) == 0
    assert lib.rvq_dims_supported(rq.rvq_dims(768, 8, 1024, 32, rq.RVQ_METRIC_L2)) == 0
    assert lib.rvq_dims_supported(rq.rvq_dims(768, 8, 2048, 32)) == -2   # K too large for d = 8
    assert lib.rvq_dims_supported(rq.rvq_dims(768, 16, 1024, 32)) == -2  # d neither 8 nor 64
    assert lib.rvq_dims_supported(rq.rvq_dims(1024, 64, 1024, 8, 2)) == -1  # unknown metric
    assert lib.rvq_tables_bytes(rq.rvq_dims(768, 8, 1024, 32, 1)) > 0
    # frame and output widths of the codec's Linear layers
    assert lib.rvq_dims_supported(rq.rvq_dims(1024, 64, 1024, 8, 0, 1024, 256)) == 0
    assert lib.rvq_dims_supported(rq.rvq_dims(1024, 64, 1024, 8, 0, 1000, 256)) == -2   # D_in % 16
    assert lib.rvq_dims_supported(rq.rvq_dims(1024, 64, 1024, 8, 0, 0, -16)) == -1
    w = rq.rvq_weights(1 << 20, None, 1 << 20, 1 << 20, None, None, None, None, None)
    fake = ctypes.c_void_p(1 << 20)
    # D_in != D without fc_w is rejected before any launch
    assert lib.rvq_prepare(rq.rvq_dims(1024, 64, 1024, 8, 0, 512, 0), ctypes.byref(w), fake, 1 << 40, None) == -1
    assert lib.rvq_tables_bytes(ok) > 8 * 1024 * 1024 * 4                # holds Z at least
    assert lib.rvq_encode_min_scratch_bytes(ok, 8) == 256 + 128 * 8 * 64 * 4
    assert lib.rvq_encode_scratch_bytes(ok, 100, 8) == 256 + 100 * 8 * 64 * 4
    assert lib.rvq_encode_scratch_bytes(ok, 10 ** 6, 8) <= 256 + (512 << 20)
    assert lib.rvq_encode(ok, None, None, 5, 8, None, None, 0, None) == -1
    assert lib.rvq_encode(ok, None, None, 0, 8, None, None, 0, None) == 0
    assert lib.rvq_decode(ok, None, None, 5, 0, None, None, None) == -1
    # scratch smaller than one 128-frame chunk is rejected before any launch
    fake = ctypes.c_void_p(1 << 20)
    assert lib.rvq_encode(ok, fake, fake, 1000, 8, fake, fake, 1000, None) == -1
    # misaligned pointers are rejected
    assert lib.rvq_decode(ok, fake, ctypes.c_void_p((1 << 20) + 4), 5, 8, fake, None, None) == -1
    # the no-allocation encode: host refusals before any CUDA call
    a, x, c = ctypes.c_void_p(1 << 20), ctypes.c_void_p(2 << 20), ctypes.c_void_p(3 << 20)
    assert lib.rvq_encode_static(ok, a, x, 0, 8, c, None) == 0
    assert lib.rvq_encode_static(ok, None, x, 10, 8, c, None) == -1
    assert lib.rvq_encode_static(ok, a, x, 10, 9, c, None) == -1
    assert lib.rvq_encode_static(ok, a, ctypes.c_void_p((2 << 20) + 8), 10, 8, c, None) == -1
    assert lib.rvq_encode_static(ok, a, x, 8192, 8, c, None) == -3            # 16 MiB holds 8191 frames
    d8 = rq.rvq_dims(768, 8, 1024, 32, rq.RVQ_METRIC_COSINE)
    assert lib.rvq_encode_static(d8, a, x, (rq.RVQ_STATIC_SCRATCH_BYTES - 256) // (32 * 8 * 4) + 1, 32, c,
                                 None) == -3
    # status readers and the pipeline's cancel hook
    n = ctypes.c_int64(0)
    assert lib.rvq_read_error_count(None, ctypes.byref(n), None) == -1
    assert lib.rvq_read_error_count(ctypes.c_void_p((1 << 20) + 4), ctypes.byref(n), None) == -1
    assert lib.rvq_read_status(ctypes.c_void_p((1 << 20) + 8), None) == -1
    assert lib.rvq_pipeline_set_cancel(None, rq.RVQ_CANCEL_FN(), None) == -1
    assert rq.rvq_status_string(-6) == "cancelled"
    assert rq.rvq_status_string(-5) == "device wait timed out"
    assert rq.rvq_status_string(-4) == "CUDA launch failed"
    assert "sm_103a" in rq.rvq_version()


def test_c99_consumer(lib_path, tmp_path):
    exe = tmp_path / "abi_c"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "abi_c.c"), "-o", str(exe), lib_path,
                    f"-Wl,-rpath,{os.path.dirname(lib_path)}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "abi_c: ok" in r.stdout
