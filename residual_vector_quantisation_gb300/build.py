"""Compile the RVQ CUDA library (librvq.so) for sm_103a with nvcc.

Each translation unit under csrc/ is compiled in parallel with
  nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo
and linked into _build/librvq.so, which exports only the rvq_* symbols of
include/rvq.h.  A stamp of the sources and flags decides whether to rebuild.

    python -m residual_vector_quantisation_gb300.build [--force] [--verbose]
"""

from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "librvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the RVQ CUDA library cannot be built")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp(extra_flags) -> str:
    h = hashlib.sha256()
    for path in sources() + sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))) \
            + [os.path.join(INCLUDE, "rvq.h")]:
        h.update(path.encode())
        h.update(open(path, "rb").read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def build_library(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    stamp_path = os.path.join(BUILD, "librvq.stamp")
    stamp = _stamp(extra_flags)
    if not force and os.path.exists(LIB) and os.path.exists(stamp_path) and open(stamp_path).read() == stamp:
        return LIB
    cc = nvcc()
    objs = []
    cmds = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=min(8, len(cmds))) as ex:
        for cmd, r in ex.map(run, cmds):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(link) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("linking librvq.so failed")
    os.replace(tmp, LIB)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
