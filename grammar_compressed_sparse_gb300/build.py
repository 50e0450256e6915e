"""Build libgcsparse.so in-tree: host C++ (g++) + sm_103a CUDA (nvcc), linked
with the static CUDA runtime. Objects go to ``_build/`` at the repo root.

    python -m grammar_compressed_sparse_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgcsparse.so")

HOST_SOURCES = ["csrv.cpp", "repair.cpp", "layer.cpp", "balance.cpp", "capi_host.cpp"]
CUDA_SOURCES = ["engine.cu", "left.cu"]
HEADERS = ["common.hpp", "layout.hpp", "flow.hpp", "loop.hpp", "policy.cuh", "left.hpp"]
# what a saved grammar depends on (the builder and its file format); a
# balanced grammar adds balance.cpp (cached_grammar's extra_sources)
BUILDER_FILES = ["csrv.cpp", "repair.cpp", "layer.cpp", "capi_host.cpp", "common.hpp", "layout.hpp"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

_lock = threading.Lock()


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgcsparse.so")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in HOST_SOURCES + CUDA_SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "gcsparse.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libgcsparse.so if any source is newer (idempotent)."""
    with _lock:
        if not force and up_to_date():
            return LIB
        os.makedirs(BUILD, exist_ok=True)
        nvcc = _nvcc()
        common = ["-O3", "-std=c++17", f"-I{INCLUDE}"]
        jobs = []
        for src in HOST_SOURCES:
            obj = os.path.join(BUILD, src + ".o")
            jobs.append((["g++", *common, "-fPIC", "-fopenmp", "-Wall", "-Wno-unknown-pragmas",
                          "-c", os.path.join(CSRC, src), "-o", obj], obj))
        for src in CUDA_SOURCES:
            obj = os.path.join(BUILD, src + ".o")
            jobs.append(([nvcc, *common, ARCH, "-lineinfo", "-Xptxas", "-v",
                          "-Xcompiler", "-fPIC,-fopenmp", "-c", os.path.join(CSRC, src), "-o", obj], obj))
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            logs = list(ex.map(lambda j: _run(j[0]), jobs))
        if verbose:
            for log in logs:
                sys.stderr.write(log)
        tmp = LIB + f".tmp{os.getpid()}"
        _run([nvcc, "-shared", ARCH, "-o", tmp, *[j[1] for j in jobs], "-Xcompiler", "-fopenmp", "-lgomp"])
        os.replace(tmp, LIB)
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            f.write("".join(logs))
        return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
