"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This module only makes inputs (matrices, graphs, vectors). It contains none of
the grammar-compressed product's arithmetic, so both sides can use it without
sharing any of the method's code. The generators themselves are in ``gen.c``
(counter-based hashing, so any row block can be regenerated independently);
``build()`` compiles it with gcc on first use.

Workloads (the pages measure on 1000 Genomes / msprime panels and a Software
Heritage graph, none of which is available; these seeded stand-ins have the
shapes and value structure described for the genotype and graph cases):

* ``GENO_SMALL``  1,000 x 2,000 genotypes, 20 founders, switch = mutation = 1e-3
* ``GENO_MEDIUM`` 10,000 x 50,000, 100 founders, switch = mutation = 1e-3
* ``GENO_LARGE``  50,000 x 200,000, 500 founders, switch = mutation = 5e-4,
  compressed per 5,000-row block
* ``GRAPH``       2,000,000-node copy-model graph, 100 initial nodes with 100
  targets each, 5% edits, 64 reachability sources
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libgcsynth.so")
_lock = threading.Lock()
_lib = None

GENO_SMALL = dict(n=1_000, m=2_000, founders=20, switch=1e-3, mutation=1e-3, seed=0)
GENO_MEDIUM = dict(n=10_000, m=50_000, founders=100, switch=1e-3, mutation=1e-3, seed=0)
GENO_LARGE = dict(n=50_000, m=200_000, founders=500, switch=5e-4, mutation=5e-4, seed=0,
                  block_rows=5_000)
GRAPH = dict(nodes=2_000_000, n0=100, d0=100, p_edit=0.05, seed=0, sources=64)


def build(force: bool = False) -> str:
    """Compile gen.c into libgcsynth.so next to it (idempotent)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, u64, dbl, vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64,
                                  ctypes.c_double, ctypes.c_void_p)
        lib.gcs_genotype_dense.argtypes = [i64, i32, dbl, dbl, u64, i64, i64, vp]
        lib.gcs_genotype_dense.restype = ctypes.c_int
        lib.gcs_genotype_csr.argtypes = [i64, i32, dbl, dbl, u64, i64, i64, vp, vp, vp, vp]
        lib.gcs_genotype_csr.restype = ctypes.c_int
        lib.gcs_dense_row_nnz.argtypes = [vp, i64, i64, vp]
        lib.gcs_dense_row_nnz.restype = None
        lib.gcs_dense_to_csr.argtypes = [vp, i64, i64, vp, vp, vp]
        lib.gcs_dense_to_csr.restype = None
        lib.gcs_copy_model.argtypes = [i32, i32, i32, dbl, u64, vp, vp]
        lib.gcs_copy_model.restype = i64
        lib.gcs_sources.argtypes = [i32, i32, u64, vp]
        lib.gcs_sources.restype = ctypes.c_int
        lib.gcs_hash3.argtypes = [u64, u64, u64, u64]
        lib.gcs_hash3.restype = u64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def genotype_dense(n, m, founders, switch, mutation, seed, r0=0, r1=None, **_):
    """Dense uint8 genotype rows [r0, r1) (values 0/1/2)."""
    r1 = n if r1 is None else r1
    out = np.empty((r1 - r0, m), dtype=np.uint8)
    if _load().gcs_genotype_dense(m, founders, switch, mutation, seed, r0, r1, _ptr(out)) != 0:
        raise RuntimeError("genotype generator rejected its arguments")
    return out


def dense_to_csr(d: np.ndarray):
    """CSR (int64 row_ptr, int32 col, float32 val) of a dense uint8 block."""
    d = np.ascontiguousarray(d, dtype=np.uint8)
    rows, m = d.shape
    nnz = np.empty(rows, dtype=np.int64)
    lib = _load()
    lib.gcs_dense_row_nnz(_ptr(d), rows, m, _ptr(nnz))
    row_ptr = np.zeros(rows + 1, dtype=np.int64)
    np.cumsum(nnz, out=row_ptr[1:])
    col = np.empty(int(row_ptr[-1]), dtype=np.int32)
    val = np.empty(int(row_ptr[-1]), dtype=np.float32)
    lib.gcs_dense_to_csr(_ptr(d), rows, m, _ptr(row_ptr), _ptr(col), _ptr(val))
    return row_ptr, col, val


def genotype_csr(n, m, founders, switch, mutation, seed, r0=0, r1=None, **_):
    """CSR (int64 row_ptr from 0, int32 col, float32 val) of genotype rows [r0, r1)."""
    r1 = n if r1 is None else r1
    lib = _load()
    nnz = np.empty(r1 - r0, dtype=np.int64)
    if lib.gcs_genotype_csr(m, founders, switch, mutation, seed, r0, r1, _ptr(nnz), None, None, None) != 0:
        raise RuntimeError("genotype generator rejected its arguments")
    row_ptr = np.zeros(r1 - r0 + 1, dtype=np.int64)
    np.cumsum(nnz, out=row_ptr[1:])
    col = np.empty(int(row_ptr[-1]), dtype=np.int32)
    val = np.empty(int(row_ptr[-1]), dtype=np.float32)
    if lib.gcs_genotype_csr(m, founders, switch, mutation, seed, r0, r1, None, _ptr(row_ptr),
                            _ptr(col), _ptr(val)) != 0:
        raise RuntimeError("genotype generator rejected its arguments")
    return row_ptr, col, val


def beta(m: int, seed: int, k: int = 1) -> np.ndarray:
    """Effect sizes ~ N(0,1) as float32: shape (m,) for k == 1, else (m, k) row-major."""
    g = np.random.default_rng(seed)
    v = g.standard_normal(m * k, dtype=np.float32)
    return v if k == 1 else v.reshape(m, k)


def copy_model_graph(nodes, n0, d0, p_edit, seed, **_):
    """Copy-model adjacency as CSR (int64 row_ptr, int32 col), rows sorted, no duplicates."""
    row_ptr = np.empty(nodes + 1, dtype=np.int64)
    col = np.empty(int(nodes) * int(d0), dtype=np.int32)
    e = _load().gcs_copy_model(nodes, n0, d0, p_edit, seed, _ptr(row_ptr), _ptr(col))
    if e < 0:
        raise RuntimeError("copy-model generator rejected its arguments")
    return row_ptr, col[:e].copy()


def sources(nodes: int, count: int, seed: int) -> np.ndarray:
    """``count`` distinct uniform source nodes."""
    out = np.empty(count, dtype=np.int32)
    if _load().gcs_sources(nodes, count, seed, _ptr(out)) != 0:
        raise RuntimeError("bad source request")
    return out


def frontier(nodes: int, srcs: np.ndarray) -> np.ndarray:
    """uint64 bitset per node: bit b set at node srcs[b]."""
    x = np.zeros(nodes, dtype=np.uint64)
    for b, s in enumerate(srcs):
        x[s] |= np.uint64(1) << np.uint64(b)
    return x


def target_lengths(col: np.ndarray, nodes: int, seed: int, hi: int = 9) -> np.ndarray:
    """Edge lengths for shortest-path workloads, as float32: edge i -> j gets
    the length of its target j, an integer drawn uniformly from 1..hi per node.
    Copied adjacency lists keep their (column, length) pairs, so a copy-model
    graph stays as repetitive as without lengths; integer lengths keep every
    path length exact in float32 below 2^24."""
    per_node = np.random.default_rng(seed).integers(1, hi + 1, nodes)
    return per_node[np.asarray(col, dtype=np.int64)].astype(np.float32)


def frontier_distances(nodes: int, srcs: np.ndarray) -> np.ndarray:
    """float32 distances before the first relaxation: 0 at the sources, +inf elsewhere."""
    x = np.full(nodes, np.inf, dtype=np.float32)
    x[np.asarray(srcs, dtype=np.int64)] = 0.0
    return x


def random_sparse(n: int, m: int, density: float, values, seed: int):
    """Small seeded sparse matrix as CSR with values drawn from ``values``.

    Each entry is non-zero with probability ``density``; zero is never drawn
    as a value. Used for tiny brute-force cases.
    """
    g = np.random.default_rng(seed)
    mask = g.random((n, m)) < density
    vals = np.asarray(values, dtype=np.float32)
    dense = np.where(mask, vals[g.integers(0, len(vals), size=(n, m))], np.float32(0))
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum((dense != 0).sum(1), out=row_ptr[1:])
    r, c = np.nonzero(dense)
    return row_ptr, c.astype(np.int32), dense[r, c].astype(np.float32), dense
