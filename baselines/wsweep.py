"""CPU baselines in C (``wsweep.c``), reported beside the GPU figures:
Theorem 2.3's W-array grammar sweep and the direct CSR product, each
sequential and OpenMP over the machine's host cores.

Timed baselines only (no part of the product, and not the oracle): bench.py's
CPU-baseline leg and the tests that pin these C routines use it. The C source
is compiled with gcc on first use into ``baselines/_build/`` (no part of the
product's build).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "wsweep.c")
LIB = os.path.join(HERE, "_build", "libwsweep.so")

_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        os.makedirs(os.path.dirname(LIB), exist_ok=True)
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", SRC, "-o", tmp], check=True,
                       capture_output=True)
        os.replace(tmp, LIB)
    lib = ctypes.CDLL(LIB)
    p = ctypes.c_void_p
    lib.ws_sweep.argtypes = [ctypes.c_int64, p, p, p, p, ctypes.c_int64, ctypes.c_int64, p, p, ctypes.c_int64, p, p, p,
                             p, p, p, p, ctypes.c_int]
    lib.ws_sweep.restype = ctypes.c_int
    lib.ws_csr.argtypes = [ctypes.c_int64, p, p, p, p, p, ctypes.c_int]
    lib.ws_csr.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class GrammarSweep:
    """y = M x by the W-array sweep over a grammar's exported raw arrays:
    rules (int32, 2 per rule: A_i, B_i, s >= 0 a rule, s < 0 terminal -s-1),
    rule_level (Eq. 3.1), c_off / c_sym (C), term_col / term_vidx, values."""

    def __init__(self, rules, rule_level, c_off, c_sym, term_col, term_vidx, values):
        r = np.asarray(rules, dtype=np.int32).reshape(-1, 2)
        self.a = np.ascontiguousarray(r[:, 0])
        self.b = np.ascontiguousarray(r[:, 1])
        lvl = np.asarray(rule_level, dtype=np.int64)
        self.depth = int(lvl.max()) if len(lvl) else 0
        self.by_level = np.argsort(lvl, kind="stable").astype(np.int32)
        counts = np.bincount(lvl, minlength=self.depth + 1)[1:] if len(lvl) else np.zeros(0, np.int64)
        self.level_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        self.c_off = np.asarray(c_off, dtype=np.int64)
        self.c_sym = np.asarray(c_sym, dtype=np.int32)
        self.term_col = np.asarray(term_col, dtype=np.int32)
        self.term_vidx = np.asarray(term_vidx, dtype=np.int32)
        self.V = np.asarray(values, dtype=np.float64)
        self.n = len(self.c_off) - 1
        self.W = np.empty(max(1, len(self.a)), dtype=np.float64)
        self.T = np.empty(max(1, len(self.term_col)), dtype=np.float64)

    @classmethod
    def from_grammar(cls, G):
        """From a built grammar_compressed_sparse_gb300.Grammar (host arrays only)."""
        return cls(*(G.export(a) for a in ("rules", "rule_level", "c_off", "c_sym", "term_col", "term_vidx", "values")))

    def __call__(self, x, threads=1):
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.empty(self.n, dtype=np.float64)
        rc = _load().ws_sweep(len(self.a), _ptr(self.a), _ptr(self.b), _ptr(self.level_off), _ptr(self.by_level),
                              self.depth, self.n, _ptr(self.c_off), _ptr(self.c_sym), len(self.term_col),
                              _ptr(self.term_col), _ptr(self.term_vidx), _ptr(self.V), _ptr(x), _ptr(y),
                              _ptr(self.W), _ptr(self.T), int(threads))
        if rc != 0:
            raise ValueError("bad thread count")
        return y

    def rate(self, x, threads, seconds):
        """Products per second over about ``seconds`` of repeated sweeps (at least one)."""
        done, t0 = 0, time.perf_counter()
        while True:
            self(x, threads)
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return done / el


class CsrProduct:
    """y = M x from the uncompressed CSR (int64 row_ptr, int32 col, float32
    val) in float64, rows in parallel: the CSR CPU baseline."""

    def __init__(self, row_ptr, col, val):
        self.rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
        self.col = np.ascontiguousarray(col, dtype=np.int32)
        self.val = np.ascontiguousarray(val, dtype=np.float32)
        self.n = len(self.rp) - 1

    def __call__(self, x, threads=1):
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.empty(self.n, dtype=np.float64)
        if _load().ws_csr(self.n, _ptr(self.rp), _ptr(self.col), _ptr(self.val), _ptr(x), _ptr(y), int(threads)) != 0:
            raise ValueError("bad thread count")
        return y

    rate = GrammarSweep.rate
