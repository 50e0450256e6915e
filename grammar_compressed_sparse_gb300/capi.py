"""ctypes binding of libgcsparse.so, one Python function per C entry point
(same names, argument marshalling only; every step of the product runs in the
library). numpy arrays are passed for host buffers, torch tensors (or raw
integer addresses) for device buffers, and a torch stream (or an integer
cudaStream_t) for streams.

The library must be built (``grammar_compressed_sparse_gb300.build.build()``);
importing this module raises if it is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

if not os.path.exists(_build.LIB):
    raise ImportError(f"libgcsparse.so is not built ({_build.LIB}); run "
                      "grammar_compressed_sparse_gb300.build.build()")

_lib = ctypes.CDLL(_build.LIB)

GC_OK, GC_ERR_ARG, GC_ERR_OOM, GC_ERR_CUDA, GC_ERR_INVALID_GRAMMAR = 0, -1, -2, -3, -4
GC_ERR_UNSUPPORTED, GC_ERR_TIMEOUT, GC_ERR_NOT_CONVERGED, GC_ERR_IO = -5, -6, -7, -8
STATUS_NAMES = {0: "GC_OK", -1: "GC_ERR_ARG", -2: "GC_ERR_OOM", -3: "GC_ERR_CUDA",
                -4: "GC_ERR_INVALID_GRAMMAR", -5: "GC_ERR_UNSUPPORTED", -6: "GC_ERR_TIMEOUT",
                -7: "GC_ERR_NOT_CONVERGED", -8: "GC_ERR_IO"}

GC_F32_SUM, GC_I64_SUM, GC_BOOL_OR, GC_F32_MIN_PLUS = 0, 1, 2, 3
GC_SCHED_PERSISTENT, GC_SCHED_PER_LEVEL, GC_SCHED_DATAFLOW = 0, 1, 2
POLICIES = {"f32": GC_F32_SUM, "i64": GC_I64_SUM, "or": GC_BOOL_OR, "minplus": GC_F32_MIN_PLUS}

ARRAYS = {  # gc_array enum -> numpy dtype
    "values": (0, np.float32), "term_col": (1, np.int32), "term_vidx": (2, np.int32),
    "rules": (3, np.int32), "c_off": (4, np.int64), "c_sym": (5, np.int32),
    "rule_level": (6, np.int32), "lvl_off": (7, np.int64), "nodes": (8, np.int32),
    "lvl_roots": (9, np.int64), "root_off": (10, np.int64), "c_ref": (11, np.int32),
    "node_id": (12, np.int32),
}


class GcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.gc_last_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")


class BuildOpts(ctypes.Structure):
    _fields_ = [("block_rows", ctypes.c_int64), ("threads", ctypes.c_int32), ("order", ctypes.c_int32)]


class GrammarStats(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in
                ("n", "m", "nnz", "n_values", "n_terminals", "n_rules", "n_pass", "n_nodes",
                 "depth", "max_width", "c_len", "n_roots", "n_blocks")] + \
               [("repair_seconds", ctypes.c_double), ("layer_seconds", ctypes.c_double)]


class ArenaLayout(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in
                ("arena_bytes", "grammar_bytes", "scratch_bytes", "staging_bytes", "csr_bytes")]


_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
_sig = {
    "gc_last_error": ([], ctypes.c_char_p),
    "gc_version": ([], ctypes.c_char_p),
    "gc_build": ([_i64, _i64, _vp, _vp, _vp, ctypes.POINTER(BuildOpts), ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_stats": ([_vp, ctypes.POINTER(GrammarStats)], ctypes.c_int),
    "gc_update": ([ctypes.c_int, _vp, _vp, ctypes.c_int64, _vp, _vp], ctypes.c_int),
    "gc_balance": ([_vp, ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_widths": ([_vp, _vp, _i64], ctypes.c_int),
    "gc_export_size": ([_vp, ctypes.c_int, ctypes.POINTER(_i64)], ctypes.c_int),
    "gc_export": ([_vp, ctypes.c_int, _vp, _i64], ctypes.c_int),
    "gc_layout": ([_vp, ctypes.c_int, _i32, ctypes.POINTER(ArenaLayout)], ctypes.c_int),
    "gc_upload": ([_vp, ctypes.c_int, _i32, _vp, _i64, _vp, ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_layout_ex": ([_vp, ctypes.c_int, _i32, _i32, ctypes.POINTER(ArenaLayout)], ctypes.c_int),
    "gc_upload_ex": ([_vp, ctypes.c_int, _i32, _i32, _vp, _i64, _vp, ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_matvec": ([_vp, _vp, _vp, _i32, _vp], ctypes.c_int),
    "gc_matvec_host": ([_vp, _vp, _vp, _i32, _vp], ctypes.c_int),
    "gc_matvec_static": ([_vp, _vp, _vp, _i32, _vp], ctypes.c_int),
    "gc_reach": ([_vp, _vp, _vp, _i32, _vp, _vp], ctypes.c_int),
    "gc_sssp": ([_vp, _vp, _vp, _i32, _vp, _vp], ctypes.c_int),
    "gc_check": ([_vp, _vp], ctypes.c_int),
    "gc_launch_count": ([_vp, ctypes.POINTER(_i64)], ctypes.c_int),
    "gc_set_schedule": ([_vp, _i32], ctypes.c_int),
    "gc_get_schedule": ([_vp, ctypes.POINTER(_i32)], ctypes.c_int),
    "gc_debug_inject": ([_vp, _i32, _i64], ctypes.c_int),
    "gc_save": ([_vp, ctypes.c_char_p], ctypes.c_int),
    "gc_load": ([ctypes.c_char_p, ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_free_grammar": ([_vp], None),
    "gc_builder_create": ([_i64, _i64, ctypes.POINTER(BuildOpts), ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_builder_add_rows": ([_vp, _i64, _i64, _vp, _vp, _vp], ctypes.c_int),
    "gc_builder_finish": ([_vp, ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_builder_free": ([_vp], None),
    "gc_free_handle": ([_vp], None),
    "gc_left_layout": ([_vp, ctypes.c_int, ctypes.POINTER(ArenaLayout)], ctypes.c_int),
    "gc_left_upload": ([_vp, ctypes.c_int, _vp, _i64, _vp, ctypes.POINTER(_vp)], ctypes.c_int),
    "gc_left_matvec": ([_vp, _vp, _vp, _vp], ctypes.c_int),
    "gc_left_launch_count": ([_vp, ctypes.POINTER(_i64)], ctypes.c_int),
    "gc_left_reach": ([_vp, _vp, _vp, _i32, _vp, _vp], ctypes.c_int),
    "gc_left_sssp": ([_vp, _vp, _vp, _i32, _vp, _vp], ctypes.c_int),
    "gc_free_left_handle": ([_vp], None),
}
for _name, (_args, _res) in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_sig)


def _check(rc: int, where: str):
    if rc != GC_OK:
        raise GcError(rc, where)


def _addr(t) -> int | None:
    """Address of a numpy array, torch tensor or raw integer (None stays None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def gc_version() -> str:
    return _lib.gc_version().decode()


def gc_last_error() -> str:
    return _lib.gc_last_error().decode()


def gc_build(n, m, row_ptr, col, val=None, block_rows=0, threads=0, order=0) -> int:
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
    col = np.ascontiguousarray(col, dtype=np.int32)
    val = None if val is None else np.ascontiguousarray(val, dtype=np.float32)
    out = _vp()
    opts = BuildOpts(block_rows, threads, order)
    _check(_lib.gc_build(n, m, _addr(row_ptr), _addr(col), _addr(val), ctypes.byref(opts),
                         ctypes.byref(out)), "gc_build")
    return out.value


def gc_balance(g):
    out = _vp()
    _check(_lib.gc_balance(g, ctypes.byref(out)), "gc_balance")
    return out.value


def gc_stats(g) -> dict:
    s = GrammarStats()
    _check(_lib.gc_stats(g, ctypes.byref(s)), "gc_stats")
    return {f: getattr(s, f) for f, _ in GrammarStats._fields_}


def gc_widths(g) -> np.ndarray:
    L = gc_stats(g)["depth"]
    w = np.zeros(max(L, 1), dtype=np.int64)
    _check(_lib.gc_widths(g, _addr(w), len(w)), "gc_widths")
    return w[:L]


def gc_export(g, which: str) -> np.ndarray:
    code, dt = ARRAYS[which]
    nb = _i64()
    _check(_lib.gc_export_size(g, code, ctypes.byref(nb)), "gc_export_size")
    out = np.empty(nb.value // np.dtype(dt).itemsize, dtype=dt)
    _check(_lib.gc_export(g, code, _addr(out) if out.size else None, nb.value), "gc_export")
    return out


def gc_layout(g, policy="f32", k_max=1) -> dict:
    lay = ArenaLayout()
    _check(_lib.gc_layout(g, POLICIES[policy], k_max, ctypes.byref(lay)), "gc_layout")
    return {f: getattr(lay, f) for f, _ in ArenaLayout._fields_}


def gc_upload(g, policy, k_max, arena, arena_bytes, stream=None) -> int:
    out = _vp()
    _check(_lib.gc_upload(g, POLICIES[policy], k_max, _addr(arena), arena_bytes, _stream(stream),
                          ctypes.byref(out)), "gc_upload")
    return out.value


SCHEDULES = {"persistent": GC_SCHED_PERSISTENT, "per_level": GC_SCHED_PER_LEVEL, "dataflow": GC_SCHED_DATAFLOW}


def gc_layout_ex(g, policy="f32", k_max=1, schedule="persistent") -> dict:
    lay = ArenaLayout()
    _check(_lib.gc_layout_ex(g, POLICIES[policy], k_max, SCHEDULES[schedule], ctypes.byref(lay)), "gc_layout_ex")
    return {f: getattr(lay, f) for f, _ in ArenaLayout._fields_}


def gc_upload_ex(g, policy, k_max, schedule, arena, arena_bytes, stream=None) -> int:
    out = _vp()
    _check(_lib.gc_upload_ex(g, POLICIES[policy], k_max, SCHEDULES[schedule], _addr(arena), arena_bytes,
                             _stream(stream), ctypes.byref(out)), "gc_upload_ex")
    return out.value


def gc_matvec(h, x, y, k=1, stream=None):
    _check(_lib.gc_matvec(h, _addr(x), _addr(y), k, _stream(stream)), "gc_matvec")


def gc_matvec_host(h, x, y, k=1, stream=None):
    _check(_lib.gc_matvec_host(h, _addr(x), _addr(y), k, _stream(stream)), "gc_matvec_host")


def gc_matvec_static(h, x, y, k=1, stream=None):
    _check(_lib.gc_matvec_static(h, _addr(x), _addr(y), k, _stream(stream)), "gc_matvec_static")


GC_STATIC_SCRATCH_BYTES = 32 << 20


def gc_reach(h, x0, x, max_iter, iters, stream=None) -> int:
    """Returns the status (GC_OK or GC_ERR_NOT_CONVERGED); raises on anything else."""
    rc = _lib.gc_reach(h, _addr(x0), _addr(x), max_iter, _addr(iters), _stream(stream))
    if rc not in (GC_OK, GC_ERR_NOT_CONVERGED):
        raise GcError(rc, "gc_reach")
    return rc


def gc_update(policy, x, y, n, changed, stream=None):
    _check(_lib.gc_update(POLICIES[policy], _addr(x), _addr(y), n, _addr(changed), _stream(stream)), "gc_update")


def gc_sssp(h, x0, x, max_iter, iters, stream=None) -> int:
    """Returns the status (GC_OK or GC_ERR_NOT_CONVERGED); raises on anything else."""
    rc = _lib.gc_sssp(h, _addr(x0), _addr(x), max_iter, _addr(iters), _stream(stream))
    if rc not in (GC_OK, GC_ERR_NOT_CONVERGED):
        raise GcError(rc, "gc_sssp")
    return rc


def gc_check(h, stream=None) -> int:
    return _lib.gc_check(h, _stream(stream))


def gc_launch_count(h) -> int:
    v = _i64()
    _check(_lib.gc_launch_count(h, ctypes.byref(v)), "gc_launch_count")
    return v.value


def gc_set_schedule(h, schedule: int):
    _check(_lib.gc_set_schedule(h, schedule), "gc_set_schedule")


def gc_get_schedule(h) -> int:
    v = _i32()
    _check(_lib.gc_get_schedule(h, ctypes.byref(v)), "gc_get_schedule")
    return v.value


def gc_debug_inject(h, what: int, timeout_cycles: int):
    _check(_lib.gc_debug_inject(h, what, timeout_cycles), "gc_debug_inject")


def gc_save(g, path: str):
    _check(_lib.gc_save(g, path.encode()), "gc_save")


def gc_load(path: str) -> int:
    out = _vp()
    _check(_lib.gc_load(path.encode(), ctypes.byref(out)), "gc_load")
    return out.value


def gc_builder_create(n, m, threads=0, order=0) -> int:
    out = _vp()
    opts = BuildOpts(0, threads, order)
    _check(_lib.gc_builder_create(n, m, ctypes.byref(opts), ctypes.byref(out)), "gc_builder_create")
    return out.value


def gc_builder_add_rows(b, r0, row_ptr, col, val=None):
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
    col = np.ascontiguousarray(col, dtype=np.int32)
    val = None if val is None else np.ascontiguousarray(val, dtype=np.float32)
    _check(_lib.gc_builder_add_rows(b, r0, len(row_ptr) - 1, _addr(row_ptr), _addr(col), _addr(val)),
           "gc_builder_add_rows")


def gc_builder_finish(b) -> int:
    out = _vp()
    _check(_lib.gc_builder_finish(b, ctypes.byref(out)), "gc_builder_finish")
    return out.value


def gc_builder_free(b):
    _lib.gc_builder_free(b)


def gc_free_grammar(g):
    _lib.gc_free_grammar(g)


def gc_free_handle(h):
    _lib.gc_free_handle(h)


def gc_left_layout(g, policy="f32") -> dict:
    lay = ArenaLayout()
    _check(_lib.gc_left_layout(g, POLICIES[policy], ctypes.byref(lay)), "gc_left_layout")
    return {f: getattr(lay, f) for f, _ in ArenaLayout._fields_}


def gc_left_upload(g, policy, arena, arena_bytes, stream=None) -> int:
    h = _vp()
    _check(_lib.gc_left_upload(g, POLICIES[policy], _addr(arena), arena_bytes, _stream(stream), ctypes.byref(h)),
           "gc_left_upload")
    return h.value


def gc_left_matvec(h, y, x, stream=None):
    _check(_lib.gc_left_matvec(h, _addr(y), _addr(x), _stream(stream)), "gc_left_matvec")


def gc_left_launch_count(h) -> int:
    v = _i64()
    _check(_lib.gc_left_launch_count(h, ctypes.byref(v)), "gc_left_launch_count")
    return v.value


def gc_left_reach(h, x0, x, max_iter, iters, stream=None) -> int:
    """Returns the status (GC_OK or GC_ERR_NOT_CONVERGED); raises on anything else."""
    rc = _lib.gc_left_reach(h, _addr(x0), _addr(x), max_iter, _addr(iters), _stream(stream))
    if rc not in (GC_OK, GC_ERR_NOT_CONVERGED):
        raise GcError(rc, "gc_left_reach")
    return rc


def gc_left_sssp(h, x0, x, max_iter, iters, stream=None) -> int:
    """Returns the status (GC_OK or GC_ERR_NOT_CONVERGED); raises on anything else."""
    rc = _lib.gc_left_sssp(h, _addr(x0), _addr(x), max_iter, _addr(iters), _stream(stream))
    if rc not in (GC_OK, GC_ERR_NOT_CONVERGED):
        raise GcError(rc, "gc_left_sssp")
    return rc


def gc_free_left_handle(h):
    _lib.gc_free_left_handle(h)
