"""Grammar-compressed right products y = Mx on one GB300.

The matrix is CSRV-encoded, RePair-compressed and made properly layered on
the host (``Grammar``); ``Engine`` uploads the packed grammar into a device
arena that torch allocates and runs the level-synchronous sweep in the
library's sm_103a kernels. Both are thin wrappers over the C ABI in
``include/gcsparse.h`` (``capi`` has the one-to-one bindings).
"""
from __future__ import annotations

import hashlib
import os

import importlib

import numpy as np


def __getattr__(name):
    # The binding loads libgcsparse.so; it is imported on first use so that
    # the ``build`` submodule can run before the library exists. Without the
    # library every product entry point raises ImportError (no fallback).
    if name in ("capi", "GcError"):
        mod = importlib.import_module(".capi", __name__)
        return mod if name == "capi" else mod.GcError
    raise AttributeError(name)


def _capi():
    return importlib.import_module(".capi", __name__)


def _sync(stream):
    """Wait for the work on ``stream`` (a torch stream, else the device)."""
    import torch
    if hasattr(stream, "synchronize"):
        stream.synchronize()
    else:
        torch.cuda.synchronize()


class Grammar:
    """A built grammar (host). ``Grammar(n, m, row_ptr, col, val)`` runs
    CSRV + RePair + levels + pass-through completion + packing."""

    def __init__(self, n=None, m=None, row_ptr=None, col=None, val=None, *, block_rows=0,
                 threads=0, order=0, _ptr=None):
        self._p = _ptr if _ptr is not None else _capi().gc_build(
            n, m, row_ptr, col, val, block_rows=block_rows, threads=threads, order=order)

    @classmethod
    def from_row_blocks(cls, n, m, block_rows, make_block, workers=1, threads=0, order=0) -> "Grammar":
        """Streaming build: ``make_block(r0, r1)`` returns the CSR (row_ptr
        from 0, col, val) of rows [r0, r1); each block is compressed as soon
        as it is made, ``workers`` blocks at a time (threads; the generator
        and the library release the GIL)."""
        from concurrent.futures import ThreadPoolExecutor
        capi = _capi()
        b = capi.gc_builder_create(n, m, threads=threads, order=order)
        try:
            def one(r0):
                r1 = min(n, r0 + block_rows)
                rp, col, val = make_block(r0, r1)
                capi.gc_builder_add_rows(b, r0, rp, col, val)
            starts = list(range(0, n, block_rows)) if n else []
            if workers > 1:
                with ThreadPoolExecutor(workers) as ex:
                    list(ex.map(one, starts))
            else:
                for r0 in starts:
                    one(r0)
            return cls(_ptr=capi.gc_builder_finish(b))
        finally:
            capi.gc_builder_free(b)

    @classmethod
    def load(cls, path: str) -> "Grammar":
        return cls(_ptr=_capi().gc_load(path))

    def save(self, path: str):
        _capi().gc_save(self._p, path)

    def stats(self) -> dict:
        return _capi().gc_stats(self._p)

    def widths(self) -> np.ndarray:
        return _capi().gc_widths(self._p)

    def balanced(self) -> "Grammar":
        """The same expansions as an AVL-balanced grammar (a new Grammar;
        products over it equal this one's, the level count L drops to about
        1.44 log2 of the longest rule expansion)."""
        return Grammar(_ptr=_capi().gc_balance(self._p))

    def export(self, which: str) -> np.ndarray:
        return _capi().gc_export(self._p, which)

    def layout(self, policy="f32", k_max=1, schedule="persistent") -> dict:
        """Device bytes for products under ``policy`` with up to ``k_max``
        right-hand sides; ``schedule="dataflow"`` sizes the dataflow layout."""
        if schedule == "persistent":
            return _capi().gc_layout(self._p, policy, k_max)
        return _capi().gc_layout_ex(self._p, policy, k_max, schedule)

    def __del__(self):
        p = getattr(self, "_p", None)
        if p:
            try:
                _capi().gc_free_grammar(p)
            except Exception:   # interpreter shutdown
                pass
            self._p = None


class Engine:
    """A grammar resident on a CUDA device, ready for products.

    The arena is one torch uint8 tensor of ``layout()["arena_bytes"]`` bytes;
    the library never allocates device memory itself.
    """

    def __init__(self, grammar: Grammar, policy="f32", k_max=1, device="cuda", stream=None, schedule="persistent"):
        """``schedule``: "persistent" (default), "per_level", or "dataflow"
        (k_max = 1; the dataflow sweep's own layout)."""
        import torch

        self.policy, self.k_max = policy, k_max
        st = grammar.stats()
        self.n, self.m = st["n"], st["m"]
        self.layout = grammar.layout(policy, k_max, schedule)
        self.device = torch.device(device)
        self.arena = torch.empty(max(self.layout["arena_bytes"], 256), dtype=torch.uint8,
                                 device=self.device)
        self._stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self._h = _capi().gc_upload_ex(grammar._p, policy, k_max, schedule, self.arena, self.arena.numel(),
                                       self._stream)
        self._stream.synchronize()

    @property
    def dtype(self):
        import torch
        return {"f32": torch.float32, "i64": torch.int64, "or": torch.int64, "minplus": torch.float32}[self.policy]

    def matvec(self, x, y=None, stream=None):
        """y = M x for a device tensor x of shape (m,) or (m, k)."""
        import torch
        k = 1 if x.dim() == 1 else x.shape[1]
        if y is None:
            y = torch.empty((self.n,) if x.dim() == 1 else (self.n, k), dtype=x.dtype, device=x.device)
        _capi().gc_matvec(self._h, x, y, k, stream if stream is not None else self._stream)
        return y

    def matvec_host(self, x: np.ndarray, y: np.ndarray | None = None, stream=None) -> np.ndarray:
        """Same product with host buffers (copies in and out, synchronises)."""
        k = 1 if x.ndim == 1 else x.shape[1]
        if y is None:
            y = np.empty((self.n,) if x.ndim == 1 else (self.n, k), dtype=x.dtype)
        _capi().gc_matvec_host(self._h, np.ascontiguousarray(x), y, k,
                            stream if stream is not None else self._stream)
        return y

    def reach(self, x0, max_iter=1000, stream=None):
        """Boolean fixpoint from a device int64/uint64 bitset tensor; returns (x, iterations, status)."""
        import torch
        x = torch.empty_like(x0)
        iters = torch.zeros(1, dtype=torch.int32, device=x0.device)
        st = stream if stream is not None else self._stream
        rc = _capi().gc_reach(self._h, x0, x, max_iter, iters, st)
        _sync(st)   # the call returns before its last batch and the iters write end
        return x, int(iters.item()), rc

    def sssp(self, x0, max_iter=1000, stream=None):
        """Tropical fixpoint x <- min(x, M (x) x) from a device float32 tensor
        (0 at the sources, +inf elsewhere); returns (x, iterations, status)."""
        import torch
        x = torch.empty_like(x0)
        iters = torch.zeros(1, dtype=torch.int32, device=x0.device)
        st = stream if stream is not None else self._stream
        rc = _capi().gc_sssp(self._h, x0, x, max_iter, iters, st)
        _sync(st)   # the call returns before its last batch and the iters write end
        return x, int(iters.item()), rc

    def check(self, stream=None) -> int:
        return _capi().gc_check(self._h, stream if stream is not None else self._stream)

    def launch_count(self) -> int:
        return _capi().gc_launch_count(self._h)

    @property
    def schedule(self) -> str:
        """"persistent" (grid barriers), "per_level" (a launch per level) or
        "dataflow" (per-block ready flags; handles with k_max = 1)."""
        return {0: "persistent", 1: "per_level", 2: "dataflow"}[_capi().gc_get_schedule(self._h)]

    @schedule.setter
    def schedule(self, name: str):
        _capi().gc_set_schedule(self._h, {"persistent": 0, "per_level": 1, "dataflow": 2}[name])

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            try:
                _capi().gc_free_handle(h)
            except Exception:   # interpreter shutdown
                pass
            self._h = None


class LeftEngine:
    """The left product x = M^T y of a grammar resident on a CUDA device (one
    right-hand side; gc_left_* of the C ABI), under the policy "f32", "i64",
    "or" or "minplus". The arena is one torch uint8 tensor; the library
    allocates no device memory itself."""

    def __init__(self, grammar: Grammar, policy="f32", device="cuda", stream=None):
        import torch

        st = grammar.stats()
        self.n, self.m = st["n"], st["m"]
        self.policy = policy
        self.layout = _capi().gc_left_layout(grammar._p, policy)
        self.device = torch.device(device)
        self.arena = torch.empty(max(self.layout["arena_bytes"], 256), dtype=torch.uint8, device=self.device)
        self._stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self._h = _capi().gc_left_upload(grammar._p, policy, self.arena, self.arena.numel(), self._stream)

    @property
    def dtype(self):
        import torch
        return {"f32": torch.float32, "i64": torch.int64, "or": torch.int64, "minplus": torch.float32}[self.policy]

    def matvec(self, y, x=None, stream=None):
        """x = M^T y for a device tensor y of shape (n,) (the policy's dtype;
        int64 bit patterns for "or")."""
        import torch
        if x is None:
            x = torch.empty(self.m, dtype=self.dtype, device=y.device)
        _capi().gc_left_matvec(self._h, y, x, stream if stream is not None else self._stream)
        return x

    def reach(self, x0, max_iter=1000, stream=None):
        """Forward Boolean fixpoint (policy "or") from an int64/uint64 bitset
        tensor: what the sources reach; returns (x, iterations, status)."""
        return self._fixpoint(_capi().gc_left_reach, x0, max_iter, stream)

    def sssp(self, x0, max_iter=1000, stream=None):
        """Forward tropical fixpoint (policy "minplus") from float32 distances
        (0 at the sources, +inf elsewhere); returns (x, iterations, status)."""
        return self._fixpoint(_capi().gc_left_sssp, x0, max_iter, stream)

    def _fixpoint(self, fn, x0, max_iter, stream):
        import torch
        x = torch.empty_like(x0)
        iters = torch.zeros(1, dtype=torch.int32, device=x0.device)
        st = stream if stream is not None else self._stream
        rc = fn(self._h, x0, x, max_iter, iters, st)
        _sync(st)   # the call returns before its last batch and the iters write end
        return x, int(iters.item()), rc

    def launch_count(self) -> int:
        return _capi().gc_left_launch_count(self._h)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            try:
                _capi().gc_free_left_handle(h)
            except Exception:   # interpreter shutdown
                pass
            self._h = None


def _builder_fingerprint(extra=()) -> str:
    from . import build as _b
    h = hashlib.sha256()
    for f in list(_b.BUILDER_FILES) + list(extra):
        with open(os.path.join(_b.CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def cached_grammar(key: str, make_csr, cache_dir=None, build=None, extra_sources=(), **build_kwargs) -> Grammar:
    """Build a grammar, reusing a saved copy when one exists.

    ``make_csr()`` returns (n, m, row_ptr, col, val); alternatively
    ``build()`` returns the Grammar itself (a streaming build). The file name
    combines ``key``, the build options and a hash of the builder's sources,
    so a changed builder never reuses an old file (``extra_sources`` names
    further csrc files the build depends on). A file that fails to load
    or validate is rebuilt. Set GCSPARSE_NO_CACHE=1 to always rebuild.
    """
    cache_dir = cache_dir or os.environ.get("GCSPARSE_CACHE",
                                            os.path.join(os.path.expanduser("~"), ".cache", "gcsparse"))
    tag = hashlib.sha256(repr((key, sorted(build_kwargs.items()))).encode()).hexdigest()[:16]
    path = os.path.join(cache_dir, f"{tag}-{_builder_fingerprint(extra_sources)}.gcg")
    if os.environ.get("GCSPARSE_NO_CACHE") != "1" and os.path.exists(path):
        try:
            return Grammar.load(path)
        except _capi().GcError:
            pass
    if build is not None:
        g = build()
    else:
        n, m, row_ptr, col, val = make_csr()
        g = Grammar(n, m, row_ptr, col, val, **build_kwargs)
    try:
        os.makedirs(cache_dir, exist_ok=True)
        tmp = path + f".tmp{os.getpid()}"
        g.save(tmp)
        os.replace(tmp, path)
    except (OSError, _capi().GcError):
        pass
    return g
