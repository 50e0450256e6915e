"""O1: the right product computed directly from the uncompressed matrix.

The grammar method reaches y = Mx exactly (up to rounding order): Lemma 2.1
(additivity), Lemma 2.2 (rows as roots) and Theorem 2.3 of the pages' Sec. 2
prove it, and pass-through nodes are identities (Sec. 4.2). So the oracle for
every policy is the plain definition y[i] = (+)_j M[i][j] (x) x[j], evaluated
one row at a time from CSR.

Precision: float64 for the (+, x) semiring (the pages state agreement "within
float precision", Sec. 6 "Correctness"); exact int64 for integer inputs;
bitwise OR/AND for the Boolean semiring (Sec. 5); float32 for the tropical
(min, +) semiring, which the pages check bit for bit (Sec. 6): each sum
M[i][j] + x[j] is rounded to float32 once and min is exact.
"""
from __future__ import annotations

import numpy as np


def matvec_f64(row_ptr, col, val, x):
    """y = Mx and b = |M||x| in float64.

    ``x`` is (m,) or (m, k) (k right-hand sides, Appendix A "Batched
    evaluation"); y and b have shape (n,) or (n, k). b is the scale the
    float32 tolerance is stated against: |y_i - y_ref_i| <= tol * b_i.
    """
    x = np.asarray(x, dtype=np.float64)
    n = len(row_ptr) - 1
    shape = (n,) if x.ndim == 1 else (n, x.shape[1])
    y = np.zeros(shape, dtype=np.float64)
    b = np.zeros(shape, dtype=np.float64)
    for i in range(n):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        v = np.asarray(val[s:e], dtype=np.float64)
        xs = x[np.asarray(col[s:e], dtype=np.int64)]
        y[i] = v @ xs
        b[i] = np.abs(v) @ np.abs(xs)
    return y, b


def matvec_i64(row_ptr, col, val, x):
    """Exact integer y = Mx (int64); values and x must be integers."""
    x = np.asarray(x, dtype=np.int64)
    v_all = np.asarray(val)
    if not np.all(np.floor(v_all) == v_all):
        raise ValueError("integer product needs integer matrix values")
    n = len(row_ptr) - 1
    shape = (n,) if x.ndim == 1 else (n, x.shape[1])
    y = np.zeros(shape, dtype=np.int64)
    for i in range(n):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        v = v_all[s:e].astype(np.int64)
        y[i] = v @ x[np.asarray(col[s:e], dtype=np.int64)]
    return y


def matvec_or(row_ptr, col, x):
    """Boolean semiring (OR, AND) on 64-bit bitsets (Sec. 5).

    Every stored entry is a true edge, so the leaf map is the identity on x
    and y[i] = OR over j in row i of x[j]; an empty row gives the OR-identity 0.
    (numpy's OR-reduction over each row's slice of x[col], so that graphs with
    10^8 edges finish in seconds.)
    """
    x = np.asarray(x, dtype=np.uint64)
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    n = len(row_ptr) - 1
    y = np.zeros(n, dtype=np.uint64)
    nonempty = row_ptr[1:] > row_ptr[:-1]
    if nonempty.any():
        y[nonempty] = np.bitwise_or.reduceat(x[np.asarray(col, dtype=np.int64)], row_ptr[:-1][nonempty])
    return y


def matvec_minplus(row_ptr, col, val, x):
    """Tropical semiring (min, +) (Sec. 5: one pass is one Bellman-Ford edge
    relaxation): y[i] = min over the stored entries M[i][j] of M[i][j] + x[j].

    The leaf map is the addition, rounded to float32; min needs no rounding,
    so the result is the same whatever order the minimum is taken in. A row
    with no stored entry gets the min-identity +inf (the semiring zero, Sec. 5).
    ``x`` is (m,) or (m, k), float32 values without NaN. (numpy's
    min-reduction over each row's slice, so that graphs with 10^8 edges
    finish in seconds.)
    """
    x = np.asarray(x, dtype=np.float32)
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    n = len(row_ptr) - 1
    shape = (n,) if x.ndim == 1 else (n, x.shape[1])
    y = np.full(shape, np.inf, dtype=np.float32)
    nonempty = row_ptr[1:] > row_ptr[:-1]
    if nonempty.any():
        v = np.asarray(val, dtype=np.float32)
        xs = x[np.asarray(col, dtype=np.int64)]
        t = (v + xs) if x.ndim == 1 else (v[:, None] + xs)    # float32 sums
        y[nonempty] = np.minimum.reduceat(t, row_ptr[:-1][nonempty], axis=0)
    return y


def left_matvec_f64(row_ptr, col, val, y, m):
    """The left product x^T = y^T M, i.e. x = M^T y, and b = |M|^T |y| in
    float64 (the dual product; the pages leave it to future work, Sec. 8).

    x[j] = sum over the stored entries M[i][j] of M[i][j] * y[i], one row at a
    time: row i adds M[i][j] * y[i] to x[j] for each of its columns j. ``y``
    is (n,); x and b have shape (m,).
    """
    y = np.asarray(y, dtype=np.float64)
    x = np.zeros(m, dtype=np.float64)
    b = np.zeros(m, dtype=np.float64)
    for i in range(len(row_ptr) - 1):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        cols = np.asarray(col[s:e], dtype=np.int64)
        v = np.asarray(val[s:e], dtype=np.float64)
        np.add.at(x, cols, v * y[i])
        np.add.at(b, cols, np.abs(v) * abs(y[i]))
    return x, b


def left_matvec_i64(row_ptr, col, val, y, m):
    """Exact integer left product x = M^T y (int64): x[j] = sum of M[i][j] * y[i]."""
    y = np.asarray(y, dtype=np.int64)
    v_all = np.asarray(val)
    if not np.all(np.floor(v_all) == v_all):
        raise ValueError("integer product needs integer matrix values")
    x = np.zeros(m, dtype=np.int64)
    for i in range(len(row_ptr) - 1):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        np.add.at(x, np.asarray(col[s:e], dtype=np.int64), v_all[s:e].astype(np.int64) * y[i])
    return x


def left_matvec_or(row_ptr, col, y, m):
    """Boolean left product (Sec. 5 semiring): x[j] = OR of y[i] over the
    stored entries (i, j); with y a frontier of 64-bit source sets, one
    forward step along the edges i -> j."""
    y = np.asarray(y, dtype=np.uint64)
    x = np.zeros(m, dtype=np.uint64)
    for i in range(len(row_ptr) - 1):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        np.bitwise_or.at(x, np.asarray(col[s:e], dtype=np.int64), y[i])
    return x


def left_matvec_minplus(row_ptr, col, val, y, m):
    """Tropical left product: x[j] = min of M[i][j] + y[i] over the stored
    entries (i, j), each sum rounded to float32, +inf for a column no row
    uses; with y distances, one forward Bellman-Ford relaxation."""
    y = np.asarray(y, dtype=np.float32)
    x = np.full(m, np.inf, dtype=np.float32)
    for i in range(len(row_ptr) - 1):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        np.minimum.at(x, np.asarray(col[s:e], dtype=np.int64), np.asarray(val[s:e], dtype=np.float32) + y[i])
    return x


def within_tolerance(y, y_ref, b, tol):
    """The float32 acceptance rule: |y - y_ref| <= tol * b elementwise, and
    y exactly 0 where b is 0 (an all-zero row or all-zero x support)."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    ok = err <= tol * b
    ok &= np.where(b == 0, y == 0, True)
    return bool(np.all(ok)), float(np.max(err / np.where(b > 0, b, 1.0))) if err.size else 0.0
