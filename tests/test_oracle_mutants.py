"""Plant plausible mistakes in the oracle and check that its pins notice.

Each mutant replaces one oracle function by a copy with a single slip (a
dropped term, min for max, an off-by-one, a per-edge instead of shared
pass-through chain, AND for OR). The pin tests in test_oracle_pins.py are
then run against the mutant and must fail. Nothing here touches a GPU.
"""
import numpy as np
import pytest

import test_oracle_pins as pins
from oracle import direct, grammar, reach


def _drop_last_term(row_ptr, col, val, x):
    x = np.asarray(x, dtype=np.float64)
    n = len(row_ptr) - 1
    y = np.zeros((n,) + x.shape[1:])
    b = np.zeros_like(y)
    for i in range(n):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        e2 = max(s, e - 1)
        v = np.asarray(val[s:e2], dtype=np.float64)
        xs = x[np.asarray(col[s:e2], dtype=np.int64)]
        y[i] = v @ xs
        b[i] = np.abs(v) @ np.abs(xs)
    return y, b


def _levels_min(R):
    lvl = np.zeros(len(R), dtype=np.int64)
    for i in range(len(R)):
        a, b = int(R[i][0]), int(R[i][1])
        lvl[i] = 1 + min(lvl[a] if a >= 0 else 0, lvl[b] if b >= 0 else 0)
    return lvl


def _eval_w_drop_right(g, V, x):
    R = g["R"]
    g2 = dict(g, R=np.array([[a, a] if b < 0 else [a, b] for a, b in R], dtype=np.int64).reshape(-1, 2))
    return _orig_eval_w(g2, V, x)


def _complete_per_edge(R, lvl):
    # one chain per (parent, child) edge instead of one per child
    L = int(lvl.max()) if len(lvl) else 0
    layers = [[] for _ in range(L)]
    for i in range(len(R)):
        K = int(lvl[i])
        ch = []
        for c in R[i]:
            c = int(c)
            if c < 0:
                ch.append(('t', -c - 1))
            elif lvl[c] == K - 1:
                ch.append(('n', c))
            else:
                for k in range(int(lvl[c]) + 1, K):
                    below = ('n', c) if k - 1 == lvl[c] else ('p', c, k - 1, i)
                    layers[k - 1].append((('p', c, k, i), (below,)))
                ch.append(('p', c, K - 1, i))
        layers[K - 1].append((('n', i), tuple(ch)))
    return layers


def _csrv_one_based_columns(row_ptr, col, val):
    V, rows = _orig_csrv(row_ptr, col, val)
    return V, [[(l, j + 1) for l, j in r] for r in rows]


def _matvec_or_and(row_ptr, col, x):
    x = np.asarray(x, dtype=np.uint64)
    n = len(row_ptr) - 1
    y = np.zeros(n, dtype=np.uint64)
    for i in range(n):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        if e > s:
            y[i] = np.bitwise_and.reduce(x[np.asarray(col[s:e], dtype=np.int64)])
    return y


def _minplus_with(reduce_op, empty, leaf):
    def f(row_ptr, col, val, x):
        x = np.asarray(x, dtype=np.float32)
        n = len(row_ptr) - 1
        y = np.full((n,) + x.shape[1:], empty, dtype=np.float32)
        for i in range(n):
            s, e = int(row_ptr[i]), int(row_ptr[i + 1])
            if e > s:
                v = np.asarray(val[s:e], dtype=np.float32)
                xs = x[np.asarray(col[s:e], dtype=np.int64)]
                y[i] = reduce_op(leaf(v if x.ndim == 1 else v[:, None], xs), axis=0)
        return y
    return f


def _sssp_without_keeping_x(row_ptr, col, val, x0, max_iter=1000):
    # x <- M (x) x, forgetting min(x, .): the sources lose their own distance
    x = np.asarray(x0, dtype=np.float32).copy()
    for it in range(1, max_iter + 1):
        nxt = direct.matvec_minplus(row_ptr, col, val, x)
        if np.array_equal(nxt, x):
            return x, it
        x = nxt
    return x, max_iter


def _left_untransposed(row_ptr, col, val, y, m):
    # x[i] += M[i][j] * y[j]: the right product's indexing, read as the left
    y = np.asarray(y, dtype=np.float64)
    x = np.zeros(m)
    b = np.zeros(m)
    for i in range(len(row_ptr) - 1):
        for e in range(int(row_ptr[i]), int(row_ptr[i + 1])):
            j = int(col[e])
            if i < m and j < len(y):
                x[i] += float(val[e]) * y[j]
                b[i] += abs(float(val[e]) * y[j])
    return x, b


def _eval_left_forward_order(g, V, y, m):
    # rules visited in creation order: children before parents, so a parent's
    # weight has not arrived when it is passed on
    g2 = dict(g, R=g["R"][::-1].copy())
    n_r = len(g["R"])
    remap = lambda s: n_r - 1 - s if s >= 0 else s
    g2["R"] = np.array([[remap(int(a)), remap(int(b))] for a, b in g["R"][::-1]], dtype=np.int64).reshape(-1, 2)
    g2["C"] = [[remap(int(s)) for s in row] for row in g["C"]]
    return _orig_eval_left(g2, V, y, m)


def _left_or_and(row_ptr, col, y, m):
    y = np.asarray(y, dtype=np.uint64)
    x = np.full(m, np.uint64(2**64 - 1), dtype=np.uint64)
    seen = np.zeros(m, bool)
    for i in range(len(row_ptr) - 1):
        for e in range(int(row_ptr[i]), int(row_ptr[i + 1])):
            x[col[e]] &= y[i]
            seen[col[e]] = True
    x[~seen] = 0
    return x


def _left_minplus_max(row_ptr, col, val, y, m):
    y = np.asarray(y, dtype=np.float32)
    x = np.full(m, np.inf, dtype=np.float32)
    seen = np.zeros(m, bool)
    for i in range(len(row_ptr) - 1):
        for e in range(int(row_ptr[i]), int(row_ptr[i + 1])):
            t = np.float32(val[e]) + y[i]
            x[col[e]] = t if not seen[col[e]] else max(x[col[e]], t)
            seen[col[e]] = True
    return x


def _forward_uses_right_products(row_ptr, col, x0, max_iter=1000):
    # the reverse direction: x <- x | (M (x) x)
    return _orig_fixpoint(row_ptr, col, x0, max_iter)


_orig_fixpoint = reach.fixpoint
_orig_eval_w = grammar.eval_w
_orig_eval_left = grammar.eval_left
_orig_csrv = grammar.csrv

MUTANTS = [
    ("direct.matvec_f64 drops a term", direct, "matvec_f64", _drop_last_term,
     ["test_worked_product_matches_fig_4_2", "test_direct_matches_dense_matmul"]),
    ("levels uses min", grammar, "levels", _levels_min,
     ["test_worked_levels_match_eq_3_1", "test_grammar_pipeline_on_random_matrices"]),
    ("eval_w drops the right child", grammar, "eval_w", _eval_w_drop_right,
     ["test_worked_grammar_eval_matches_fig_4_2", "test_grammar_pipeline_on_random_matrices"]),
    ("completion per edge", grammar, "complete", _complete_per_edge,
     ["test_grammar_pipeline_on_random_matrices"]),
    ("csrv columns off by one", grammar, "csrv", _csrv_one_based_columns,
     ["test_worked_csrv_matches_eq_2_2"]),
    ("boolean product uses AND", direct, "matvec_or", _matvec_or_and,
     ["test_direct_or_matches_dense_boolean"]),
    ("min-plus product uses max", direct, "matvec_minplus",
     _minplus_with(np.max, np.inf, lambda v, x: v + x),
     ["test_minplus_matches_fp64_rounded_once", "test_minplus_closed_forms_on_worked_example"]),
    ("min-plus empty row gives 0", direct, "matvec_minplus",
     _minplus_with(np.min, 0.0, lambda v, x: v + x),
     ["test_minplus_matches_fp64_rounded_once"]),
    ("min-plus leaf multiplies", direct, "matvec_minplus",
     _minplus_with(np.min, np.inf, lambda v, x: v * x),
     ["test_minplus_matches_fp64_rounded_once", "test_minplus_closed_forms_on_worked_example"]),
    ("left product not transposed", direct, "left_matvec_f64", _left_untransposed,
     ["test_left_matches_dense_transposed_matmul", "test_left_closed_forms_on_worked_example"]),
    ("left grammar sweep children first", grammar, "eval_left", _eval_left_forward_order,
     ["test_left_grammar_sweep_matches_dense"]),
    ("Boolean left product uses AND", direct, "left_matvec_or", _left_or_and,
     ["test_left_products_equal_right_products_of_the_transpose", "test_left_boolean_and_minplus_brute_force"]),
    ("tropical left product uses max", direct, "left_matvec_minplus", _left_minplus_max,
     ["test_left_products_equal_right_products_of_the_transpose", "test_left_boolean_and_minplus_brute_force"]),
    ("forward fixpoint runs towards the sources", reach, "forward_fixpoint", _forward_uses_right_products,
     ["test_forward_fixpoints_match_scipy"]),
    ("shortest-path fixpoint drops min(x, .)", reach, "sssp_fixpoint", _sssp_without_keeping_x,
     ["test_sssp_matches_scipy_dijkstra", "test_sssp_iterations_on_a_path"]),
]


@pytest.mark.parametrize("name,mod,attr,fn,tests", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, mod, attr, fn, tests, monkeypatch, worked):
    monkeypatch.setattr(mod, attr, fn)
    if mod is direct and attr == "matvec_or":
        monkeypatch.setattr(reach, "matvec_or", fn)
    if mod is direct and attr == "matvec_minplus":
        monkeypatch.setattr(reach, "matvec_minplus", fn)
    for t in tests:
        f = getattr(pins, t)
        with pytest.raises(AssertionError):
            if "worked" in f.__code__.co_varnames[:f.__code__.co_argcount]:
                f(worked)
            elif f.__code__.co_argcount == 1:
                f(1)
            else:
                f()
