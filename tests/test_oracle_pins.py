"""Pins for the CPU oracle, against things other than the oracle itself:
the pages' worked example (tests/golden/worked_example.json), library
routines (numpy dense matmul, scipy BFS), closed forms and brute force.

Each test is chosen so that a plausible slip in the oracle -- a dropped term,
a wrong index, a transposed operand, min for max -- fails at least one of
them (tests/test_oracle_mutants.py plants such slips and checks that).
"""
import itertools

import numpy as np
import pytest
import scipy.sparse as sp
from scipy.sparse.csgraph import breadth_first_order, dijkstra

import gcsynth
from oracle import direct, grammar, reach
from conftest import dense_to_csr


# ---------------------------------------------------------------- worked example
def test_worked_product_matches_fig_4_2(worked):
    rp, c, v = dense_to_csr(worked["M"], np.float64)
    y, b = direct.matvec_f64(rp, c, v, worked["x"])
    np.testing.assert_allclose(y, worked["y"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(b, np.abs(worked["M"]) @ np.abs(worked["x"]), atol=1e-12)


def test_worked_csrv_matches_eq_2_2(worked):
    rp, c, v = dense_to_csr(worked["M"], np.float64)
    V, rows = grammar.csrv(rp, c, v)
    np.testing.assert_allclose(V, worked["V"], atol=0)
    assert rows == worked["S"]


def test_worked_grammar_decompresses_to_S(worked):
    # Eqs. 2.3 + 2.4 must expand to exactly the string of Eq. 2.2
    assert grammar.decompress(worked["grammar"]) == worked["S"]


def test_worked_grammar_eval_matches_fig_4_2(worked):
    g = worked["grammar"]
    y = grammar.eval_w(g, worked["V"], worked["x"])
    np.testing.assert_allclose(y, worked["y"], atol=1e-12)
    rv = worked["raw"]["product"]["root_values"]
    for name, want in rv.items():
        got = grammar.eval_recursive(int(name[1:]) - 1, g["R"], g["term_l"], g["term_j"],
                                     worked["V"], worked["x"])
        assert abs(got - want) < 1e-12


def test_worked_levels_match_eq_3_1(worked):
    lvl = grammar.levels(worked["grammar"]["R"])
    assert int(lvl.max()) == worked["raw"]["levels"]["L"]
    for k, members in enumerate(worked["level_sets"], start=1):
        assert sorted(np.nonzero(lvl == k)[0].tolist()) == sorted(members)


def test_worked_completion_matches_sec_4_2(worked):
    g = worked["grammar"]
    R = g["R"]
    lvl = grammar.levels(R)
    pt = worked["raw"]["pass_through"]
    u = int(pt["carried"][1:]) - 1
    reader = int(pt["reader"][1:]) - 1
    layers = grammar.complete(R, lvl)
    added = [key for layer in layers for key, _ in layer if key[0] == 'p']
    assert added == [('p', u, pt["level"])]
    assert grammar.pass_through_count(R, lvl) == pt["count"]
    node_children = {key: ch for layer in layers for key, ch in layer}
    assert ('p', u, pt["level"]) in node_children[('n', reader)]
    assert grammar.is_properly_layered(layers)
    # widths = printed strata plus the printed pass-through at its level
    want = [len(s) for s in worked["level_sets"]]
    want[pt["level"] - 1] += 1
    assert [len(layer) for layer in layers] == want
    assert grammar.live_widths(R, lvl) == want
    y = grammar.eval_layered(layers, g, worked["V"], worked["x"])
    np.testing.assert_allclose(y, worked["y"], atol=1e-12)


def test_worked_repair_is_valid(worked):
    g = grammar.repair(worked["S"])
    assert grammar.decompress(g) == worked["S"]
    _assert_repair_final(g)
    y = grammar.eval_w(g, worked["V"], worked["x"])
    np.testing.assert_allclose(y, worked["y"], atol=1e-12)


def test_uncompleted_grammar_is_not_properly_layered(worked):
    # the raw Eq. 2.3 grammar has the skip edge N8 -> N4; a layering that
    # simply drops pass-throughs must be rejected by the checker
    R = worked["grammar"]["R"]
    lvl = grammar.levels(R)
    layers = [[(key, ch) for key, ch in layer if key[0] == 'n'] for layer in grammar.complete(R, lvl)]
    bad = []
    for layer in layers:
        bad.append([(key, tuple(('n', c[1]) if c[0] == 'p' else c for c in ch)) for key, ch in layer])
    assert not grammar.is_properly_layered(bad)


# ---------------------------------------------------------------- helpers
def _assert_repair_final(g):
    # stop rule: no pair of adjacent symbols occurs twice in the final C
    seen = {}
    for row in g["C"]:
        for i in range(len(row) - 1):
            p = (row[i], row[i + 1])
            seen[p] = seen.get(p, 0) + 1
    assert all(v < 2 for v in seen.values())
    # topological numbering and every rule referenced
    R = g["R"]
    used = np.zeros(len(R), dtype=bool)
    for i, (a, b) in enumerate(R):
        for c in (a, b):
            if c >= 0:
                assert c < i
                used[c] = True
    for row in g["C"]:
        for s in row:
            if s >= 0:
                used[s] = True
    assert used.all()


def _random_cases():
    for seed in range(8):
        n = 3 + seed % 5
        m = 4 + (seed * 3) % 7
        rp, c, v, dense = gcsynth.random_sparse(n, m, 0.6, [1.0, 2.0, -0.5], seed)
        yield seed, rp, c, v, dense.astype(np.float64)
    # genotype-shaped rows (few distinct repeated rows) exercise deep grammars
    d = gcsynth.genotype_dense(n=12, m=40, founders=3, switch=0.05, mutation=0.01, seed=3)
    rp, c, v = gcsynth.dense_to_csr(d)
    yield 100, rp, c, v, d.astype(np.float64)


# ---------------------------------------------------------------- library routines
@pytest.mark.parametrize("k", [1, 3])
def test_direct_matches_dense_matmul(k):
    for seed, rp, c, v, dense in _random_cases():
        x = np.random.default_rng(seed).standard_normal((dense.shape[1], k))
        x = x[:, 0] if k == 1 else x
        y, b = direct.matvec_f64(rp, c, v, x)
        np.testing.assert_allclose(y, dense @ x, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(b, np.abs(dense) @ np.abs(x), rtol=1e-12, atol=1e-12)


def test_direct_int_matches_dense_int_matmul():
    for seed, rp, c, v, dense in _random_cases():
        M = np.round(dense * 2).astype(np.int64)       # integer matrix
        rp2, c2, v2 = dense_to_csr(M, np.float64)
        x = np.random.default_rng(seed).integers(-10**6, 10**6, dense.shape[1])
        assert np.array_equal(direct.matvec_i64(rp2, c2, v2, x), M @ x)


def test_direct_or_matches_dense_boolean():
    for seed, rp, c, v, dense in _random_cases():
        x = np.random.default_rng(seed).integers(0, 2**63, dense.shape[1], dtype=np.uint64)
        y = direct.matvec_or(rp, c, x)
        A = dense != 0
        for bit in range(64):
            xb = ((x >> np.uint64(bit)) & np.uint64(1)).astype(np.int64)
            want = (A.astype(np.int64) @ xb) > 0
            got = ((y >> np.uint64(bit)) & np.uint64(1)).astype(bool)
            assert np.array_equal(got, want)


def test_tolerance_rule():
    ok, _ = direct.within_tolerance([1.0, 0.0], np.array([1.0, 0.0]), np.array([1.0, 0.0]), 1e-4)
    assert ok
    ok, _ = direct.within_tolerance([1.0, 1e-30], np.array([1.0, 0.0]), np.array([1.0, 0.0]), 1e-4)
    assert not ok
    ok, _ = direct.within_tolerance([1.001], np.array([1.0]), np.array([1.0]), 1e-4)
    assert not ok


# ---------------------------------------------------------------- brute force
def test_grammar_pipeline_on_random_matrices():
    for seed, rp, c, v, dense in _random_cases():
        V, rows = grammar.csrv(rp, c, v)
        # CSRV decodes back to the matrix
        back = np.zeros_like(dense)
        for i, r in enumerate(rows):
            for l, j in r:
                back[i, j] = V[l]
        np.testing.assert_array_equal(back, dense)
        g = grammar.repair(rows)
        assert grammar.decompress(g) == rows
        _assert_repair_final(g)
        x = np.random.default_rng(seed + 7).standard_normal(dense.shape[1])
        want = dense @ x
        np.testing.assert_allclose(grammar.eval_w(g, V, x), want, atol=1e-12)
        for i, row in enumerate(g["C"]):
            got = sum(grammar.eval_recursive(s, g["R"], g["term_l"], g["term_j"], V, x) for s in row)
            assert abs(got - want[i]) < 1e-12
        lvl = grammar.levels(g["R"])
        # Eq. 3.1 checked edge by edge: a parent is strictly above each child,
        # and exactly one above its highest child
        for i, (a, b) in enumerate(g["R"]):
            ch = [lvl[s] if s >= 0 else 0 for s in (a, b)]
            assert lvl[i] == 1 + max(ch)
        layers = grammar.complete(g["R"], lvl)
        assert grammar.is_properly_layered(layers)
        widths = [len(layer) for layer in layers]
        assert widths == grammar.live_widths(g["R"], lvl)
        assert sum(widths) == len(g["R"]) + grammar.pass_through_count(g["R"], lvl)
        np.testing.assert_allclose(grammar.eval_layered(layers, g, V, x), want, atol=1e-12)


def test_exhaustive_small_binary_matrices():
    # every 0/1 matrix of shape 3x3 through the grammar pipeline
    x = np.array([1.5, -2.0, 0.25])
    for bits in itertools.product([0, 1], repeat=9):
        dense = np.array(bits, dtype=np.float64).reshape(3, 3)
        rp, c, v = dense_to_csr(dense, np.float64)
        V, rows = grammar.csrv(rp, c, v)
        g = grammar.repair(rows)
        np.testing.assert_allclose(grammar.eval_w(g, V, x) if len(V) else np.zeros(3), dense @ x, atol=1e-12)


def test_repeated_rows_compress_to_one_root():
    # n identical rows of length m: RePair must end with one symbol per row
    dense = np.tile(np.arange(1, 9, dtype=np.float64), (5, 1))
    rp, c, v = dense_to_csr(dense, np.float64)
    V, rows = grammar.csrv(rp, c, v)
    g = grammar.repair(rows)
    assert all(len(r) == 1 for r in g["C"]) and len({r[0] for r in g["C"]}) == 1
    assert len(g["R"]) == 7         # a string of 8 symbols needs 7 binary rules


# ---------------------------------------------------------------- reachability
def _random_graph(n, deg, seed):
    g = np.random.default_rng(seed)
    rows = [np.unique(g.integers(0, n, g.integers(0, deg + 1))) for _ in range(n)]
    rp = np.zeros(n + 1, dtype=np.int64)
    np.cumsum([len(r) for r in rows], out=rp[1:])
    col = np.concatenate(rows).astype(np.int32) if rp[-1] else np.zeros(0, np.int32)
    return rp, col


def test_reach_matches_scipy_bfs():
    for seed in range(5):
        n = 60
        rp, col = _random_graph(n, 2, seed)
        srcs = np.random.default_rng(seed).choice(n, 10, replace=False)
        x0 = gcsynth.frontier(n, srcs)
        xs, iters = reach.fixpoint(rp, col, x0)
        A = sp.csr_matrix((np.ones(len(col)), col, rp), shape=(n, n))
        AT = A.T.tocsr()
        want = np.zeros(n, dtype=np.uint64)
        for b, s in enumerate(srcs):
            nodes = breadth_first_order(AT, int(s), directed=True, return_predecessors=False)
            want[nodes] |= np.uint64(1) << np.uint64(b)
        assert np.array_equal(xs, want)
        assert np.array_equal(reach.reach_bfs(rp, col, n, srcs), want)


def test_reach_iterations_on_a_path():
    # 0 -> 1 -> ... -> n-1, source n-1: n-1 products spread the bit to node 0,
    # the n-th changes nothing
    n = 9
    rp = np.concatenate([np.arange(n, dtype=np.int64), [n - 1]])
    col = np.arange(1, n, dtype=np.int32)
    x0 = gcsynth.frontier(n, np.array([n - 1]))
    xs, iters = reach.fixpoint(rp, col, x0)
    assert iters == n
    assert np.all(xs == 1)


# ---------------------------------------------------------------- tropical (min, +)
def _minplus_cases():
    """The random cases, plus one with empty rows and a column no row uses."""
    yield from _random_cases()
    dense = np.zeros((6, 5))
    dense[0, [1, 3]] = [2.0, -1.5]
    dense[2, 0] = 4.0
    dense[3, [0, 1, 3]] = [1.0, 1.0, 7.25]
    dense[5, 3] = -3.0
    rp, c, v = dense_to_csr(dense, np.float64)
    yield 200, rp, c, v, dense


def _minplus_fp64_rounded_once(dense, x):
    # every sum in float64, one rounding to float32 at the end, dense loops:
    # rounding is monotone, so min commutes with it, and a float64 sum of two
    # float32 numbers rounded to float32 is the correctly rounded float32 sum
    # (double rounding is harmless for + when 53 >= 2 * 24 + 2)
    n, m = dense.shape
    k = 1 if x.ndim == 1 else x.shape[1]
    xx = x.reshape(m, k)
    out = np.empty((n, k), dtype=np.float32)
    for i in range(n):
        for c in range(k):
            best = float("inf")
            for j in range(m):
                if dense[i, j] != 0:
                    best = min(best, float(np.float32(dense[i, j])) + float(xx[j, c]))
            out[i, c] = np.float32(best)
    return out.reshape(n) if x.ndim == 1 else out


@pytest.mark.parametrize("k", [1, 3])
def test_minplus_matches_fp64_rounded_once(k):
    for seed, rp, c, v, dense in _minplus_cases():
        g = np.random.default_rng(seed + 11)
        # wide dynamic range, so that a float32 sum often rounds
        x = (g.standard_normal((dense.shape[1], k)) * 10.0 ** g.uniform(-6, 6, (dense.shape[1], k)))
        x = x.astype(np.float32)
        x = x[:, 0] if k == 1 else x
        got = direct.matvec_minplus(rp, c, v, x)
        want = _minplus_fp64_rounded_once(dense, x)
        assert got.dtype == np.float32
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_minplus_closed_forms_on_worked_example(worked):
    M = worked["M"]
    rp, c, v = dense_to_csr(M, np.float64)
    nz = M != 0
    rowmin = np.array([M[i, nz[i]].min() for i in range(M.shape[0])], dtype=np.float32)
    m = M.shape[1]
    # x = 0: each row's smallest stored value
    assert np.array_equal(direct.matvec_minplus(rp, c, v, np.zeros(m, np.float32)), rowmin)
    # x = 2.5 everywhere: shifted by 2.5 (exact: the values are small dyadics)
    assert np.array_equal(direct.matvec_minplus(rp, c, v, np.full(m, 2.5, np.float32)), rowmin + np.float32(2.5))
    # x = +inf everywhere: nothing reachable
    assert np.all(np.isinf(direct.matvec_minplus(rp, c, v, np.full(m, np.inf, np.float32))))
    # one finite column j0 (the rest +inf): exactly the rows that store j0
    for j0 in range(m):
        x = np.full(m, np.inf, np.float32)
        x[j0] = -100.0
        y = direct.matvec_minplus(rp, c, v, x)
        want = np.where(nz[:, j0], M[:, j0].astype(np.float32) - np.float32(100.0), np.float32(np.inf))
        assert np.array_equal(y, want)


def test_minplus_grammar_sweep_matches_direct(worked):
    rp, c, v = dense_to_csr(worked["M"], np.float64)
    x = np.random.default_rng(5).standard_normal(worked["M"].shape[1]).astype(np.float32)
    assert np.array_equal(grammar.eval_w_minplus(worked["grammar"], worked["V"], x),
                          direct.matvec_minplus(rp, c, v, x))
    for seed, rp, c, v, dense in _minplus_cases():
        V, rows = grammar.csrv(rp, c, v)
        g = grammar.repair(rows)
        x = np.random.default_rng(seed + 3).standard_normal((dense.shape[1], 2)).astype(np.float32)
        want = _minplus_fp64_rounded_once(dense, x)
        got = grammar.eval_w_minplus(g, V, x) if len(V) else np.full((dense.shape[0], 2), np.inf, np.float32)
        assert np.array_equal(got, want)


def _weighted_graph(n, deg, seed):
    rp, col = _random_graph(n, deg, seed)
    w = np.random.default_rng(seed + 1).integers(1, 10, len(col)).astype(np.float32)
    return rp, col, w


def test_sssp_matches_scipy_dijkstra():
    # integer edge lengths: every path length is exact in float32
    for seed in range(5):
        n = 80
        rp, col, w = _weighted_graph(n, 3, seed)
        srcs = np.random.default_rng(seed).choice(n, 4, replace=False)
        x0 = np.full(n, np.inf, np.float32)
        x0[srcs] = 0.0
        xs, iters = reach.sssp_fixpoint(rp, col, w, x0)
        A = sp.csr_matrix((w.astype(np.float64), col, rp), shape=(n, n))
        # distance i -> s along out-edges = distance s -> i in the transpose
        want = dijkstra(A.T.tocsr(), directed=True, indices=srcs, min_only=True)
        assert np.array_equal(xs.astype(np.float64), want)


def test_sssp_iterations_on_a_path():
    # 0 -> 1 -> ... -> n-1 with lengths 1..n-1, source n-1 at distance 0:
    # x*[i] = sum of the lengths from i on; n-1 products, then one unchanged
    n = 9
    rp = np.concatenate([np.arange(n, dtype=np.int64), [n - 1]])
    col = np.arange(1, n, dtype=np.int32)
    w = np.arange(1, n, dtype=np.float32)
    x0 = np.full(n, np.inf, np.float32)
    x0[n - 1] = 0.0
    xs, iters = reach.sssp_fixpoint(rp, col, w, x0)
    assert iters == n
    assert np.array_equal(xs, np.array([w[i:].sum() for i in range(n)], dtype=np.float32))


# ---------------------------------------------------------------- left product x = M^T y
def test_left_matches_dense_transposed_matmul():
    for seed, rp, c, v, dense in _random_cases():
        y = np.random.default_rng(seed + 21).standard_normal(dense.shape[0])
        x, b = direct.left_matvec_f64(rp, c, v, y, dense.shape[1])
        np.testing.assert_allclose(x, dense.T @ y, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(b, np.abs(dense).T @ np.abs(y), rtol=1e-12, atol=1e-12)


def test_left_closed_forms_on_worked_example(worked):
    M = worked["M"]
    rp, c, v = dense_to_csr(M, np.float64)
    n, m = M.shape
    # y = e_r picks row r of M; y = 1 gives the column sums
    for r in range(n):
        y = np.zeros(n)
        y[r] = 1.0
        x, _ = direct.left_matvec_f64(rp, c, v, y, m)
        assert np.array_equal(x, M[r])
    x, _ = direct.left_matvec_f64(rp, c, v, np.ones(n), m)
    assert np.array_equal(x, M.sum(axis=0))
    # duality: y . (M x) == (M^T y) . x
    g = np.random.default_rng(3)
    xv, yv = g.standard_normal(m), g.standard_normal(n)
    lhs = yv @ direct.matvec_f64(rp, c, v, xv)[0]
    rhs = direct.left_matvec_f64(rp, c, v, yv, m)[0] @ xv
    assert abs(lhs - rhs) < 1e-12


def test_left_grammar_sweep_matches_dense(worked):
    M = worked["M"]
    y = np.random.default_rng(4).standard_normal(M.shape[0])
    np.testing.assert_allclose(grammar.eval_left(worked["grammar"], worked["V"], y, M.shape[1]), M.T @ y,
                               rtol=0, atol=1e-12)
    for seed, rp, c, v, dense in _random_cases():
        V, rows = grammar.csrv(rp, c, v)
        g = grammar.repair(rows)
        y = np.random.default_rng(seed + 5).standard_normal(dense.shape[0])
        np.testing.assert_allclose(grammar.eval_left(g, V, y, dense.shape[1]), dense.T @ y, rtol=0, atol=1e-12)


def _transpose_csr(rp, c, v, n, m):
    T = sp.csr_matrix((np.asarray(v, np.float64), np.asarray(c), np.asarray(rp)), shape=(n, m)).T.tocsr()
    T.sort_indices()
    return T.indptr.astype(np.int64), T.indices.astype(np.int32), T.data


def test_left_products_equal_right_products_of_the_transpose():
    # every left product is the right product of M^T, built by scipy; the
    # right products are pinned above
    for seed, rp, c, v, dense in _minplus_cases():
        n, m = dense.shape
        trp, tc, tv = _transpose_csr(rp, c, v, n, m)
        g = np.random.default_rng(seed + 31)
        y = g.standard_normal(n)
        np.testing.assert_allclose(direct.left_matvec_f64(rp, c, v, y, m)[0], direct.matvec_f64(trp, tc, tv, y)[0],
                                   rtol=1e-12, atol=1e-12)
        yi = g.integers(-1000, 1000, n)
        vi = np.round(np.asarray(v) * 2)
        trp2, tc2, tv2 = _transpose_csr(rp, c, vi, n, m)
        assert np.array_equal(direct.left_matvec_i64(rp, c, vi, yi, m), direct.matvec_i64(trp2, tc2, tv2, yi))
        yb = g.integers(0, 2**63, n, dtype=np.uint64)
        assert np.array_equal(direct.left_matvec_or(rp, c, yb, m), direct.matvec_or(trp, tc, yb))
        yf = (g.standard_normal(n) * 10.0 ** g.uniform(-4, 4, n)).astype(np.float32)
        assert np.array_equal(direct.left_matvec_minplus(rp, c, v, yf, m).view(np.uint32),
                              direct.matvec_minplus(trp, tc, tv, yf).view(np.uint32))


def test_left_boolean_and_minplus_brute_force():
    for seed, rp, c, v, dense in _minplus_cases():
        n, m = dense.shape
        nz = dense != 0
        g = np.random.default_rng(seed + 41)
        yb = g.integers(0, 2**63, n, dtype=np.uint64)
        want = np.zeros(m, np.uint64)
        yf = g.standard_normal(n).astype(np.float32)
        wantf = np.full(m, np.inf, np.float32)
        for i in range(n):
            for j in range(m):
                if nz[i, j]:
                    want[j] |= yb[i]
                    wantf[j] = min(wantf[j], np.float32(dense[i, j]) + yf[i])
        assert np.array_equal(direct.left_matvec_or(rp, c, yb, m), want)
        assert np.array_equal(direct.left_matvec_minplus(rp, c, v, yf, m), wantf)


def test_forward_fixpoints_match_scipy():
    # left-product fixpoints run along out-edges from the sources: scipy's
    # BFS and Dijkstra on the graph itself (not its transpose)
    for seed in range(5):
        n = 70
        rp, col, w = _weighted_graph(n, 3, seed)
        srcs = np.random.default_rng(seed + 9).choice(n, 5, replace=False)
        A = sp.csr_matrix((w.astype(np.float64), col, rp), shape=(n, n))
        want = np.zeros(n, dtype=np.uint64)
        for b, s in enumerate(srcs):
            nodes = breadth_first_order(A, int(s), directed=True, return_predecessors=False)
            want[nodes] |= np.uint64(1) << np.uint64(b)
        xs, _ = reach.forward_fixpoint(rp, col, gcsynth.frontier(n, srcs))
        assert np.array_equal(xs, want)
        d0 = np.full(n, np.inf, np.float32)
        d0[srcs] = 0.0
        ds, _ = reach.forward_sssp_fixpoint(rp, col, w, d0)
        assert np.array_equal(ds.astype(np.float64), dijkstra(A, directed=True, indices=srcs, min_only=True))


def test_forward_iterations_on_a_path():
    # 0 -> 1 -> ... -> n-1 from source 0: n-1 products reach n-1, one more changes nothing
    n = 9
    rp = np.concatenate([np.arange(n, dtype=np.int64), [n - 1]])
    col = np.arange(1, n, dtype=np.int32)
    xs, iters = reach.forward_fixpoint(rp, col, gcsynth.frontier(n, np.array([0])))
    assert iters == n and np.all(xs == 1)
    w = np.arange(1, n, dtype=np.float32)
    d0 = np.full(n, np.inf, np.float32)
    d0[0] = 0.0
    ds, iters = reach.forward_sssp_fixpoint(rp, col, w, d0)
    assert iters == n and np.array_equal(ds, np.concatenate([[0], np.cumsum(w)]).astype(np.float32))


def test_cpu_grammar_sweep_matches_dense_and_thread_counts():
    # the C W-array sweep over the oracle's own RePair grammar (same symbol
    # encoding as the library's export): equal to the dense product, and the
    # same bits with any number of threads
    from baselines.wsweep import GrammarSweep
    for seed, rp, c, v, dense in _random_cases():
        V, rows = grammar.csrv(rp, c, v)
        if not len(V):
            continue
        g = grammar.repair(rows)
        R = np.asarray(g["R"], dtype=np.int64).reshape(-1, 2)
        c_off = np.concatenate([[0], np.cumsum([len(r) for r in g["C"]])])
        c_sym = np.array([s for r in g["C"] for s in r], dtype=np.int64)
        sw = GrammarSweep(R, grammar.levels(g["R"]) if len(R) else np.zeros(0, np.int64), c_off, c_sym,
                          g["term_j"], g["term_l"], V)
        x = np.random.default_rng(seed).standard_normal(dense.shape[1])
        y1 = sw(x, 1)
        np.testing.assert_allclose(y1, dense @ x, rtol=1e-12, atol=1e-12)
        assert np.array_equal(sw(x, 3), y1)


def test_cpu_csr_product_matches_dense():
    from baselines.wsweep import CsrProduct
    for seed, rp, c, v, dense in _random_cases():
        x = np.random.default_rng(seed + 2).standard_normal(dense.shape[1])
        p = CsrProduct(rp, c, v)
        y = p(x, 1)
        np.testing.assert_allclose(y, dense @ x, rtol=1e-12, atol=1e-12)
        assert np.array_equal(p(x, 3), y)
