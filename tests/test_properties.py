"""Property tests (Hypothesis) over tiny matrices, n, m <= 12, with values
from a small set so that pairs repeat and RePair builds rules: the host
builder's packed, layered grammar, evaluated by the CPU emulator of the
packed layout, against brute-force dense products for every policy --
float sums, exact integer sums, Boolean OR and tropical min-plus -- and the
grammar oracle's left product against the dense transpose. No GPU.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from conftest import dense_to_csr, export_all  # noqa: E402
from oracle import grammar  # noqa: E402
from packed_emulator import emulate  # noqa: E402

VALUES = [1.0, 2.0, -1.0, 0.5]


@st.composite
def tiny_matrix(draw):
    n = draw(st.integers(1, 12))
    m = draw(st.integers(1, 12))
    cells = draw(st.lists(st.sampled_from([0.0, 0.0] + VALUES), min_size=n * m, max_size=n * m))
    d = np.array(cells, dtype=np.float64).reshape(n, m)
    if draw(st.booleans()):            # repeated rows: sharing across rows
        d[n // 2:] = d[: n - n // 2]
    return d


@settings(max_examples=150, deadline=None)
@given(d=tiny_matrix(), seed=st.integers(0, 2**31 - 1))
def test_packed_grammar_matches_dense_for_every_policy(gcs, d, seed):
    n, m = d.shape
    rp, c, v = dense_to_csr(d, np.float32)
    G = gcs.Grammar(n, m, rp, c, v)
    ex = export_all(G)
    g = np.random.default_rng(seed)
    nz = d != 0
    # float sum (float64 emulation: exact on these values)
    x = g.standard_normal(m)
    np.testing.assert_allclose(emulate(ex, x), d @ x, rtol=1e-12, atol=1e-12)
    X = g.standard_normal((m, 3))
    np.testing.assert_allclose(emulate(ex, X), d @ X, rtol=1e-12, atol=1e-12)
    # exact integer sum (integer-valued matrices only)
    if np.all(np.floor(d) == d):
        xi = g.integers(-1000, 1000, m)
        assert np.array_equal(emulate(ex, xi, "i64"), d.astype(np.int64) @ xi)
    # Boolean OR over 64-bit sets (stored entries are edges)
    xb = g.integers(0, 2**63, m, dtype=np.uint64)
    want = np.zeros(n, np.uint64)
    for i in range(n):
        for j in np.nonzero(nz[i])[0]:
            want[i] |= xb[j]
    assert np.array_equal(emulate(ex, xb, "or"), want)
    # tropical min-plus, float32 leaves, +inf for an empty row
    xf = g.standard_normal(m).astype(np.float32)
    wantf = np.full(n, np.inf, np.float32)
    for i in range(n):
        for j in np.nonzero(nz[i])[0]:
            wantf[i] = min(wantf[i], np.float32(d[i, j]) + xf[j])
    assert np.array_equal(emulate(ex, xf, "minplus"), wantf)


@settings(max_examples=150, deadline=None)
@given(d=tiny_matrix(), seed=st.integers(0, 2**31 - 1))
def test_oracle_left_product_matches_dense_transpose(d, seed):
    n, m = d.shape
    rp, c, v = dense_to_csr(d, np.float64)
    V, rows = grammar.csrv(rp, c, v)
    y = np.random.default_rng(seed).standard_normal(n)
    want = d.T @ y
    if not len(V):
        assert np.all(want == 0)
        return
    g = grammar.repair(rows)
    np.testing.assert_allclose(grammar.eval_left(g, V, y, m), want, rtol=1e-12, atol=1e-12)
