"""GPU parity for the tropical (min, +) policy through the C ABI.

The pages name the tropical semiring (Sec. 5: min as the combine, + as the
leaf map, +inf as the identity; one product is one Bellman-Ford relaxation)
and verify it bit for bit (Sec. 6). min is exact and each leaf sum is rounded
to float32 once, so every comparison here is bit for bit against
oracle.direct.matvec_minplus and oracle.reach.sssp_fixpoint, in every emit
mode (row, slice, level), at k = 1 and k = 16, on both schedules.
"""
import numpy as np
import pytest

import gcsynth
from oracle import direct, reach

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_same_bits(got, want):
    assert got.shape == want.shape
    bad = np.nonzero(_bits(got).ravel() != _bits(want).ravel())[0]
    assert bad.size == 0, f"{bad.size} elements differ, first at {bad[0]}: {got.ravel()[bad[0]]} vs {want.ravel()[bad[0]]}"


def _cases():
    for seed in range(3):
        rp, c, v, _ = gcsynth.random_sparse(5 + 9 * seed, 7 + 11 * seed, 0.5, [1.0, 2.0, -0.5, 3.25], seed)
        yield f"rand{seed}", len(rp) - 1, 7 + 11 * seed, rp, c, v
    d = gcsynth.genotype_dense(n=300, m=900, founders=6, switch=0.01, mutation=0.005, seed=4)
    rp, c, v = gcsynth.dense_to_csr(d)
    yield "geno300x900", 300, 900, rp, c, v
    # long rows of bare terminals: the level emit with few levels
    rp, c, v, _ = gcsynth.random_sparse(40, 3000, 0.4, [1.0, -1.0, 0.5], 8)
    yield "cheavy40x3000", 40, 3000, rp, c, v


CASES = list(_cases())


@pytest.mark.parametrize("name,n,m,rp,c,v", CASES, ids=[s[0] for s in CASES])
def test_small_minplus_k1_and_k16(gcs, torch, name, n, m, rp, c, v):
    G = gcs.Grammar(n, m, rp, c, v)
    g = np.random.default_rng(11)
    for k_max in (1, 16):
        eng = gcs.Engine(G, "minplus", k_max)
        x = g.standard_normal(m).astype(np.float32)
        x[g.random(m) < 0.2] = np.inf                 # unreached columns
        y = eng.matvec(_dev(torch, x)).cpu().numpy()
        assert eng.check() == 0
        assert_same_bits(y, direct.matvec_minplus(rp, c, v, x))
        if k_max == 16:
            X = (g.standard_normal((m, 16)) * 10.0 ** g.uniform(-3, 3, (m, 16))).astype(np.float32)
            Y = eng.matvec(_dev(torch, X)).cpu().numpy()
            assert_same_bits(Y, direct.matvec_minplus(rp, c, v, X))


def test_genotype_small_minplus(gcs, torch):
    cfg = gcsynth.GENO_SMALL
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(cfg["n"], cfg["m"], rp, c, v)
    eng = gcs.Engine(G, "minplus", 16)
    x = gcsynth.beta(cfg["m"], seed=0)
    y = eng.matvec(_dev(torch, x)).cpu().numpy()
    assert_same_bits(y, direct.matvec_minplus(rp, c, v, x))
    np.testing.assert_array_equal(eng.matvec_host(x), y)
    X = gcsynth.beta(cfg["m"], seed=1, k=16)
    Y = eng.matvec(_dev(torch, X)).cpu().numpy()
    assert_same_bits(Y, direct.matvec_minplus(rp, c, v, X))
    # the per-level schedule and the allocation-free entry point agree bit for bit
    eng.schedule = "per_level"
    assert_same_bits(eng.matvec(_dev(torch, x)).cpu().numpy(), y)
    eng.schedule = "persistent"
    ys = torch.empty(cfg["n"], dtype=torch.float32, device="cuda")
    gcs.capi.gc_matvec_static(eng._h, _dev(torch, x), ys, 1)
    assert_same_bits(ys.cpu().numpy(), y)


@pytest.mark.parametrize("rows,k_max", [(600, 1), (300, 16)])
def test_genotype_wide_slice_minplus(gcs, torch, rows, k_max):
    # slice emit (k_max 1) and level emit with carry slots (k_max 16), both
    # schedules, on a slice of the 50,000-variant generator
    cfg = dict(gcsynth.GENO_MEDIUM, n=rows)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(rows, cfg["m"], rp, c, v)
    eng = gcs.Engine(G, "minplus", k_max)
    x = gcsynth.beta(cfg["m"], seed=7)
    want = direct.matvec_minplus(rp, c, v, x)
    y = eng.matvec(_dev(torch, x)).cpu().numpy()
    assert eng.check() == 0
    assert_same_bits(y, want)
    eng.schedule = "per_level"
    assert_same_bits(eng.matvec(_dev(torch, x)).cpu().numpy(), want)
    if k_max == 16:
        eng.schedule = "persistent"
        X = gcsynth.beta(cfg["m"], seed=8, k=16)
        assert_same_bits(eng.matvec(_dev(torch, X)).cpu().numpy(), direct.matvec_minplus(rp, c, v, X))


def test_edge_cases_minplus(gcs, torch):
    cases = [
        (4, 6, np.zeros(5, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32)),      # all rows empty
        (3, 3, np.array([0, 0, 1, 1], np.int64), np.array([2], np.int32), np.array([5.0], np.float32)),
        (2, 4, np.array([0, 2, 4], np.int64), np.array([0, 1, 2, 3], np.int32),
         np.array([1, 2, 3, 4], np.float32)),                                             # no rules (L = 0)
        (1, 1, np.array([0, 1], np.int64), np.array([0], np.int32), np.array([-2.5], np.float32)),
    ]
    for n, m, rp, c, v in cases:
        G = gcs.Grammar(n, m, rp, c, v)
        eng = gcs.Engine(G, "minplus", 1)
        x = np.arange(1, m + 1, dtype=np.float32)
        y = eng.matvec(_dev(torch, x)).cpu().numpy()
        assert_same_bits(y, direct.matvec_minplus(rp, c, v, x))
    G = gcs.Grammar(4, 6, np.zeros(5, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32))
    y = gcs.Engine(G, "minplus", 1).matvec(_dev(torch, np.zeros(6, np.float32))).cpu().numpy()
    assert np.all(y == np.inf)      # empty rows get the min-identity


def test_shortest_paths_fixpoint(gcs, torch):
    scipy_sparse = pytest.importorskip("scipy.sparse")
    from scipy.sparse.csgraph import dijkstra
    N = 3000
    rp, col = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=1)
    w = gcsynth.target_lengths(col, N, seed=2)
    G = gcs.Grammar(N, N, rp, col, w)
    eng = gcs.Engine(G, "minplus", 1)
    x = np.random.default_rng(2).standard_normal(N).astype(np.float32)
    assert_same_bits(eng.matvec(_dev(torch, x)).cpu().numpy(), direct.matvec_minplus(rp, col, w, x))
    srcs = gcsynth.sources(N, 8, seed=0)
    x0 = gcsynth.frontier_distances(N, srcs)
    xs, iters, rc = eng.sssp(_dev(torch, x0))
    assert rc == 0
    want, want_iters = reach.sssp_fixpoint(rp, col, w, x0)
    assert iters == want_iters
    got = xs.cpu().numpy()
    assert_same_bits(got, want)
    A = scipy_sparse.csr_matrix((w.astype(np.float64), col, rp), shape=(N, N))
    np.testing.assert_array_equal(got.astype(np.float64),
                                  dijkstra(A.T.tocsr(), directed=True, indices=srcs, min_only=True))
    # not converged within one product: status and count say so, once
    _, iters1, rc1 = eng.sssp(_dev(torch, x0), max_iter=1)
    assert rc1 == gcs.capi.GC_ERR_NOT_CONVERGED and iters1 == -1
    assert eng.check() == gcs.capi.GC_ERR_NOT_CONVERGED
    assert eng.check() == 0
    # in place (x == x0)
    xin = _dev(torch, x0)
    it = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert gcs.capi.gc_sssp(eng._h, xin, xin, 1000, it) == 0
    assert_same_bits(xin.cpu().numpy(), want)


def test_minplus_argument_errors(gcs, torch):
    rp, c, v, _ = gcsynth.random_sparse(20, 20, 0.5, [1.0, 2.0], 0)
    G = gcs.Grammar(20, 20, rp, c, v)
    f32 = gcs.Engine(G, "f32", 1)
    mp = gcs.Engine(G, "minplus", 1)
    x = torch.zeros(20, device="cuda")
    it = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_sssp(f32._h, x, x, 5, it)        # needs the min-plus policy
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_reach(mp._h, x, x, 5, it)        # reach needs the OR policy
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        mp.matvec(torch.zeros((20, 16), device="cuda"))   # k = 16 on a k_max = 1 handle
    rect = gcs.Grammar(20, 30, *gcsynth.random_sparse(20, 30, 0.5, [1.0], 1)[:3])
    rect_eng = gcs.Engine(rect, "minplus", 1)
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_sssp(rect_eng._h, x, x, 5, it)   # n != m
