"""GPU parity for the left product x = M^T y (gc_left_* through the C ABI),
under every policy.

The pages name left multiplication by pull-based reduction as future work
(Sec. 8). Tolerance as for the right product: |x_j - x_ref_j| <= 1e-4 *
(|M|^T |y|)_j with x_j exactly 0 where that bound is 0, x_ref in float64
(oracle.direct.left_matvec_f64). The exact, Boolean and tropical left
products match the oracle bit for bit. Determinism: the same y gives the
same x bit for bit.
"""
import numpy as np
import pytest

import gcsynth
from conftest import dense_to_csr
from oracle import direct

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def left_parity(gcs, torch, n, m, rp, c, v, seed=0, y=None):
    G = gcs.Grammar(n, m, rp, c, v)
    eng = gcs.LeftEngine(G)
    if y is None:
        y = np.random.default_rng(seed).standard_normal(n).astype(np.float32)
    yd = torch.from_numpy(y).cuda()
    x = eng.matvec(yd).cpu().numpy()
    x_ref, b = direct.left_matvec_f64(rp, c, v, y, m)
    ok, worst = direct.within_tolerance(x, x_ref, b, TOL)
    assert ok, f"max scaled error {worst:.3e}"
    np.testing.assert_array_equal(eng.matvec(yd).cpu().numpy(), x)       # deterministic
    # seed, one step per level, terminals, columns; steps with nothing to sum are skipped
    assert 1 <= eng.launch_count() <= G.stats()["depth"] + 3
    return x, eng


def test_worked_example_left(gcs, torch, worked):
    rp, c, v = dense_to_csr(worked["M"], np.float32)
    for r in range(8):                   # y = e_r picks row r
        y = np.zeros(8, np.float32)
        y[r] = 1.0
        x, _ = left_parity(gcs, torch, 8, 7, rp, c, v, y=y)
        np.testing.assert_array_equal(x, worked["M"][r].astype(np.float32))
    left_parity(gcs, torch, 8, 7, rp, c, v, seed=1)


def test_small_and_genotype_left(gcs, torch):
    for seed in range(3):
        rp, c, v, _ = gcsynth.random_sparse(5 + 9 * seed, 7 + 11 * seed, 0.5, [1.0, 2.0, -0.5, 3.25], seed)
        left_parity(gcs, torch, len(rp) - 1, 7 + 11 * seed, rp, c, v, seed=seed)
    cfg = gcsynth.GENO_SMALL
    left_parity(gcs, torch, cfg["n"], cfg["m"], *gcsynth.genotype_csr(**cfg), seed=3)
    cfg = dict(gcsynth.GENO_MEDIUM, n=600)
    left_parity(gcs, torch, 600, cfg["m"], *gcsynth.genotype_csr(**cfg), seed=4)
    rp, c, v, _ = gcsynth.random_sparse(40, 3000, 0.4, [1.0, -1.0, 0.5], 8)   # bare terminals in C
    left_parity(gcs, torch, 40, 3000, rp, c, v, seed=5)


def test_graph_left(gcs, torch):
    N = 3000
    rp, col = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=1)
    left_parity(gcs, torch, N, N, rp, col, gcsynth.target_lengths(col, N, seed=2), seed=6)


def test_long_parent_lists_left(gcs, torch):
    # one column in every row and rows of two kinds: warp-wide (HEAVY) sums
    d = np.zeros((3000, 64), np.float32)
    d[:, 7] = 1.0
    d[::2, 11] = 2.0
    d[1::3, 40] = -0.5
    left_parity(gcs, torch, 3000, 64, *dense_to_csr(d, np.float32), seed=7)


def test_edge_cases_left(gcs, torch):
    cases = [
        (4, 6, np.zeros(5, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32)),      # all rows empty
        (3, 3, np.array([0, 0, 1, 1], np.int64), np.array([2], np.int32), np.array([5.0], np.float32)),
        (2, 4, np.array([0, 2, 4], np.int64), np.array([0, 1, 2, 3], np.int32),
         np.array([1, 2, 3, 4], np.float32)),                                             # no rules (L = 0)
        (1, 1, np.array([0, 1], np.int64), np.array([0], np.int32), np.array([-2.5], np.float32)),
    ]
    for i, (n, m, rp, c, v) in enumerate(cases):
        x, _ = left_parity(gcs, torch, n, m, rp, c, v, seed=10 + i)
    x, eng = left_parity(gcs, torch, 4, 6, *cases[0][2:], seed=1)
    assert np.all(x == 0)
    assert eng.launch_count() == 1          # only the columns step has segments


def test_left_argument_errors(gcs, torch):
    rp, c, v, _ = gcsynth.random_sparse(20, 30, 0.5, [1.0, 2.0], 0)
    G = gcs.Grammar(20, 30, rp, c, v)
    lay = gcs.capi.gc_left_layout(G._p, "f32")
    arena = torch.empty(lay["arena_bytes"] + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_left_upload(G._p, "f32", arena.data_ptr() + 16, arena.numel() - 16)    # misaligned
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_left_upload(G._p, "f32", arena, 256)                                   # too small
    eng = gcs.LeftEngine(G)
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_left_matvec(eng._h, None, torch.zeros(30, device="cuda"))
    with pytest.raises(gcs.GcError, match="GC_ERR_UNSUPPORTED"):
        gcs.LeftEngine(G, "or")                        # OR needs every stored entry to be 1


def test_left_graph_follows_new_pointers(gcs, torch):
    # the steps run as one graph built on the first call; later calls with
    # other y / x buffers must read and write those, in any order
    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(300, cfg["m"], rp, c, v)
    eng = gcs.LeftEngine(G)
    ys = [gcsynth.beta(300, seed=s) for s in (1, 2)]
    yd = [torch.from_numpy(y).cuda() for y in ys]
    xd = [torch.full((cfg["m"],), float("nan"), device="cuda") for _ in range(2)]
    want = []
    for y in ys:
        x_ref, b = direct.left_matvec_f64(rp, c, v, y, cfg["m"])
        want.append((x_ref, b))
    for i, j in [(0, 0), (1, 1), (0, 1), (1, 0), (1, 0)]:
        xd[j].fill_(float("nan"))
        eng.matvec(yd[i], xd[j])
        x = xd[j].cpu().numpy()
        assert direct.within_tolerance(x, *want[i], TOL)[0], (i, j)


def _policy_cases():
    rp, c, v, _ = gcsynth.random_sparse(30, 41, 0.4, [1.0, 2.0, -3.0], 3)
    yield "rand30x41", 30, 41, rp, c, v
    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    yield "geno300", 300, cfg["m"], *gcsynth.genotype_csr(**cfg)
    N = 3000
    grp, gcol = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=1)
    yield "graph3000", N, N, grp, gcol, gcsynth.target_lengths(gcol, N, seed=2)
    d = np.zeros((3000, 64), np.float32)
    d[:, 7] = 1.0
    d[::2, 11] = 2.0
    yield "longlists", 3000, 64, *dense_to_csr(d, np.float32)


POLICY_CASES = list(_policy_cases())


@pytest.mark.parametrize("name,n,m,rp,c,v", POLICY_CASES, ids=[s[0] for s in POLICY_CASES])
def test_left_policies_bit_exact(gcs, torch, name, n, m, rp, c, v):
    G = gcs.Grammar(n, m, rp, c, v)
    g = np.random.default_rng(8)
    # tropical: float32 min-plus, +inf for unused columns
    yf = g.standard_normal(n).astype(np.float32)
    yf[g.random(n) < 0.2] = np.inf
    xf = gcs.LeftEngine(G, "minplus").matvec(torch.from_numpy(yf).cuda()).cpu().numpy()
    assert np.array_equal(xf.view(np.uint32), direct.left_matvec_minplus(rp, c, v, yf, m).view(np.uint32))
    # exact integer sums (integer-valued matrices)
    if np.all(np.floor(v) == v):
        yi = g.integers(-10**6, 10**6, n)
        xi = gcs.LeftEngine(G, "i64").matvec(torch.from_numpy(yi).cuda()).cpu().numpy()
        assert np.array_equal(xi, direct.left_matvec_i64(rp, c, v, yi, m))
    # Boolean OR on the 0/1 pattern: one forward step of 64 source sets
    Gb = gcs.Grammar(n, m, rp, c, None)
    yb = g.integers(0, 2**63, n, dtype=np.uint64)
    eng = gcs.LeftEngine(Gb, "or")
    xb = eng.matvec(torch.from_numpy(yb.view(np.int64)).cuda()).cpu().numpy().view(np.uint64)
    assert np.array_equal(xb, direct.left_matvec_or(rp, c, yb, m))
    assert np.array_equal(eng.matvec(torch.from_numpy(yb.view(np.int64)).cuda()).cpu().numpy().view(np.uint64), xb)


def test_forward_fixpoints(gcs, torch):
    # reachability from the sources and distances from them, by left
    # products, against the oracle and scipy's BFS / Dijkstra on the graph
    scipy_sparse = pytest.importorskip("scipy.sparse")
    from scipy.sparse.csgraph import breadth_first_order, dijkstra
    from oracle import reach
    N = 3000
    rp, col = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=1)
    w = gcsynth.target_lengths(col, N, seed=2)
    srcs = gcsynth.sources(N, 64, seed=0)
    A = scipy_sparse.csr_matrix((w.astype(np.float64), col, rp), shape=(N, N))
    # Boolean: 64 source sets at once
    eng = gcs.LeftEngine(gcs.Grammar(N, N, rp, col, None), "or")
    x0 = gcsynth.frontier(N, srcs)
    xs, iters, rc = eng.reach(torch.from_numpy(x0.view(np.int64)).cuda())
    assert rc == 0
    want, want_iters = reach.forward_fixpoint(rp, col, x0)
    assert iters == want_iters
    got = xs.cpu().numpy().view(np.uint64)
    assert np.array_equal(got, want)
    for b in (0, 17, 63):
        nodes = breadth_first_order(A, int(srcs[b]), directed=True, return_predecessors=False)
        assert np.array_equal(np.nonzero((got >> np.uint64(b)) & np.uint64(1))[0], np.sort(nodes))
    _, it1, rc1 = eng.reach(torch.from_numpy(x0.view(np.int64)).cuda(), max_iter=1)
    assert rc1 == gcs.capi.GC_ERR_NOT_CONVERGED and it1 == -1
    # tropical: distances from the nearest of 8 sources
    engm = gcs.LeftEngine(gcs.Grammar(N, N, rp, col, w), "minplus")
    d0 = gcsynth.frontier_distances(N, srcs[:8])
    ds, diters, drc = engm.sssp(torch.from_numpy(d0).cuda())
    assert drc == 0
    dwant, dwant_iters = reach.forward_sssp_fixpoint(rp, col, w, d0)
    assert diters == dwant_iters
    dgot = ds.cpu().numpy()
    assert np.array_equal(dgot.view(np.uint32), dwant.view(np.uint32))
    np.testing.assert_array_equal(dgot.astype(np.float64), dijkstra(A, directed=True, indices=srcs[:8], min_only=True))
    # in place, and the wrong policy refused
    xin = torch.from_numpy(d0).cuda()
    it = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert gcs.capi.gc_left_sssp(engm._h, xin, xin, 1000, it) == 0
    assert np.array_equal(xin.cpu().numpy().view(np.uint32), dwant.view(np.uint32))
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_left_reach(engm._h, xin, xin, 10, it)
