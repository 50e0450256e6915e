"""Full-size parity, in the launch configuration bench.py times.

* 10,000 x 50,000 genotype matrix (2.3e8 non-zeros, one grammar): every row of
  y = G beta against the float64 oracle, persistent schedule; every row of a
  16-wide product.
* 2,000,000-node copy-model graph (about 2e8 edges): the Boolean product and the
  reachability fixpoint from 64 sources, bit for bit against the oracle.
* The left product x = M^T y on the genotype matrix: every column against the
  float64 oracle.
* The tropical (min, +) policy on both: every row of the genotype product, and
  the shortest-path fixpoint (unit lengths: hop distance to the nearest of the
  64 sources), bit for bit.

Grammars are built once per session (RePair takes a minute or two of host
time) and reused through the grammar cache when present.
"""
import numpy as np
import pytest

import gcsynth
from oracle import direct, reach

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 1e-4


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def medium(gcs):
    gen = gcsynth.GENO_MEDIUM
    rp, c, v = gcsynth.genotype_csr(**gen)
    G = gcs.cached_grammar(f"genotype:{sorted(gen.items())}", lambda: (gen["n"], gen["m"], rp, c, v))
    return gen, rp, c, v, G


def test_medium_single_vector_all_rows(gcs, torch, medium):
    gen, rp, c, v, G = medium
    st = G.stats()
    assert st["nnz"] == rp[-1] and st["depth"] >= 10
    eng = gcs.Engine(G, "f32", 1)
    assert eng.schedule == "persistent"
    for seed in (0, 99):
        x = gcsynth.beta(gen["m"], seed=seed)
        y = eng.matvec(torch.from_numpy(x).cuda()).cpu().numpy()
        assert eng.check() == 0
        y_ref, b = direct.matvec_f64(rp, c, v, x)
        ok, worst = direct.within_tolerance(y, y_ref, b, TOL)
        assert ok, f"seed {seed}: max scaled error {worst:.3e}"
    # footprint below the CSR of the same matrix
    lay = G.layout("f32", 1)
    assert lay["grammar_bytes"] + lay["scratch_bytes"] < lay["csr_bytes"]


def test_medium_sixteen_vectors(gcs, torch, medium):
    gen, rp, c, v, G = medium
    eng = gcs.Engine(G, "f32", 16)
    X = gcsynth.beta(gen["m"], seed=0, k=16)
    Y = eng.matvec(torch.from_numpy(X).cuda()).cpu().numpy()
    assert eng.check() == 0
    # every row, all 16 columns
    Y_ref, b = direct.matvec_f64(rp, c, v, X)
    ok, worst = direct.within_tolerance(Y, Y_ref, b, TOL)
    assert ok, f"max scaled error {worst:.3e}"


def test_graph_fixpoint(gcs, torch):
    gp = gcsynth.GRAPH
    rp, col = gcsynth.copy_model_graph(**gp)
    N = gp["nodes"]
    G = gcs.cached_grammar(f"graph:{sorted(gp.items())}", lambda: (N, N, rp, col, None))
    st = G.stats()
    assert st["nnz"] == len(col) > 1.5e8
    eng = gcs.Engine(G, "or", 1)
    x = np.random.default_rng(0).integers(0, 2**63, N, dtype=np.uint64)
    y = eng.matvec(torch.from_numpy(x.view(np.int64)).cuda()).cpu().numpy().view(np.uint64)
    np.testing.assert_array_equal(y, direct.matvec_or(rp, col, x))
    x0 = gcsynth.frontier(N, gcsynth.sources(N, gp["sources"], gp["seed"]))
    xs, iters, rc = eng.reach(torch.from_numpy(x0.view(np.int64)).cuda())
    assert rc == 0
    want, want_iters = reach.fixpoint(rp, col, x0)
    assert iters == want_iters
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint64), want)


def _same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a, np.float32).view(np.uint32),
                          np.ascontiguousarray(b, np.float32).view(np.uint32))


def test_medium_minplus_all_rows(gcs, torch, medium):
    gen, rp, c, v, G = medium
    eng = gcs.Engine(G, "minplus", 1)
    x = gcsynth.beta(gen["m"], seed=0)
    y = eng.matvec(torch.from_numpy(x).cuda()).cpu().numpy()
    assert eng.check() == 0
    assert _same_bits(y, direct.matvec_minplus(rp, c, v, x))


def test_graph_shortest_paths(gcs, torch):
    gp = gcsynth.GRAPH
    rp, col = gcsynth.copy_model_graph(**gp)
    N = gp["nodes"]
    G = gcs.cached_grammar(f"graph:{sorted(gp.items())}", lambda: (N, N, rp, col, None))
    eng = gcs.Engine(G, "minplus", 1)
    ones = np.ones(len(col), np.float32)
    x0 = gcsynth.frontier_distances(N, gcsynth.sources(N, gp["sources"], gp["seed"]))
    y = eng.matvec(torch.from_numpy(x0).cuda()).cpu().numpy()
    assert _same_bits(y, direct.matvec_minplus(rp, col, ones, x0))
    xs, iters, rc = eng.sssp(torch.from_numpy(x0).cuda())
    assert rc == 0
    want, want_iters = reach.sssp_fixpoint(rp, col, ones, x0)
    assert iters == want_iters
    assert _same_bits(xs.cpu().numpy(), want)


def test_medium_left_all_columns(gcs, torch, medium):
    gen, rp, c, v, G = medium
    eng = gcs.LeftEngine(G)
    y = gcsynth.beta(gen["n"], seed=5)
    x = eng.matvec(torch.from_numpy(y).cuda()).cpu().numpy()
    x_ref, b = direct.left_matvec_f64(rp, c, v, y, gen["m"])
    ok, worst = direct.within_tolerance(x, x_ref, b, TOL)
    assert ok, f"max scaled error {worst:.3e}"
