"""GPU parity over height-balanced (AVL) grammars: the same products as the
RePair grammar's, checked against the CPU oracle under every policy and
schedule. Integer and Boolean results must equal the unbalanced grammar's
bit for bit; float32 stays within the 1e-4 * (|M||x|)_i bound."""
import numpy as np
import pytest

import gcsynth
from oracle import direct, reach

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("schedule", ["persistent", "per_level", "dataflow"])
def test_balanced_genotype_products(gcs, torch, schedule):
    cfg = dict(gcsynth.GENO_MEDIUM, n=400)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(cfg["n"], cfg["m"], rp, c, v)
    B = G.balanced()
    assert B.stats()["depth"] < G.stats()["depth"]
    x = gcsynth.beta(cfg["m"], seed=3)
    xi = np.random.default_rng(4).integers(-1000, 1000, cfg["m"])
    y_ref, b = direct.matvec_f64(rp, c, v, x)
    yi_ref = direct.matvec_i64(rp, c, v, xi)
    sched = "dataflow" if schedule == "dataflow" else "persistent"
    ef = gcs.Engine(B, "f32", 1, schedule=sched)
    ei = gcs.Engine(B, "i64", 1, schedule=sched)
    if schedule == "per_level":
        ef.schedule = ei.schedule = "per_level"
    y = ef.matvec(_dev(torch, x)).cpu().numpy()
    ok, worst = direct.within_tolerance(y, y_ref, b, TOL)
    assert ok, worst
    assert ef.check() == 0
    np.testing.assert_array_equal(ei.matvec(_dev(torch, xi)).cpu().numpy(), yi_ref)
    assert ei.check() == 0
    if schedule == "persistent":
        # k = 16 on the balanced grammar, every column
        e16 = gcs.Engine(B, "f32", 16)
        X = gcsynth.beta(cfg["m"], seed=5, k=16)
        Y = e16.matvec(_dev(torch, X)).cpu().numpy()
        y_ref16, b16 = direct.matvec_f64(rp, c, v, X)
        ok, worst = direct.within_tolerance(Y, y_ref16, b16, TOL)
        assert ok, worst


def test_balanced_graph_reach(gcs, torch):
    N = 3000
    rp, col = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=1)
    G = gcs.Grammar(N, N, rp, col, None)
    B = G.balanced()
    assert B.stats()["depth"] <= G.stats()["depth"]
    x = np.random.default_rng(2).integers(0, 2**63, N, dtype=np.uint64)
    want = direct.matvec_or(rp, col, x)
    for sched in ("persistent", "dataflow"):
        eng = gcs.Engine(B, "or", 1, schedule=sched)
        y = eng.matvec(_dev(torch, x.view(np.int64))).cpu().numpy().view(np.uint64)
        np.testing.assert_array_equal(y, want)
        x0 = gcsynth.frontier(N, gcsynth.sources(N, 64, seed=0))
        xs, iters, rc = eng.reach(_dev(torch, x0.view(np.int64)))
        assert rc == 0
        fx, fit = reach.fixpoint(rp, col, x0)
        np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint64), fx)
        assert iters == fit
