"""GPU parity: the CUDA sweep through the C ABI against the CPU oracle.

Tolerance for float32 (+, x): |y_i - y_ref_i| <= 1e-4 * (|M||x|)_i with y_i
exactly 0 where (|M||x|)_i = 0, y_ref in float64 (oracle.direct). Integer
and Boolean policies must match bit for bit.
"""
import numpy as np
import pytest

import gcsynth
from conftest import dense_to_csr
from oracle import direct, reach

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _dev(torch, a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def f32_product(gcs, torch, G, x, k_max=1):
    eng = gcs.Engine(G, "f32", k_max)
    y = eng.matvec(_dev(torch, x.astype(np.float32)))
    torch.cuda.synchronize()
    assert eng.check() == 0
    return y.cpu().numpy(), eng


def assert_f32_parity(y, rp, c, v, x):
    y_ref, b = direct.matvec_f64(rp, c, v, x.astype(np.float32))
    ok, worst = direct.within_tolerance(y, y_ref, b, TOL)
    assert ok, f"max scaled error {worst:.3e} > {TOL}"
    return worst


def _small_cases():
    for seed in range(4):
        rp, c, v, _ = gcsynth.random_sparse(5 + 7 * seed, 6 + 9 * seed, 0.5, [1.0, 2.0, -0.5, 3.25], seed)
        yield f"rand{seed}", len(rp) - 1, 6 + 9 * seed, rp, c, v
    d = gcsynth.genotype_dense(n=300, m=900, founders=6, switch=0.01, mutation=0.005, seed=4)
    rp, c, v = gcsynth.dense_to_csr(d)
    yield "geno300x900", 300, 900, rp, c, v


SMALL = list(_small_cases())


def test_worked_example_f32(gcs, torch, worked):
    rp, c, v = dense_to_csr(worked["M"], np.float32)
    G = gcs.Grammar(8, 7, rp, c, v)
    y, _ = f32_product(gcs, torch, G, worked["x"])
    b = np.abs(worked["M"]) @ np.abs(worked["x"])
    assert np.all(np.abs(y - worked["y"]) <= TOL * b)
    assert_f32_parity(y, rp, c, v, worked["x"])


@pytest.mark.parametrize("name,n,m,rp,c,v", SMALL, ids=[s[0] for s in SMALL])
def test_small_f32_k1_and_k16(gcs, torch, name, n, m, rp, c, v):
    G = gcs.Grammar(n, m, rp, c, v)
    x = np.random.default_rng(3).standard_normal(m).astype(np.float32)
    y, eng = f32_product(gcs, torch, G, x, k_max=16)
    assert_f32_parity(y, rp, c, v, x)
    X = np.random.default_rng(4).standard_normal((m, 16)).astype(np.float32)
    Y = eng.matvec(_dev(torch, X)).cpu().numpy()
    for col in range(16):
        assert_f32_parity(Y[:, col], rp, c, v, X[:, col])


@pytest.mark.parametrize("name,n,m,rp,c,v", SMALL, ids=[s[0] for s in SMALL])
def test_small_i64_exact(gcs, torch, name, n, m, rp, c, v):
    vi = np.round(v * 4).astype(np.float32)          # integer-valued matrix
    keep = vi != 0
    rp2 = np.concatenate([[0], np.cumsum([keep[rp[i]:rp[i + 1]].sum() for i in range(n)])]).astype(np.int64)
    c2, vi = c[keep], vi[keep]
    G = gcs.Grammar(n, m, rp2, c2, vi)
    x = np.random.default_rng(5).integers(-10**9, 10**9, m)
    eng = gcs.Engine(G, "i64", 1)
    y = eng.matvec(_dev(torch, x)).cpu().numpy()
    np.testing.assert_array_equal(y, direct.matvec_i64(rp2, c2, vi, x))


def test_genotype_small_config(gcs, torch):
    cfg = gcsynth.GENO_SMALL
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(cfg["n"], cfg["m"], rp, c, v)
    st = G.stats()
    assert st["depth"] > 3 and st["n_pass"] > 0
    x = gcsynth.beta(cfg["m"], seed=0)
    y, eng = f32_product(gcs, torch, G, x, k_max=16)
    assert_f32_parity(y, rp, c, v, x)
    # deterministic: the same input gives the same bits
    y2 = eng.matvec(_dev(torch, x)).cpu().numpy()
    np.testing.assert_array_equal(y, y2)
    # host-buffer entry point gives the same bits
    np.testing.assert_array_equal(eng.matvec_host(x), y)
    X = gcsynth.beta(cfg["m"], seed=1, k=16)
    Y = eng.matvec(_dev(torch, X)).cpu().numpy()
    y_ref, b = direct.matvec_f64(rp, c, v, X)
    ok, worst = direct.within_tolerance(Y, y_ref, b, TOL)
    assert ok, worst
    np.testing.assert_array_equal(eng.matvec_host(X), Y)
    # integer policy on the same matrix, exact
    xi = np.random.default_rng(9).integers(-1000, 1000, cfg["m"])
    ei = gcs.Engine(G, "i64", 1)
    np.testing.assert_array_equal(ei.matvec(_dev(torch, xi)).cpu().numpy(),
                                  direct.matvec_i64(rp, c, v, xi))


def test_genotype_wide_slice(gcs, torch):
    # 600 rows of the 50,000-variant generator: many tiles per level, ragged tails
    cfg = dict(gcsynth.GENO_MEDIUM, n=600)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(600, cfg["m"], rp, c, v)
    x = gcsynth.beta(cfg["m"], seed=7)
    y, _ = f32_product(gcs, torch, G, x)
    assert_f32_parity(y, rp, c, v, x)


def test_boolean_product_and_fixpoint(gcs, torch):
    N = 3000
    rp, col = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=1)
    G = gcs.Grammar(N, N, rp, col, None)
    eng = gcs.Engine(G, "or", 1)
    x = np.random.default_rng(2).integers(0, 2**63, N, dtype=np.uint64)
    y = eng.matvec(_dev(torch, x.view(np.int64))).cpu().numpy().view(np.uint64)
    np.testing.assert_array_equal(y, direct.matvec_or(rp, col, x))
    srcs = gcsynth.sources(N, 64, seed=0)
    x0 = gcsynth.frontier(N, srcs)
    xs, iters, rc = eng.reach(_dev(torch, x0.view(np.int64)))
    assert rc == 0
    want, want_iters = reach.fixpoint(rp, col, x0)
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint64), want)
    assert iters == want_iters
    # not converged within one product: status and iteration count say so
    xs1, iters1, rc1 = eng.reach(_dev(torch, x0.view(np.int64)), max_iter=1)
    assert rc1 == gcs.capi.GC_ERR_NOT_CONVERGED and iters1 == -1
    assert eng.check() == gcs.capi.GC_ERR_NOT_CONVERGED
    assert eng.check() == 0          # the status word is cleared once read


def test_edge_cases(gcs, torch):
    cases = [
        (4, 6, np.zeros(5, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32)),      # all rows empty
        (3, 3, np.array([0, 0, 1, 1], np.int64), np.array([2], np.int32), np.array([5.0], np.float32)),
        (2, 4, np.array([0, 2, 4], np.int64), np.array([0, 1, 2, 3], np.int32),
         np.array([1, 2, 3, 4], np.float32)),                                             # no rules (L = 0)
        (1, 1, np.array([0, 1], np.int64), np.array([0], np.int32), np.array([-2.5], np.float32)),
    ]
    for n, m, rp, c, v in cases:
        G = gcs.Grammar(n, m, rp, c, v)
        x = np.arange(1, m + 1, dtype=np.float32)
        y, _ = f32_product(gcs, torch, G, x)
        assert_f32_parity(y, rp, c, v, x)
    # long rows made of bare terminals plus one repeated row: C-heavy emit
    rp, c, v, _ = gcsynth.random_sparse(40, 3000, 0.4, [1.0, -1.0, 0.5], 8)
    G = gcs.Grammar(40, 3000, rp, c, v)
    x = np.random.default_rng(1).standard_normal(3000).astype(np.float32)
    y, _ = f32_product(gcs, torch, G, x)
    assert_f32_parity(y, rp, c, v, x)


def test_argument_errors(gcs, torch):
    rp, c, v, _ = gcsynth.random_sparse(20, 30, 0.5, [1.0, 2.0], 0)
    G = gcs.Grammar(20, 30, rp, c, v)
    eng = gcs.Engine(G, "f32", 1)
    X = torch.zeros((30, 16), device="cuda")
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        eng.matvec(X)                                 # k = 16 on a k_max = 1 handle
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_reach(eng._h, X, X, 5, X)        # reach needs the OR policy
    arena = torch.empty(G.layout("f32", 1)["arena_bytes"] + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_upload(G._p, "f32", 1, arena.data_ptr() + 16, arena.numel() - 16)
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_upload(G._p, "f32", 1, arena, 1024)


def test_schedules_agree_bit_for_bit(gcs, torch):
    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(300, cfg["m"], rp, c, v)
    eng = gcs.Engine(G, "f32", 16)
    assert eng.schedule == "persistent"          # cooperative launch on this GPU
    x = _dev(torch, gcsynth.beta(cfg["m"], seed=3))
    y_p = eng.matvec(x).cpu().numpy()
    assert eng.launch_count() == 1
    X = _dev(torch, gcsynth.beta(cfg["m"], seed=4, k=16))
    Y_p = eng.matvec(X).cpu().numpy()
    eng.schedule = "per_level"
    assert eng.schedule == "per_level"
    y_l = eng.matvec(x).cpu().numpy()
    # one kernel per level, then the emit (one kernel, or chunks + row sums)
    assert G.stats()["depth"] + 1 <= eng.launch_count() <= G.stats()["depth"] + 2
    Y_l = eng.matvec(X).cpu().numpy()
    np.testing.assert_array_equal(y_p, y_l)
    np.testing.assert_array_equal(Y_p, Y_l)
    assert_f32_parity(y_p, rp, c, v, gcsynth.beta(cfg["m"], seed=3))


@pytest.mark.parametrize("policy", ["f32", "i64", "or", "minplus"])
def test_dataflow_and_per_level_agree(gcs, torch, policy):
    # one value a node: the dataflow sweep (one cooperative launch, blocks
    # started by ready flags) and its per-level launch sequence give the same
    # bits, and both match the oracle; slice emit (long rows) and row emit
    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    rp2, col2 = gcsynth.copy_model_graph(nodes=3000, n0=20, d0=15, p_edit=0.05, seed=1)
    for n, m, rp_, c_, v_ in ((300, cfg["m"], rp, c, v), (3000, 3000, rp2, col2, np.ones(len(col2), np.float32))):
        if policy == "or":
            v_ = np.ones_like(v_)
        G = gcs.Grammar(n, m, rp_, c_, v_)
        assert gcs.Engine(G, policy, 1).schedule == "persistent"     # the default layout
        eng = gcs.Engine(G, policy, 1, schedule="dataflow")
        assert eng.schedule == "dataflow"
        rng = np.random.default_rng(n)
        if policy == "f32":
            x = gcsynth.beta(m, seed=9)
        elif policy == "minplus":
            x = rng.integers(0, 40, m).astype(np.float32)
        else:
            x = rng.integers(-500, 500, m).astype(np.int64) if policy == "i64" else \
                rng.integers(0, 2**63, m, dtype=np.int64)
        xd = _dev(torch, x)
        y_d = eng.matvec(xd).cpu().numpy()
        assert eng.check() == 0
        launches_d = eng.launch_count()
        eng.schedule = "per_level"
        y_l = eng.matvec(xd).cpu().numpy()
        assert eng.launch_count() >= launches_d   # a launch per level with regular blocks, one for the final block
        eng.schedule = "persistent"              # on this handle: the dataflow schedule
        assert eng.schedule == "dataflow"
        np.testing.assert_array_equal(y_d.view(np.uint8), y_l.view(np.uint8))
        if policy == "f32":
            assert_f32_parity(y_d, rp_, c_, v_, x)
        elif policy == "minplus":
            np.testing.assert_array_equal(y_d.view(np.uint32), direct.matvec_minplus(rp_, c_, v_, x).view(np.uint32))
        elif policy == "i64":
            np.testing.assert_array_equal(y_d, direct.matvec_i64(rp_, c_, v_, x))
        else:
            np.testing.assert_array_equal(y_d.view(np.uint64), direct.matvec_or(rp_, c_, x.view(np.uint64)))
        # repeated products on the same handle (the ready flags carry the product number)
        for _ in range(3):
            np.testing.assert_array_equal(eng.matvec(xd).cpu().numpy().view(np.uint8), y_d.view(np.uint8))
        assert eng.check() == 0


def test_dataflow_fixpoints_and_timeout(gcs, torch):
    # the Boolean and tropical fixpoints on dataflow handles (device-side
    # loop), against the oracle; then a dependency wait that runs out (CTA 0
    # never publishes its first block) is reported, not hung, and the handle
    # computes correctly after gc_check
    rp, col = gcsynth.copy_model_graph(nodes=20000, n0=40, d0=20, p_edit=0.05, seed=3)
    n = 20000
    ones = np.ones(len(col), np.float32)
    G = gcs.Grammar(n, n, rp, col, ones)
    srcs = gcsynth.sources(n, 64, 3)
    eng = gcs.Engine(G, "or", 1, schedule="dataflow")
    x0 = gcsynth.frontier(n, srcs)
    x, iters, rc = eng.reach(_dev(torch, x0.view(np.int64)))
    assert rc == 0 and iters >= 2
    want, want_iters = reach.fixpoint(rp, col, x0)
    np.testing.assert_array_equal(x.cpu().numpy().view(np.uint64), want)
    assert iters == want_iters
    mp = gcs.Engine(G, "minplus", 1, schedule="dataflow")
    d0 = gcsynth.frontier_distances(n, srcs)
    d, it2, rc2 = mp.sssp(_dev(torch, d0))
    assert rc2 == 0
    want_d, want_it = reach.sssp_fixpoint(rp, col, ones, d0)
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint32), want_d.view(np.uint32))
    assert it2 == want_it
    # the injected timeout
    cfg = dict(gcsynth.GENO_MEDIUM, n=200)
    rp3, c3, v3 = gcsynth.genotype_csr(**cfg)
    G3 = gcs.Grammar(200, cfg["m"], rp3, c3, v3)
    e3 = gcs.Engine(G3, "f32", 1, schedule="dataflow")
    xg = _dev(torch, gcsynth.beta(cfg["m"], seed=5))
    y_ok = e3.matvec(xg).cpu().numpy()
    gcs.capi.gc_debug_inject(e3._h, 1, 2_000_000)
    e3.matvec(xg)
    torch.cuda.synchronize()
    assert e3.check() == gcs.capi.GC_ERR_TIMEOUT
    gcs.capi.gc_debug_inject(e3._h, 0, 4_000_000_000)
    np.testing.assert_array_equal(e3.matvec(xg).cpu().numpy(), y_ok)
    assert e3.check() == 0


def test_barrier_timeout_is_reported_not_hung(gcs, torch):
    # CTA 0 skips its first barrier arrival; every other CTA's bounded wait
    # runs out (about a millisecond), the kernel returns with GC_ERR_TIMEOUT
    cfg = dict(gcsynth.GENO_MEDIUM, n=200)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(200, cfg["m"], rp, c, v)
    eng = gcs.Engine(G, "f32", 1)
    x = _dev(torch, gcsynth.beta(cfg["m"], seed=5))
    y_ok = eng.matvec(x).cpu().numpy()
    gcs.capi.gc_debug_inject(eng._h, 1, 2_000_000)
    y = torch.full((200,), float("nan"), device="cuda")
    eng.matvec(x, y)
    torch.cuda.synchronize()
    assert eng.check() == gcs.capi.GC_ERR_TIMEOUT
    assert eng.check() == 0
    # while a timeout is unread, products are skipped
    gcs.capi.gc_debug_inject(eng._h, 1, 2_000_000)
    eng.matvec(x, y)
    y2 = torch.full((200,), float("nan"), device="cuda")
    gcs.capi.gc_debug_inject(eng._h, 0, 4_000_000_000)
    eng.matvec(x, y2)
    assert torch.isnan(y2).all()
    assert eng.check() == gcs.capi.GC_ERR_TIMEOUT
    # after the check the same handle computes correctly again
    np.testing.assert_array_equal(eng.matvec(x).cpu().numpy(), y_ok)
    assert eng.check() == 0


@pytest.mark.parametrize("k", [4, 8, 32, 64, 128, 256])
def test_batch_widths(gcs, torch, k):
    # Appendix A's batched product at every width the float32 sum takes:
    # a slice of the 50,000-variant generator (level emit, carry slots, a
    # tail) and a short-row genotype matrix (row emit); every row and column
    # against the float64 oracle, both schedules bit for bit, the
    # allocation-free entry point bit for bit, and a one-vector product on
    # the same handle
    cfg = dict(gcsynth.GENO_MEDIUM, n=200)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    d = gcsynth.genotype_dense(n=300, m=900, founders=6, switch=0.01, mutation=0.005, seed=4)
    rp2, c2, v2 = gcsynth.dense_to_csr(d)
    for n, m, rp_, c_, v_ in ((200, cfg["m"], rp, c, v), (300, 900, rp2, c2, v2)):
        G = gcs.Grammar(n, m, rp_, c_, v_)
        eng = gcs.Engine(G, "f32", k)
        X = gcsynth.beta(m, seed=k, k=k)
        Xd = _dev(torch, X)
        Y = eng.matvec(Xd).cpu().numpy()
        assert eng.check() == 0
        y_ref, b = direct.matvec_f64(rp_, c_, v_, X)
        ok, worst = direct.within_tolerance(Y, y_ref, b, TOL)
        assert ok, f"k={k} n={n}: max scaled error {worst:.3e}"
        eng.schedule = "per_level"
        np.testing.assert_array_equal(eng.matvec(Xd).cpu().numpy(), Y)
        eng.schedule = "persistent"
        if eng.layout["scratch_bytes"] < gcs.capi.GC_STATIC_SCRATCH_BYTES // 2:
            Ys = torch.empty((n, k), dtype=torch.float32, device="cuda")
            gcs.capi.gc_matvec_static(eng._h, Xd, Ys, k)
            np.testing.assert_array_equal(Ys.cpu().numpy(), Y)
        x1 = gcsynth.beta(m, seed=1)
        y1 = eng.matvec(_dev(torch, x1)).cpu().numpy()
        assert_f32_parity(y1, rp_, c_, v_, x1)
    # a narrower supported width runs on the wide handle; other widths are refused
    if k >= 8:
        Xn = _dev(torch, gcsynth.beta(m, seed=2, k=4))
        Yn = eng.matvec(Xn).cpu().numpy()
        y_ref, b = direct.matvec_f64(rp_, c_, v_, gcsynth.beta(m, seed=2, k=4))
        assert direct.within_tolerance(Yn, y_ref, b, TOL)[0]
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        eng.matvec(torch.zeros((m, 12), device="cuda"))


def test_fixpoint_loop_edges_and_streams(gcs, torch):
    # the loop keeps one batch enqueued ahead: max_iter at and just below
    # the product count, a product on another stream straight after the
    # call returns (ordered after the loop's last batch), and a handle freed
    # with the last batch still on the stream
    N = 3000
    rp, col = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=3)
    G = gcs.Grammar(N, N, rp, col, None)
    x0 = gcsynth.frontier(N, gcsynth.sources(N, 64, seed=1))
    want, want_iters = reach.fixpoint(rp, col, x0)
    assert want_iters >= 3
    for sched in ("persistent", "dataflow"):
        eng = gcs.Engine(G, "or", 1, schedule=sched)
        x0d = _dev(torch, x0.view(np.int64))
        xs, iters, rc = eng.reach(x0d, max_iter=want_iters)
        assert rc == 0 and iters == want_iters
        np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint64), want)
        xs, iters, rc = eng.reach(x0d, max_iter=want_iters - 1)
        assert rc == gcs.capi.GC_ERR_NOT_CONVERGED and iters == -1
        assert eng.check() == gcs.capi.GC_ERR_NOT_CONVERGED
        assert eng.check() == 0
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        xr = torch.empty_like(x0d)
        it = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        assert gcs.capi.gc_reach(eng._h, x0d, xr, 1000, it, s1) == 0
        xv = _dev(torch, want.view(np.int64))
        yv = torch.empty_like(xv)
        torch.cuda.synchronize()
        eng.matvec(xv, yv, stream=s2)
        s2.synchronize()
        s1.synchronize()
        np.testing.assert_array_equal(yv.cpu().numpy().view(np.uint64), direct.matvec_or(rp, col, want))
        np.testing.assert_array_equal(xr.cpu().numpy().view(np.uint64), want)
        assert int(it.item()) == want_iters
        assert gcs.capi.gc_reach(eng._h, x0d, xr, 1000, it, s1) == 0
        del eng                          # freed with the last batch possibly still running
        s1.synchronize()
        np.testing.assert_array_equal(xr.cpu().numpy().view(np.uint64), want)


def test_fixpoint_in_one_launch_and_its_timeout(gcs, torch):
    # row-emit handles (the graph) run the whole fixpoint in one persistent
    # launch; a handle with the slice emit (long rows) keeps the batched loop.
    # Both against the oracle; then an injected barrier timeout inside the
    # one-launch fixpoint is reported, and the handle recovers after gc_check
    N = 3000
    rp, col = gcsynth.copy_model_graph(nodes=N, n0=20, d0=15, p_edit=0.05, seed=5)
    G = gcs.Grammar(N, N, rp, col, None)
    eng = gcs.Engine(G, "or", 1)
    x0 = gcsynth.frontier(N, gcsynth.sources(N, 64, seed=2))
    want, want_iters = reach.fixpoint(rp, col, x0)
    xs, iters, rc = eng.reach(_dev(torch, x0.view(np.int64)))
    assert rc == 0 and iters == want_iters and eng.launch_count() == 1
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint64), want)
    # products after the fixpoint still compute (barrier counters consistent)
    xv = _dev(torch, want.view(np.int64))
    np.testing.assert_array_equal(eng.matvec(xv).cpu().numpy().view(np.uint64), direct.matvec_or(rp, col, want))
    gcs.capi.gc_debug_inject(eng._h, 1, 2_000_000)
    _, iters_t, rc_t = eng.reach(_dev(torch, x0.view(np.int64)))
    assert rc_t == gcs.capi.GC_ERR_NOT_CONVERGED and iters_t == -1
    assert eng.check() == gcs.capi.GC_ERR_TIMEOUT
    gcs.capi.gc_debug_inject(eng._h, 0, 4_000_000_000)
    xs, iters, rc = eng.reach(_dev(torch, x0.view(np.int64)))
    assert rc == 0 and iters == want_iters
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint64), want)
    assert eng.check() == 0
    # a square matrix with long rows: the slice emit, the batched loop
    n = 800
    rp2, c2, v2, _ = gcsynth.random_sparse(n, n, 0.5, [1.0, 2.0, 3.0], 9)   # |C| / n about 193
    G2 = gcs.Grammar(n, n, rp2, c2, v2)
    mp = gcs.Engine(G2, "minplus", 1)
    d0 = np.full(n, np.inf, np.float32)
    d0[[3, 77]] = 0.0
    d, it2, rc2 = mp.sssp(_dev(torch, d0))
    want_d, want_it = reach.sssp_fixpoint(rp2, c2, v2, d0)
    assert rc2 == 0 and it2 == want_it and mp.launch_count() > 1
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint32), want_d.view(np.uint32))
    # a barrier timeout inside the batched loop: not converged, the status
    # word keeps the timeout, and the handle recovers after gc_check
    gcs.capi.gc_debug_inject(mp._h, 1, 2_000_000)
    _, it3, rc3 = mp.sssp(_dev(torch, d0), max_iter=5)
    assert rc3 == gcs.capi.GC_ERR_NOT_CONVERGED and it3 == -1
    assert mp.check() == gcs.capi.GC_ERR_TIMEOUT
    gcs.capi.gc_debug_inject(mp._h, 0, 4_000_000_000)
    d, it2, rc2 = mp.sssp(_dev(torch, d0))
    assert rc2 == 0 and it2 == want_it
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint32), want_d.view(np.uint32))
    assert mp.check() == 0
