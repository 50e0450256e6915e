"""gc_matvec_static: the product for callers that cannot allocate device memory
where it runs (their device memory is reserved up front, or they only receive
input and output buffers). Its scratch is a fixed array inside the library.

Through the C ABI, two calls in a row (the array keeps the previous call's
contents) must give what gc_matvec gives, bit for bit -- both run the same
kernels in the same order -- and what the oracle gives: within the float32
tolerance of the other parity tests for the float32 sum, bit for bit for the
exact, Boolean and tropical policies. A product too large for the array is
refused with a clear error.

Kept in its own file so pytest collects it last.
"""
import numpy as np
import pytest

import gcsynth
from oracle import direct

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _inputs(policy, m, k, seed):
    """x for the policy (numpy), the torch dtype it travels in."""
    rng = np.random.default_rng(seed)
    if policy == "f32":
        return gcsynth.beta(m, seed=seed, k=k)
    if policy == "minplus":
        x = rng.integers(0, 50, size=(m,) if k == 1 else (m, k)).astype(np.float32)
        x[rng.random(x.shape) < 0.1] = np.inf
        return x
    if policy == "i64":
        return rng.integers(-1000, 1000, size=m).astype(np.int64)
    return rng.integers(0, 2**63, size=m, dtype=np.int64)   # "or": 64 bit lanes


def _oracle_check(policy, rp, c, v, x_np, y):
    if policy == "f32":
        y_ref, bound = direct.matvec_f64(rp, c, v, x_np.astype(np.float64))
        ok, worst = direct.within_tolerance(y, y_ref, bound, TOL)
        assert ok, worst
    elif policy == "minplus":
        assert np.array_equal(y.view(np.uint32), direct.matvec_minplus(rp, c, v, x_np).view(np.uint32))
    elif policy == "i64":
        assert np.array_equal(y, direct.matvec_i64(rp, c, v.astype(np.int64), x_np))
    else:
        assert np.array_equal(y.view(np.uint64), direct.matvec_or(rp, c, x_np.view(np.uint64)))


CASES = [
    ("small", "f32", 1, 1, "persistent"), ("small", "f32", 16, 16, "persistent"),
    ("small", "f32", 16, 4, "persistent"), ("rows600", "f32", 1, 1, "persistent"),
    ("small", "i64", 1, 1, "persistent"), ("small", "or", 1, 1, "persistent"),
    ("small", "minplus", 1, 1, "persistent"), ("small", "minplus", 16, 16, "persistent"),
    ("small", "f32", 1, 1, "dataflow"), ("rows600", "or", 1, 1, "dataflow"),
]


@pytest.mark.parametrize("mat,policy,k_max,k,schedule", CASES)
def test_static_scratch_matches_matvec(gcs, torch, mat, policy, k_max, k, schedule):
    cfg = gcsynth.GENO_SMALL if mat == "small" else dict(gcsynth.GENO_MEDIUM, n=600)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    if policy == "or":
        v = np.ones_like(v)
    G = gcs.Grammar(cfg["n"], cfg["m"], rp, c, v)
    eng = gcs.Engine(G, policy, k_max, schedule=schedule)
    capi = gcs.capi
    stream = torch.cuda.current_stream()
    shape = (cfg["n"],) if k == 1 else (cfg["n"], k)
    tdt = torch.float32 if policy in ("f32", "minplus") else torch.int64
    for seed in (11, 12):                       # two calls in a row share the array
        x_np = _inputs(policy, cfg["m"], k, seed)
        x = torch.from_numpy(x_np).cuda()
        y_ref = torch.empty(shape, dtype=tdt, device="cuda")
        capi.gc_matvec(eng._h, x, y_ref, k, stream)
        y_st = torch.full(shape, -7, dtype=tdt, device="cuda")
        capi.gc_matvec_static(eng._h, x, y_st, k, stream)
        torch.cuda.synchronize()
        a, b_ = y_st.cpu().numpy(), y_ref.cpu().numpy()
        # same kernels, same order of evaluation: the same bits
        assert np.array_equal(a.view(np.uint8), b_.view(np.uint8))
        _oracle_check(policy, rp, c, v, x_np, a)
    assert eng.check() == 0


def test_static_scratch_refuses_oversize(gcs, torch):
    cfg = dict(gcsynth.GENO_MEDIUM, n=600)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(cfg["n"], cfg["m"], rp, c, v)
    eng = gcs.Engine(G, "f32", 16)              # 16 wide: far beyond the fixed array
    X = torch.zeros((cfg["m"], 16), device="cuda")
    Y = torch.zeros((cfg["n"], 16), device="cuda")
    with pytest.raises(gcs.GcError, match="GC_ERR_UNSUPPORTED") as e:
        gcs.capi.gc_matvec_static(eng._h, X, Y, 16, torch.cuda.current_stream())
    assert "bytes of scratch" in str(e.value)
