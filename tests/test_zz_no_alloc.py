"""gc_matvec_static: the product for callers that cannot allocate device memory
where it runs (their device memory is reserved up front, or they only receive
input and output buffers). Its scratch is a fixed array inside the library;
the test checks, through the C ABI, that two calls in a row give what
gc_matvec gives, within the float32 tolerance of the other parity tests, and
that a product too large for the array is refused with a clear error.

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


def _within(y_a, y_b, b):
    return np.all(np.abs(y_a.astype(np.float64) - y_b.astype(np.float64)) <= TOL * b)


@pytest.mark.parametrize("rows,k", [(None, 1), (None, 16), (600, 1)])
def test_static_scratch_matches_matvec(gcs, torch, rows, k):
    if rows is None:
        cfg = gcsynth.GENO_SMALL
    else:
        cfg = dict(gcsynth.GENO_MEDIUM, n=rows)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(cfg["n"], cfg["m"], rp, c, v)
    eng = gcs.Engine(G, "f32", k)
    capi = gcs.capi
    stream = torch.cuda.current_stream()
    shape = (cfg["n"],) if k == 1 else (cfg["n"], k)
    for seed in (11, 12):                       # two calls in a row share the array
        x_np = gcsynth.beta(cfg["m"], seed=seed, k=k)
        x = torch.from_numpy(x_np).cuda()
        y_ref = torch.empty(shape, device="cuda")
        capi.gc_matvec(eng._h, x, y_ref, k, stream)
        y_st = torch.full(shape, float("nan"), device="cuda")
        capi.gc_matvec_static(eng._h, x, y_st, k, stream)
        torch.cuda.synchronize()
        a, b_ = y_st.cpu().numpy(), y_ref.cpu().numpy()
        assert not np.isnan(a).any()
        _, bound = direct.matvec_f64(rp, c, v, x_np)
        assert _within(a, b_, bound)
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
