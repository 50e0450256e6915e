"""Row-blocked grammars on the GPU (the pages' Sec. 1 row-block partitioning;
the 50,000 x 200,000 workload is built one 5,000-row block at a time).

A reduced matrix of the same structure -- the 500-founder generator with
switch = mutation = 5e-4, 4 blocks of 1,000 rows, 20,000 columns -- is built
two ways: by gc_build with block_rows (blocks compressed one after the other
in one call) and by the streaming builder (Grammar.from_row_blocks, blocks
compressed concurrently as they are generated). Both must be the same grammar
(blocks merged level by level, rules numbered block after block), and every
row of y = M x must match the float64 oracle at k = 1 (persistent sweep and
the dataflow schedule, slice emit) and k = 16 (level emit), with the two builds
giving the same bits.
"""
import numpy as np
import pytest

import gcsynth
from oracle import direct

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 1e-4
CFG = dict(gcsynth.GENO_LARGE, n=4000, m=20000, block_rows=1000)


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def blocked(gcs):
    rp, c, v = gcsynth.genotype_csr(**CFG)
    G1 = gcs.Grammar(CFG["n"], CFG["m"], rp, c, v, block_rows=CFG["block_rows"])
    G2 = gcs.Grammar.from_row_blocks(CFG["n"], CFG["m"], CFG["block_rows"],
                                     lambda r0, r1: gcsynth.genotype_csr(**CFG, r0=r0, r1=r1), workers=4)
    return rp, c, v, G1, G2


def test_blocked_builds_agree(gcs, blocked):
    rp, c, v, G1, G2 = blocked
    s1, s2 = G1.stats(), G2.stats()
    assert s1["n_blocks"] == s2["n_blocks"] == 4
    assert s1["nnz"] == s2["nnz"] == rp[-1]
    for key in ("n_rules", "n_pass", "depth", "max_width", "c_len", "n_roots"):
        assert s1[key] == s2[key], key
    np.testing.assert_array_equal(G1.export("nodes"), G2.export("nodes"))
    np.testing.assert_array_equal(G1.export("c_ref"), G2.export("c_ref"))


@pytest.mark.parametrize("k", [1, 16])
def test_blocked_every_row(gcs, torch, blocked, k):
    rp, c, v, G1, G2 = blocked
    X = gcsynth.beta(CFG["m"], seed=k, k=k)
    y_ref, b = direct.matvec_f64(rp, c, v, X)
    ys = []
    for G in (G1, G2):
        eng = gcs.Engine(G, "f32", k)
        assert eng.schedule == "persistent"
        Y = eng.matvec(torch.from_numpy(X).cuda()).cpu().numpy()
        assert eng.check() == 0
        ok, worst = direct.within_tolerance(Y, y_ref, b, TOL)
        assert ok, f"k={k}: max scaled error {worst:.3e}"
        ys.append(Y)
        if k == 1:   # the dataflow schedule's own layout: the same bits
            eng_d = gcs.Engine(G, "f32", 1, schedule="dataflow")
            Yd = eng_d.matvec(torch.from_numpy(X).cuda()).cpu().numpy()
            assert eng_d.check() == 0
            ok, worst = direct.within_tolerance(Yd, y_ref, b, TOL)
            assert ok, f"dataflow: max scaled error {worst:.3e}"
        lay = G.layout("f32", k)
        if k == 1:
            assert lay["grammar_bytes"] + lay["scratch_bytes"] < lay["csr_bytes"]
    np.testing.assert_array_equal(ys[0], ys[1])
