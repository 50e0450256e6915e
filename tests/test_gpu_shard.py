"""The row-sharded GPU path on one rank (NCCL, world size 1): ShardedEngine
builds the rank's row-block grammar and runs the library's products, and the
fixpoints' update step runs in the library (gc_update); all against the CPU
oracle. Several ranks run as gloo processes on the CPU (test_shard_gloo.py)."""
import os
import socket

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


@pytest.fixture(scope="module")
def group(torch):
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    yield None
    dist.destroy_process_group()


def test_gc_update_matches_numpy(gcs, torch):
    rng = np.random.default_rng(0)
    for n in (0, 1, 1000, 300001):
        a = rng.integers(0, 2**63, n, dtype=np.int64)
        b = rng.integers(0, 2**63, n, dtype=np.int64) & rng.integers(0, 2**63, n, dtype=np.int64)
        x = torch.from_numpy(a.copy()).cuda()
        ch = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        gcs.capi.gc_update("or", x, torch.from_numpy(b).cuda(), n, ch)
        np.testing.assert_array_equal(x.cpu().numpy(), a | b)
        assert int(ch.item()) == int(((a | b) != a).any())
        # no change: flag 0
        gcs.capi.gc_update("or", x, torch.from_numpy(b).cuda(), n, ch)
        assert int(ch.item()) == 0
        f = rng.standard_normal(n).astype(np.float32)
        g = rng.standard_normal(n).astype(np.float32)
        f[::3] = np.inf
        xf = torch.from_numpy(f.copy()).cuda()
        gcs.capi.gc_update("minplus", xf, torch.from_numpy(g).cuda(), n, ch)
        np.testing.assert_array_equal(xf.cpu().numpy(), np.minimum(f, g))
        assert int(ch.item()) == int((np.minimum(f, g) != f).any())
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.capi.gc_update("f32", x, x, 1, ch)


def test_sharded_engine_one_rank(gcs, torch, group):
    from grammar_compressed_sparse_gb300.shard import ShardedEngine, local_rows
    cfg = dict(gcsynth.GENO_SMALL, n=300, m=900)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    se = ShardedEngine(300, 900, lambda r0, r1: local_rows(rp, c, v, r0, r1), block_rows=64)
    x = gcsynth.beta(900, seed=1)
    y = se.matvec(torch.from_numpy(x).cuda()).cpu().numpy()
    y_ref, b = direct.matvec_f64(rp, c, v, x)
    assert direct.within_tolerance(y, y_ref, b, 1e-4)[0]

    N = 1500
    grp, gcol = gcsynth.copy_model_graph(nodes=N, n0=20, d0=12, p_edit=0.05, seed=3)
    w = gcsynth.target_lengths(gcol, N, seed=4)
    srcs = gcsynth.sources(N, 64, seed=0)
    x0 = gcsynth.frontier(N, srcs)
    for balance in (False, True):
        so = ShardedEngine(N, N, lambda r0, r1: local_rows(grp, gcol, None, r0, r1), policy="or", block_rows=64,
                           balance=balance)
        xs, iters = so.reach(torch.from_numpy(x0.view(np.int64)).cuda())
        want, want_iters = reach.fixpoint(grp, gcol, x0)
        assert iters == want_iters
        np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint64), want)
    sm = ShardedEngine(N, N, lambda r0, r1: local_rows(grp, gcol, w, r0, r1), policy="minplus", block_rows=64)
    d0 = gcsynth.frontier_distances(N, srcs[:4])
    ds, diters = sm.sssp(torch.from_numpy(d0).cuda())
    dwant, dwant_iters = reach.sssp_fixpoint(grp, gcol, w, d0)
    assert diters == dwant_iters
    assert np.array_equal(ds.cpu().numpy().view(np.uint32), dwant.view(np.uint32))
