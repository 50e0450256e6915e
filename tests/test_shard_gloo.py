"""Row-block sharding over two ranks (gloo, CPU): the multi-rank logic of
grammar_compressed_sparse_gb300.shard, with no GPU.

Each rank builds the grammar of its own rows (whole 64-row blocks) with the
host builder, evaluates its rows of the product with the CPU emulator of the
packed layout (a stand-in for the device sweep) and updates them with CPU
stand-ins of the library's update step, and the ranks gather the rows; the
fixpoints gather the new vector and all-reduce the changed flag (a bool from
one stand-in, a tensor from the other) once per iteration. The GPU path
(ShardedEngine, gc_update) is tested on one rank in test_gpu_shard.py. Everything is compared with the oracle on the whole
matrix, on every rank.
"""
import os
import socket

import numpy as np
import pytest

import gcsynth
from conftest import export_all
from oracle import direct, reach
from packed_emulator import emulate


def test_row_shards_cover_in_order():
    from grammar_compressed_sparse_gb300.shard import row_shards
    for n, world, block in [(10, 3, 0), (1000, 4, 64), (100, 8, 64), (0, 2, 0), (7, 1, 3)]:
        sh = row_shards(n, world, block)
        assert len(sh) == world and sh[0][0] == 0 and sh[-1][1] == n
        for (a0, a1), (b0, b1) in zip(sh, sh[1:]):
            assert a1 == b0 and a0 <= a1
        if block:
            assert all(r0 % block == 0 for r0, _ in sh)
    assert row_shards(100, 8, 64) == [(0, 0), (0, 0), (0, 0), (0, 64), (64, 64), (64, 64), (64, 64), (64, 100)]
    with pytest.raises(ValueError):
        row_shards(10, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, errors):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import grammar_compressed_sparse_gb300 as gcs
        from grammar_compressed_sparse_gb300.shard import gather_rows, local_rows, row_shards, sharded_fixpoint

        # CPU stand-ins of the library's update step (gc_update runs on the GPU)
        def or_update(old, new):
            out = old | new
            return out, bool((out != old).any())

        def min_update(old, new):
            out = torch.minimum(old, new)
            return out, torch.tensor([int((out != old).any())], dtype=torch.int32)
        # genotype rows: y = G beta, rows sharded by 64-row blocks
        cfg = dict(gcsynth.GENO_SMALL, n=300, m=900)
        rp, c, v = gcsynth.genotype_csr(**cfg)
        sh = row_shards(300, world, 64)
        r0, r1 = sh[rank]
        lrp, lc, lv = local_rows(rp, c, v, r0, r1)
        ex = export_all(gcs.Grammar(r1 - r0, 900, lrp, lc, lv))
        x = gcsynth.beta(900, seed=1)
        y = gather_rows(torch.from_numpy(emulate(ex, x)), sh).numpy()
        y_ref, b = direct.matvec_f64(rp, c, v, x)
        assert direct.within_tolerance(y, y_ref, b, 1e-9)[0], "sharded product"

        # copy-model graph: reachability and shortest paths, rows sharded
        N = 1500
        grp, gcol = gcsynth.copy_model_graph(nodes=N, n0=20, d0=12, p_edit=0.05, seed=3)
        w = gcsynth.target_lengths(gcol, N, seed=4)
        gsh = row_shards(N, world, 64)
        g0, g1 = gsh[rank]
        prp, pc, _ = local_rows(grp, gcol, None, g0, g1)
        exo = export_all(gcs.Grammar(g1 - g0, N, prp, pc, None))
        _, _, pw = local_rows(grp, gcol, w, g0, g1)
        exw = export_all(gcs.Grammar(g1 - g0, N, prp, pc, pw))
        srcs = gcsynth.sources(N, 64, seed=0)
        x0 = gcsynth.frontier(N, srcs)
        xs, iters = sharded_fixpoint(
            lambda xt: torch.from_numpy(emulate(exo, xt.numpy().view(np.uint64), "or").view(np.int64)),
            torch.from_numpy(x0.view(np.int64)), gsh, or_update)
        want, want_iters = reach.fixpoint(grp, gcol, x0)
        assert iters == want_iters and np.array_equal(xs.numpy().view(np.uint64), want), "sharded reachability"
        d0 = gcsynth.frontier_distances(N, srcs[:4])
        ds, diters = sharded_fixpoint(lambda xt: torch.from_numpy(emulate(exw, xt.numpy(), "minplus")),
                                      torch.from_numpy(d0), gsh, min_update)
        dwant, dwant_iters = reach.sssp_fixpoint(grp, gcol, w, d0)
        assert diters == dwant_iters and np.array_equal(ds.numpy(), dwant), "sharded shortest paths"
    except Exception as e:   # reported to the parent
        errors.put(f"rank {rank}: {type(e).__name__}: {e}")
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo(gcs):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    errors = ctx.Queue()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, errors), nprocs=2, join=True, start_method="spawn")
    msgs = []
    while not errors.empty():
        msgs.append(errors.get())
    assert not msgs, "; ".join(msgs)
