"""Row-block sharding of the product over several ranks (host-side plumbing).

The right product shards by rows: blocks of rows are independent grammars
(the row-block build, Sec. 1 "row blocks" of the pages), x is replicated and
each rank's rows of y are disjoint, so one product needs no exchange; a rank
that needs the whole y gathers the other ranks' rows. The Boolean and
tropical fixpoints exchange once per iteration: every rank gathers the new
vector (the next product reads all of x) and the ranks agree on whether
anything changed (an all-reduce of the changed flag).

``ShardedEngine`` is the GPU path: each rank builds the grammar of its own
row blocks, uploads it to its GPU and runs the library's products; the
fixpoints' update step (x = x OR y, or min) runs in the library too
(``gc_update``), and the exchanges go over the process group (NCCL). The loop
itself (``sharded_fixpoint``) takes the product and the update as callables,
so its exchange logic also runs with CPU stand-ins (gloo) in tests. Nothing
here computes any part of the product.
"""
from __future__ import annotations

import numpy as np


def row_shards(n: int, world: int, block_rows: int = 0) -> list[tuple[int, int]]:
    """Contiguous row ranges [r0, r1), one per rank, covering 0..n in order.

    With block_rows > 0 the cuts fall on block boundaries (a rank owns whole
    blocks; the blocks are dealt as evenly as their count allows); otherwise
    rows are dealt as evenly as possible. A rank may get an empty range when
    there are fewer blocks than ranks.
    """
    if world < 1 or n < 0:
        raise ValueError("world must be >= 1 and n >= 0")
    unit = block_rows if block_rows > 0 else 1
    units = -(-n // unit) if n else 0
    out = []
    for r in range(world):
        u0 = (units * r) // world
        u1 = (units * (r + 1)) // world
        out.append((min(n, u0 * unit), min(n, u1 * unit)))
    return out


def gather_rows(part, shards, group=None):
    """Concatenate every rank's rows (``part``: this rank's rows, a CPU or
    device torch tensor of shape (r1 - r0,) or (r1 - r0, k)) into the whole
    vector on every rank, in row order. Ranges may differ in length."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    longest = max(r1 - r0 for r0, r1 in shards)
    shape = (longest,) + tuple(part.shape[1:])
    padded = torch.zeros(shape, dtype=part.dtype, device=part.device)
    padded[: part.shape[0]] = part
    bufs = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(bufs, padded, group=group)
    return torch.cat([b[: r1 - r0] for b, (r0, r1) in zip(bufs, shards)])


def sharded_fixpoint(product, x0, shards, update, max_iter=1000, group=None):
    """x <- update(x, M x) to the fixpoint, M's rows sharded over the ranks.

    ``product(x)`` returns this rank's rows of M x for the whole vector x;
    ``update(old_rows, new_rows)`` returns (rows, changed) -- OR for
    reachability, min for shortest paths -- with changed a bool or a one-
    element int32 tensor on x's device (0 or 1). Each iteration gathers the
    rows of every rank and all-reduces the changed flag (MAX), so every rank
    stops at the same iteration. Returns (x, iterations) with iterations
    counting the products, the last of which changed nothing, or -1 if
    max_iter was reached first.
    """
    import torch
    import torch.distributed as dist

    rank = dist.get_rank(group)
    r0, r1 = shards[rank]
    x = x0.clone()
    for it in range(1, max_iter + 1):
        rows, changed = update(x[r0:r1], product(x))
        if isinstance(changed, torch.Tensor):
            flag = changed.to(device=x.device, dtype=torch.int32).reshape(1)
        else:
            flag = torch.tensor([1 if changed else 0], dtype=torch.int32, device=x.device)
        dist.all_reduce(flag, op=dist.ReduceOp.MAX, group=group)
        x = gather_rows(rows, shards, group)
        if int(flag.item()) == 0:
            return x, it
    return x, -1


def library_update(policy: str, stream=None):
    """The fixpoint step of ``policy`` ("or" or "minplus") on a rank's rows,
    in the library (gc_update): old rows updated in place, changed flag left
    on the device."""
    from . import _capi

    def update(old, new):
        import torch
        changed = torch.empty(1, dtype=torch.int32, device=old.device)
        st = stream if stream is not None else torch.cuda.current_stream(old.device)
        _capi().gc_update(policy, old, new, old.numel(), changed, st)
        return old, changed
    return update


class ShardedEngine:
    """This rank's share of a row-sharded matrix on its GPU.

    ``rows_csr(r0, r1)`` returns the CSR (row_ptr from 0, col, val or None) of
    rows [r0, r1); each rank builds and uploads the grammar of its own rows
    (whole ``block_rows`` blocks when given). ``matvec`` returns the whole y
    on every rank (one all-gather); ``matvec_rows`` only this rank's rows
    (no exchange). ``reach`` / ``sssp`` run the fixpoints with one all-gather
    and one all-reduce per iteration. Requires an initialised process group
    whose backend handles device tensors (NCCL).
    """

    def __init__(self, n, m, rows_csr, policy="f32", k_max=1, block_rows=0, group=None, device=None,
                 balance=False, threads=0):
        import torch
        import torch.distributed as dist
        from . import Engine, Grammar

        self.n, self.m, self.policy, self.group = n, m, policy, group
        self.shards = row_shards(n, dist.get_world_size(group), block_rows)
        self.r0, self.r1 = self.shards[dist.get_rank(group)]
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.engine = None
        if self.r1 > self.r0:
            rp, col, val = rows_csr(self.r0, self.r1)
            g = Grammar(self.r1 - self.r0, m, rp, col, val, block_rows=block_rows, threads=threads)
            if balance:
                g = g.balanced()
            self.engine = Engine(g, policy, k_max, device=self.device)

    def matvec_rows(self, x, stream=None):
        """This rank's rows of M x (x: the whole vector on this rank's device)."""
        import torch
        if self.engine is None:
            shape = (0,) if x.dim() == 1 else (0, x.shape[1])
            return torch.empty(shape, dtype=x.dtype, device=x.device)
        return self.engine.matvec(x, stream=stream)

    def matvec(self, x, stream=None):
        """The whole M x on every rank."""
        return gather_rows(self.matvec_rows(x, stream), self.shards, self.group)

    def reach(self, x0, max_iter=1000):
        """Boolean fixpoint x <- x OR (M (x) x) over the ranks; (x, iterations)."""
        if self.policy != "or":
            raise ValueError("reach needs the 'or' policy")
        return sharded_fixpoint(self.matvec_rows, x0, self.shards, library_update("or"), max_iter, self.group)

    def sssp(self, x0, max_iter=1000):
        """Tropical fixpoint x <- min(x, M (x) x) over the ranks; (x, iterations)."""
        if self.policy != "minplus":
            raise ValueError("sssp needs the 'minplus' policy")
        return sharded_fixpoint(self.matvec_rows, x0, self.shards, library_update("minplus"), max_iter,
                                self.group)


def local_rows(row_ptr, col, val, r0, r1):
    """The CSR of rows [r0, r1) of a matrix (offsets rebased to 0), for
    building one rank's grammar."""
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    s, e = int(row_ptr[r0]), int(row_ptr[r1])
    rp = row_ptr[r0 : r1 + 1] - s
    return rp, np.asarray(col[s:e]), (None if val is None else np.asarray(val[s:e]))
