"""Row-block sharding of the product over several ranks (host-side plumbing).

The right product shards by rows: blocks of rows are independent grammars
(the row-block build, Sec. 1 "row blocks" of the pages), x is replicated and
each rank's rows of y are disjoint, so one product needs no exchange; a rank
that needs the whole y gathers the other ranks' rows. The Boolean and
tropical fixpoints exchange once per iteration: every rank gathers the new
vector (the next product reads all of x) and the ranks agree on whether
anything changed (an all-reduce of the changed flag).

The product itself is a callable, so the same logic runs with an Engine on a
GPU (NCCL) and with a CPU stand-in in tests (gloo). Nothing here computes any
part of the product.
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
    ``update(old_rows, new_rows)`` returns (rows, changed: bool) -- OR for
    reachability, min for shortest paths. Each iteration gathers the rows of
    every rank and all-reduces the changed flag (MAX of 0/1), so every rank
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
        flag = torch.tensor([1 if changed else 0], dtype=torch.int32, device=x.device)
        dist.all_reduce(flag, op=dist.ReduceOp.MAX, group=group)
        x = gather_rows(rows, shards, group)
        if int(flag.item()) == 0:
            return x, it
    return x, -1


def or_update(old, new):
    """Reachability step on this rank's rows: old | new, and whether it changed."""
    out = old | new
    return out, bool((out != old).any())


def min_update(old, new):
    """Shortest-path step on this rank's rows: min(old, new), and whether it changed."""
    import torch
    out = torch.minimum(old, new)
    return out, bool((out != old).any())


def local_rows(row_ptr, col, val, r0, r1):
    """The CSR of rows [r0, r1) of a matrix (offsets rebased to 0), for
    building one rank's grammar."""
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    s, e = int(row_ptr[r0]), int(row_ptr[r1])
    rp = row_ptr[r0 : r1 + 1] - s
    return rp, np.asarray(col[s:e]), (None if val is None else np.asarray(val[s:e]))
