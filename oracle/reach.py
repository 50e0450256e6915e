"""Boolean-semiring reachability and tropical shortest paths (Sec. 5 "Beyond
(+,x)"), in both directions: with right products (towards the sources) and
with left products (away from them).

One (OR, AND) product expands a BFS frontier by one step; the pages measure a
single pass and name the iteration to the fixpoint as the next step
(Sec. 5, Sec. 7 item 4). Reading taken here: with y[i] = OR over out-edges
i -> j of x[j], iterating x <- x OR y from a frontier with bit b set at source
s_b reaches the fixpoint in which bit b of x[i] is set exactly when i can
reach s_b (reflexively).

The tropical semiring (min, +) gives single-source shortest paths the same
way (Sec. 5: a pass is one Bellman-Ford edge relaxation): iterating
x <- min(x, M (x) x) from x0 (0 at the sources, +inf elsewhere) reaches the
fixpoint x[i] = min over sources s of (length of a shortest path i -> s along
out-edges, M[i][j] the length of edge i -> j) + x0[s], when no cycle has
negative length.
"""
from __future__ import annotations

from collections import deque

import numpy as np

from .direct import left_matvec_minplus, left_matvec_or, matvec_minplus, matvec_or


def fixpoint(row_ptr, col, x0, max_iter=1000):
    """Iterate x <- x | (M (x) x) until it stops changing.

    Returns (x, iterations), where iterations counts the products computed,
    the last of which changed nothing. Raises if max_iter is reached first.
    """
    x = np.asarray(x0, dtype=np.uint64).copy()
    for it in range(1, max_iter + 1):
        nxt = x | matvec_or(row_ptr, col, x)
        if np.array_equal(nxt, x):
            return x, it
        x = nxt
    raise RuntimeError("fixpoint not reached")


def sssp_fixpoint(row_ptr, col, val, x0, max_iter=1000):
    """Iterate x <- min(x, M (x) x) in float32 until it stops changing.

    Returns (x, iterations), iterations counting the products computed, the
    last of which changed nothing. Raises if max_iter is reached first.
    """
    x = np.asarray(x0, dtype=np.float32).copy()
    for it in range(1, max_iter + 1):
        nxt = np.minimum(x, matvec_minplus(row_ptr, col, val, x))
        if np.array_equal(nxt, x):
            return x, it
        x = nxt
    raise RuntimeError("fixpoint not reached")


def forward_fixpoint(row_ptr, col, x0, max_iter=1000):
    """The forward direction with left products: x <- x | (M^T (x) x), i.e.
    x[j] gains the sets of every i with an edge i -> j, until nothing changes.
    Bit b of the fixpoint at j is set iff s_b reaches j (reflexively).
    Returns (x, iterations) as fixpoint() does."""
    x = np.asarray(x0, dtype=np.uint64).copy()
    n = len(x)
    for it in range(1, max_iter + 1):
        nxt = x | left_matvec_or(row_ptr, col, x, n)
        if np.array_equal(nxt, x):
            return x, it
        x = nxt
    raise RuntimeError("fixpoint not reached")


def forward_sssp_fixpoint(row_ptr, col, val, x0, max_iter=1000):
    """Forward shortest paths with left products: x <- min(x, M^T (x) x), so
    x[j] = min over edges i -> j of x[i] + M[i][j] at the fixpoint: the
    distance from the nearest source (x0 = 0 there, +inf elsewhere) along
    out-edges, float32 as sssp_fixpoint."""
    x = np.asarray(x0, dtype=np.float32).copy()
    n = len(x)
    for it in range(1, max_iter + 1):
        nxt = np.minimum(x, left_matvec_minplus(row_ptr, col, val, x, n))
        if np.array_equal(nxt, x):
            return x, it
        x = nxt
    raise RuntimeError("fixpoint not reached")


def reach_bfs(row_ptr, col, n, srcs):
    """Textbook BFS on the reversed graph from every source: bit b of the
    result at node i is set iff i reaches srcs[b] along out-edges."""
    indeg_lists = [[] for _ in range(n)]
    for i in range(n):
        for e in range(int(row_ptr[i]), int(row_ptr[i + 1])):
            indeg_lists[int(col[e])].append(i)
    out = np.zeros(n, dtype=np.uint64)
    for b, s in enumerate(srcs):
        seen = np.zeros(n, dtype=bool)
        seen[s] = True
        q = deque([int(s)])
        while q:
            v = q.popleft()
            for u in indeg_lists[v]:
                if not seen[u]:
                    seen[u] = True
                    q.append(u)
        out[seen] |= np.uint64(1) << np.uint64(b)
    return out
