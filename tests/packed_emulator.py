"""CPU emulator of the packed, level-major grammar (a debugging aid for the
packing, not the oracle): it reads exactly the arrays the device reads and
evaluates them the way the kernels do -- T[0] identity, T[p+1] leaf values,
one buffer per level read through signed child references, roots captured
into RV, then the row sums over C -- in float64 (or int64 / uint64 OR /
float32 min-plus).
"""
import numpy as np


def emulate(ex, x, mode="f64"):
    """ex: dict of exported arrays (values, term_col, term_vidx, nodes, lvl_off,
    lvl_roots, root_off, c_off, c_ref). x: (m,) or (m, k)."""
    if mode == "or":
        x = np.asarray(x, dtype=np.uint64)
        leaf = x[ex["term_col"]]
        ident = np.uint64(0)
        comb = np.bitwise_or
        dt = np.uint64
    elif mode == "minplus":
        dt = np.float32
        x = np.asarray(x, dtype=dt)
        v = ex["values"].astype(dt)[ex["term_vidx"]]
        xs = x[ex["term_col"]]
        leaf = (v[:, None] + xs) if x.ndim == 2 else v + xs
        ident = dt(np.inf)
        comb = np.minimum
    else:
        dt = np.int64 if mode == "i64" else np.float64
        x = np.asarray(x, dtype=dt)
        v = ex["values"].astype(dt)[ex["term_vidx"]]
        xs = x[ex["term_col"]]
        leaf = (v[:, None] * xs) if x.ndim == 2 else v * xs
        ident = dt(0)
        comb = np.add
    kshape = x.shape[1:]
    T = np.zeros((len(leaf) + 1,) + kshape, dtype=dt)
    T[0] = ident
    T[1:] = leaf
    nodes = ex["nodes"].reshape(-1, 2)
    lvl_off = ex["lvl_off"]
    L = len(lvl_off) - 2
    RV = np.zeros((int(ex["lvl_roots"].sum()),) + kshape, dtype=dt)
    prev = np.zeros((0,) + kshape, dtype=dt)

    def cv(c, prev):
        c = c.astype(np.int64)
        out = np.empty((len(c),) + kshape, dtype=dt)
        pos = c >= 0
        out[pos] = prev[c[pos]]
        out[~pos] = T[-c[~pos] - 1]
        return out

    for k in range(1, L + 1):
        nk = nodes[lvl_off[k]:lvl_off[k + 1]]
        cur = comb(cv(nk[:, 0], prev), cv(nk[:, 1], prev))
        r = int(ex["lvl_roots"][k])
        RV[ex["root_off"][k]:ex["root_off"][k] + r] = cur[:r]
        prev = cur
    c_off, c_ref = ex["c_off"], ex["c_ref"]
    n = len(c_off) - 1
    y = np.zeros((n,) + kshape, dtype=dt)
    vals = cv(c_ref, RV) if len(c_ref) else np.zeros((0,) + kshape, dtype=dt)
    for r in range(n):
        acc = np.full(kshape, ident, dtype=dt) if kshape else ident
        for q in range(int(c_off[r]), int(c_off[r + 1])):
            acc = comb(acc, vals[q])
        y[r] = acc
    return y
