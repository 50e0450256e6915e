"""Grammar side of the oracle: CSRV, RePair, decompression, evaluation,
levels and pass-through completion, each written straight from the pages.

Symbol encoding used throughout this module (its own, independent of the
product library): a symbol s >= 0 is the nonterminal N_s (0-based rule
index); s < 0 is the terminal with index t = -s - 1 into a terminal table
(term_l[t], term_j[t]) = <l, j>, meaning value V[l] in column j, both 0-based.

Readings of the pages taken here (they print 1-based V[1..k] and columns):
  * indices are 0-based;
  * V holds the distinct non-zero values sorted ascending (as printed), compared
    by value; zeros are not stored;
  * within a row, pairs come in ascending column order (row-by-row scan);
  * RePair breaks ties between equally frequent pairs by first occurrence in
    the row-major scan; the pages leave the tie-break open, and any choice
    gives a valid grammar with the same product.
"""
from __future__ import annotations

from collections import Counter

import numpy as np


# ----------------------------------------------------------------------------
# CSRV (Sec. 2 "CSRV", Eqs. 2.1-2.2)
# ----------------------------------------------------------------------------
def csrv(row_ptr, col, val):
    """CSRV encoding: value dictionary V and the row strings of S.

    Returns (V, rows) where V is the ascending array of distinct non-zero
    values and rows[i] is the list of pairs (l, j) of row i in column order,
    with M[i][j] = V[l]. The row delimiter $ is implicit in the row split.
    """
    val = np.asarray(val, dtype=np.float64)
    nz = val != 0
    V = np.unique(val[nz])
    rows = []
    for i in range(len(row_ptr) - 1):
        s, e = int(row_ptr[i]), int(row_ptr[i + 1])
        pairs = []
        order = np.argsort(np.asarray(col[s:e]), kind="stable")
        for q in order:
            v = val[s + q]
            if v != 0:
                pairs.append((int(np.searchsorted(V, v)), int(col[s + q])))
        rows.append(pairs)
    return V, rows


def terminal_table(rows):
    """Distinct terminals <l, j> of S, sorted by (j, l); returns (term_l, term_j, index)."""
    terms = sorted({p for r in rows for p in r}, key=lambda p: (p[1], p[0]))
    index = {p: t for t, p in enumerate(terms)}
    return (np.array([p[0] for p in terms], dtype=np.int64),
            np.array([p[1] for p in terms], dtype=np.int64), index)


# ----------------------------------------------------------------------------
# RePair (Sec. 2 "Grammar", Sec. 4.1) -- naive, for small inputs only
# ----------------------------------------------------------------------------
def repair(rows):
    """RePair with row boundaries.

    Repeatedly replaces the most frequent pair of adjacent symbols (never
    across a row delimiter) by a new nonterminal N_i -> A_i B_i, numbered in
    creation order (so children precede parents), and stops once no pair
    occurs more than once. Occurrences are counted and replaced left to right
    without overlap.

    Returns dict(term_l, term_j, R (|R| x 2 int64), C (list of symbol lists)).
    """
    term_l, term_j, index = terminal_table(rows)
    seqs = [[-(index[p] + 1) for p in r] for r in rows]
    R = []
    while True:
        counts = Counter()
        first_seen = {}
        order = 0
        for s in seqs:
            last_start = {}
            for i in range(len(s) - 1):
                p = (s[i], s[i + 1])
                if last_start.get(p, -2) == i - 1:   # overlapping occurrence (a a a)
                    continue
                last_start[p] = i
                counts[p] += 1
                if p not in first_seen:
                    first_seen[p] = order
                    order += 1
        if not counts:
            break
        best = max(counts.values())
        if best < 2:
            break
        pair = min((p for p, c in counts.items() if c == best), key=lambda p: first_seen[p])
        new = len(R)
        R.append(pair)
        for r, s in enumerate(seqs):
            out = []
            i = 0
            while i < len(s):
                if i + 1 < len(s) and (s[i], s[i + 1]) == pair:
                    out.append(new)
                    i += 2
                else:
                    out.append(s[i])
                    i += 1
            seqs[r] = out
    return dict(term_l=term_l, term_j=term_j,
                R=np.array(R, dtype=np.int64).reshape(-1, 2), C=seqs)


# ----------------------------------------------------------------------------
# Decompression and evaluation (Sec. 2, Lemmas 2.1-2.2, Theorem 2.3)
# ----------------------------------------------------------------------------
def expand(sym, R, term_l, term_j):
    """The terminal string a symbol derives: list of (l, j) pairs."""
    out = []
    stack = [int(sym)]
    while stack:
        s = stack.pop()
        if s < 0:
            t = -s - 1
            out.append((int(term_l[t]), int(term_j[t])))
        else:
            a, b = R[s]
            stack.append(int(b))
            stack.append(int(a))
    return out


def decompress(g):
    """Every row of C expanded back to its pair string (the rows of S)."""
    return [[p for s in row for p in expand(s, g["R"], g["term_l"], g["term_j"])] for row in g["C"]]


def eval_recursive(sym, R, term_l, term_j, V, x):
    """eval_x by the definition: V[l] * x[j] at a terminal, and
    eval(A) + eval(B) at N -> A B (Lemma 2.1). Exponential on deep DAGs with
    heavy sharing; tiny inputs only."""
    s = int(sym)
    if s < 0:
        t = -s - 1
        return float(V[term_l[t]]) * float(x[term_j[t]])
    a, b = R[s]
    return (eval_recursive(a, R, term_l, term_j, V, x)
            + eval_recursive(b, R, term_l, term_j, V, x))


def eval_w(g, V, x):
    """Theorem 2.3's CPU sweep in float64: W[i] = cv(A_i) + cv(B_i) in rule
    order, cv(N_j) = W[j], cv(<l,j>) = V[l] x[j]; then y[r] is the sum of cv
    over row r's symbols in C (Lemma 2.2; a row may hold several symbols and
    bare terminals). ``x`` is (m,) or (m, k)."""
    x = np.asarray(x, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    R, tl, tj = g["R"], g["term_l"], g["term_j"]
    k_shape = () if x.ndim == 1 else (x.shape[1],)
    W = np.zeros((len(R),) + k_shape)

    def cv(s):
        return W[s] if s >= 0 else V[tl[-s - 1]] * x[tj[-s - 1]]

    for i in range(len(R)):
        W[i] = cv(int(R[i][0])) + cv(int(R[i][1]))
    y = np.zeros((len(g["C"]),) + k_shape)
    for r, row in enumerate(g["C"]):
        for s in row:
            y[r] = y[r] + cv(int(s))
    return y


def eval_w_minplus(g, V, x):
    """Theorem 2.3's sweep over the tropical semiring (Sec. 5: the schedule
    needs only an associative combine): W[i] = min(cv(A_i), cv(B_i)) in rule
    order, cv(N_j) = W[j], cv(<l,j>) = V[l] + x[j] rounded to float32; then
    y[r] is the min of cv over row r's symbols in C, +inf for an empty row.
    ``x`` is (m,) or (m, k)."""
    x = np.asarray(x, dtype=np.float32)
    V = np.asarray(V, dtype=np.float32)
    R, tl, tj = g["R"], g["term_l"], g["term_j"]
    k_shape = () if x.ndim == 1 else (x.shape[1],)
    W = np.full((len(R),) + k_shape, np.inf, dtype=np.float32)

    def cv(s):
        return W[s] if s >= 0 else V[tl[-s - 1]] + x[tj[-s - 1]]

    for i in range(len(R)):
        W[i] = np.minimum(cv(int(R[i][0])), cv(int(R[i][1])))
    y = np.full((len(g["C"]),) + k_shape, np.inf, dtype=np.float32)
    for r, row in enumerate(g["C"]):
        for s in row:
            y[r] = np.minimum(y[r], cv(int(s)))
    return y


def eval_left(g, V, y, m):
    """The left product x = M^T y from the grammar, top-down, in float64: a
    symbol's weight is the sum of y over its occurrences in the rows'
    expansions. Row r gives each symbol of its C row the weight y[r]; rules
    are visited in reverse creation order (every parent before its
    children, since a rule only names earlier rules), and N_i -> A B adds
    N_i's weight to A and to B; a terminal <l, j> then adds V[l] times its
    weight to x[j]. The reverse reading of Lemmas 2.1-2.2."""
    y = np.asarray(y, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    R, tl, tj = g["R"], g["term_l"], g["term_j"]
    wr = np.zeros(len(R))
    wt = np.zeros(len(tl))
    for r, row in enumerate(g["C"]):
        for s in row:
            s = int(s)
            if s >= 0:
                wr[s] += y[r]
            else:
                wt[-s - 1] += y[r]
    for i in range(len(R) - 1, -1, -1):
        for c in R[i]:
            c = int(c)
            if c >= 0:
                wr[c] += wr[i]
            else:
                wt[-c - 1] += wr[i]
    x = np.zeros(m)
    for t in range(len(tl)):
        x[tj[t]] += V[tl[t]] * wt[t]
    return x


# ----------------------------------------------------------------------------
# Levels (Sec. 3, Eq. 3.1) and pass-through completion (Sec. 4.2)
# ----------------------------------------------------------------------------
def levels(R):
    """Eq. 3.1: lvl(terminal) = 0, lvl(N_i) = 1 + max(lvl A_i, lvl B_i).
    Computed in rule order, which is topological. Returns int64 array."""
    lvl = np.zeros(len(R), dtype=np.int64)
    for i in range(len(R)):
        a, b = int(R[i][0]), int(R[i][1])
        la = lvl[a] if a >= 0 else 0
        lb = lvl[b] if b >= 0 else 0
        lvl[i] = 1 + max(la, lb)
    return lvl


def max_parent_level(R, lvl):
    """For every nonterminal, the highest level of a rule that has it as a
    child (0 when it has no parent)."""
    mp = np.zeros(len(R), dtype=np.int64)
    for i in range(len(R)):
        for c in R[i]:
            c = int(c)
            if c >= 0:
                mp[c] = max(mp[c], lvl[i])
    return mp


def live_widths(R, lvl):
    """Per-level live set, the quantity the completed widths must equal
    (Sec. 4.2: a pass-through crossing level k is a value alive but not yet
    consumed there). w_k counts the nonterminals at level k plus those below k
    whose highest parent sits above k. Returns w[1..L] as a list."""
    L = int(lvl.max()) if len(lvl) else 0
    mp = max_parent_level(R, lvl)
    w = []
    for k in range(1, L + 1):
        at = int(np.sum(lvl == k))
        carried = int(np.sum((lvl < k) & (mp > k)))
        w.append(at + carried)
    return w


def pass_through_count(R, lvl):
    """Nodes completion must add: sum over nonterminals u of
    max(0, maxpar(u) - lvl(u) - 1), one shared chain per skipping node."""
    mp = max_parent_level(R, lvl)
    return int(np.sum(np.maximum(0, mp - lvl - 1)))


def complete(R, lvl):
    """Pass-through completion (Sec. 4.2, Fig. 3.1).

    For a nonterminal u whose highest parent is d > 1 levels above it, insert
    the chain u = u_0, u_1, ..., u_{d-1} of identity nodes u_i -> u_{i-1}, at
    levels lvl(u)+1 ... maxpar(u)-1. One chain per node, shared by all its
    skipping parents (the reading under which widths equal live sets); a
    parent at level K reads u itself if lvl(u) = K-1, else the chain element
    at level K-1. Terminal children are left alone (Def. 3.2).

    Returns a list ``layers`` with layers[k-1] = list of (key, children) for
    level k, where key is ('n', i) for rule N_i or ('p', u, k) for the pass-
    through of u at level k, and children are references: ('t', t) terminal,
    ('n', i) / ('p', u, k-1) node of level k-1.
    """
    L = int(lvl.max()) if len(lvl) else 0
    mp = max_parent_level(R, lvl)
    layers = [[] for _ in range(L)]

    def ref(c, K):
        c = int(c)
        if c < 0:
            return ('t', -c - 1)
        return ('n', c) if lvl[c] == K - 1 else ('p', c, K - 1)

    for i in range(len(R)):
        K = int(lvl[i])
        layers[K - 1].append((('n', i), (ref(R[i][0], K), ref(R[i][1], K))))
    for u in range(len(R)):
        for k in range(int(lvl[u]) + 1, int(mp[u])):
            below = ('n', u) if k - 1 == lvl[u] else ('p', u, k - 1)
            layers[k - 1].append((('p', u, k), (below,)))
    return layers


def is_properly_layered(layers):
    """Def. 3.2: every nonterminal child of a level-k node sits at level k-1."""
    prev = set()
    for k, layer in enumerate(layers, start=1):
        for _, ch in layer:
            for c in ch:
                if c[0] != 't' and c not in prev:
                    return False
        prev = {key for key, _ in layer}
    return True


def eval_layered(layers, g, V, x):
    """The level-synchronous sweep on a completed grammar (Lemma 3.3, Sec. 4.3),
    in float64: level k reads only level k-1 (prev) and the terminals,
    pass-throughs copy their child, roots (symbols of C) are recorded the
    moment their level is done; then y[r] sums row r's symbols."""
    x = np.asarray(x, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    tl, tj = g["term_l"], g["term_j"]
    roots = {int(s) for row in g["C"] for s in row if s >= 0}
    rv = {}
    prev = {}

    def cv(c):
        return V[tl[c[1]]] * x[tj[c[1]]] if c[0] == 't' else prev[c]

    for layer in layers:
        cur = {}
        for key, ch in layer:
            v = cv(ch[0])
            for c in ch[1:]:
                v = v + cv(c)
            cur[key] = v
            if key[0] == 'n' and key[1] in roots:
                rv[key[1]] = v
        prev = cur
    k_shape = () if x.ndim == 1 else (x.shape[1],)
    y = np.zeros((len(g["C"]),) + k_shape)
    for r, row in enumerate(g["C"]):
        for s in row:
            s = int(s)
            y[r] = y[r] + (rv[s] if s >= 0 else V[tl[-s - 1]] * x[tj[-s - 1]])
    return y
