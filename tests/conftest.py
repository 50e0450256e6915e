import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300); run with -m gpu")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of host time")


@pytest.fixture(scope="session")
def worked():
    """The pages' running example, converted to 0-based indices.

    Returns dict with M (8x7 float64), V, S rows (list of (l, j)), the
    grammar in the oracle's symbol encoding (R, C, term_l, term_j), the
    printed level sets, x and the expected y.
    """
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    M = np.array(g["M"]["rows"], dtype=np.float64)
    V = np.array(g["V"]["values"], dtype=np.float64)
    S = {}
    for r, pairs in g["S"]["distinct_rows"].items():
        S[int(r) - 1] = [(l - 1, j - 1) for l, j in pairs]
    for r, src in g["S"]["repeats"].items():
        S[int(r) - 1] = S[int(src) - 1]
    S_rows = [S[i] for i in range(M.shape[0])]
    # terminal table: every distinct <l, j> in the rules, sorted by (j, l)
    terms = set()
    for rhs in g["R"]["rules"].values():
        for c in rhs:
            if not isinstance(c, str):
                terms.add((c[0] - 1, c[1] - 1))
    terms = sorted(terms, key=lambda p: (p[1], p[0]))
    tindex = {p: t for t, p in enumerate(terms)}
    names = [f"N{i}" for i in range(1, len(g["R"]["rules"]) + 1)]

    def sym(c):
        if isinstance(c, str):
            return int(c[1:]) - 1
        return -(tindex[(c[0] - 1, c[1] - 1)] + 1)

    R = np.array([[sym(c) for c in g["R"]["rules"][nm]] for nm in names], dtype=np.int64)
    C = [[sym(s)] for s in g["C"]["rows"]]
    x = np.array(g["product"]["x"], dtype=np.float64)
    rv = g["product"]["root_values"]
    y = np.array([rv[s] for s in g["C"]["rows"]], dtype=np.float64)
    return dict(raw=g, M=M, V=V, S=S_rows, x=x, y=y,
                grammar=dict(R=R, C=C, term_l=np.array([p[0] for p in terms]),
                             term_j=np.array([p[1] for p in terms])),
                level_sets=[[int(nm[1:]) - 1 for nm in s] for s in g["levels"]["sets"]],
                names=names)


def dense_to_csr(M, dtype=np.float32):
    """CSR (int64 row_ptr, int32 col, values as ``dtype``) of a dense matrix."""
    M = np.asarray(M)
    row_ptr = np.zeros(M.shape[0] + 1, dtype=np.int64)
    np.cumsum((M != 0).sum(1), out=row_ptr[1:])
    r, c = np.nonzero(M)
    return row_ptr, c.astype(np.int32), M[r, c].astype(dtype)


@pytest.fixture(scope="session")
def gcs():
    """The product package with its library built (compiles on first use)."""
    from grammar_compressed_sparse_gb300 import build
    build.build()
    import grammar_compressed_sparse_gb300 as pkg
    return pkg


def export_all(G):
    names = ["values", "term_col", "term_vidx", "rules", "c_off", "c_sym", "rule_level", "lvl_off",
             "nodes", "lvl_roots", "root_off", "c_ref", "node_id"]
    return {a: G.export(a) for a in names}


def oracle_grammar(ex):
    """The builder's raw SLP in the oracle's representation."""
    R = ex["rules"].reshape(-1, 2).astype(np.int64)
    c_off = ex["c_off"]
    C = [ex["c_sym"][c_off[r]:c_off[r + 1]].astype(np.int64).tolist() for r in range(len(c_off) - 1)]
    return dict(R=R, C=C, term_l=ex["term_vidx"].astype(np.int64), term_j=ex["term_col"].astype(np.int64))
