"""Host builder (CSRV, RePair, levels, completion, packing) checked against
the oracle on the CPU, through the C ABI. No GPU needed."""
import os
import re

import numpy as np
import pytest

import gcsynth
from conftest import ROOT, dense_to_csr, export_all, oracle_grammar
from oracle import direct, grammar
from packed_emulator import emulate


def _cases():
    for seed in range(6):
        n = 4 + seed * 3
        m = 5 + seed * 4
        rp, c, v, dense = gcsynth.random_sparse(n, m, 0.5, [1.0, 2.0, -0.5, 3.25], seed)
        yield f"rand{seed}", rp, c, v
    for seed, (n, m, F) in enumerate([(30, 200, 3), (64, 500, 5), (200, 300, 8)]):
        d = gcsynth.genotype_dense(n=n, m=m, founders=F, switch=0.02, mutation=0.005, seed=seed)
        rp, c, v = gcsynth.dense_to_csr(d)
        yield f"geno{n}x{m}", rp, c, v


CASES = list(_cases())


def check_grammar(G, rp, c, v, n, m, block_rows=0, repair_end_state=True):
    ex = export_all(G)
    st = G.stats()
    og = oracle_grammar(ex)
    V, rows = grammar.csrv(rp, c, v)
    # CSRV: same dictionary; terminal table is the sorted set of used <l, j>
    np.testing.assert_array_equal(ex["values"].astype(np.float64), V.astype(np.float32).astype(np.float64))
    # O3: decompression reproduces S
    assert grammar.decompress(og) == rows
    # RePair end state: no pair of adjacent symbols repeats in C, topological numbering
    # (per row block when blocks are compressed separately)
    seen = {}
    for r, row in enumerate(og["C"]):
        blk = r // block_rows if block_rows else 0
        for i in range(len(row) - 1):
            key = (blk, row[i], row[i + 1])
            seen[key] = seen.get(key, 0) + 1
    assert all(cnt < 2 for cnt in seen.values()) or not repair_end_state
    for i, (a, b) in enumerate(og["R"]):
        assert (a < 0 or a < i) and (b < 0 or b < i)
    # O4: Eq. 3.1 levels, live-set widths, pass-through count
    lvl = grammar.levels(og["R"])
    np.testing.assert_array_equal(ex["rule_level"], lvl)
    assert st["depth"] == (int(lvl.max()) if len(lvl) else 0)
    np.testing.assert_array_equal(G.widths(), grammar.live_widths(og["R"], lvl))
    assert st["n_pass"] == grammar.pass_through_count(og["R"], lvl)
    assert st["n_nodes"] == st["n_rules"] + st["n_pass"]
    # packed nodes are the oracle's completed grammar, level by level
    layers = grammar.complete(og["R"], lvl)
    node_id = ex["node_id"]
    lo = ex["lvl_off"]
    nodes = ex["nodes"].reshape(-1, 2)
    roots = {s for row in og["C"] for s in row if s >= 0}
    for k in range(1, st["depth"] + 1):
        ids = node_id[lo[k]:lo[k + 1]]
        want = sorted([key[1] if key[0] == 'n' else -(key[1] + 1) for key, _ in layers[k - 1]])
        assert sorted(ids.tolist()) == want
        nr = int(ex["lvl_roots"][k])
        assert all(i >= 0 and i in roots for i in ids[:nr])
        assert not any(i >= 0 and i in roots for i in ids[nr:])
        prev_ids = node_id[lo[k - 1]:lo[k]] if k > 1 else np.zeros(0, np.int32)
        for q, i in enumerate(ids):
            a, b = nodes[lo[k] + q]
            kids = [int(og["R"][i][0]), int(og["R"][i][1])] if i >= 0 else [-i - 1]
            refs = [a, b] if i >= 0 else [a]
            if i < 0:
                assert b == -1
            for kid, ref in zip(kids, refs):
                if kid < 0:
                    assert ref == kid - 1           # terminal t -> T[t+1]
                else:
                    assert ref >= 0
                    assert prev_ids[ref] in (kid, -(kid + 1))
    # values: packed emulator and W-array sweep against the direct product
    x = np.random.default_rng(1).standard_normal(m)
    y_ref, b = direct.matvec_f64(rp, c, v, x)
    np.testing.assert_allclose(grammar.eval_w(og, ex["values"], x), y_ref, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(emulate(ex, x), y_ref, rtol=1e-9, atol=1e-9)
    X = np.random.default_rng(2).standard_normal((m, 3))
    np.testing.assert_allclose(emulate(ex, X), direct.matvec_f64(rp, c, v, X)[0], rtol=1e-9, atol=1e-9)
    return ex


def test_library_exports_every_header_symbol(gcs):
    text = open(os.path.join(ROOT, "include", "gcsparse.h")).read()
    declared = set(re.findall(r"^\s*(?:gc_status|void|const char\*)\s+(gc_\w+)\s*\(", text, re.M))
    assert declared, "no declarations parsed"
    import ctypes
    lib = ctypes.CDLL(gcs.capi._build.LIB)
    for name in sorted(declared):
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert declared == set(gcs.capi.EXPORTED)


def test_worked_example_builds(gcs, worked):
    rp, c, v = dense_to_csr(worked["M"], np.float32)
    G = gcs.Grammar(8, 7, rp, c, v)
    ex = check_grammar(G, rp, c, v, 8, 7)
    y = emulate(ex, worked["x"])
    np.testing.assert_allclose(y, worked["y"], rtol=1e-6)
    st = G.stats()
    assert st["n_values"] == 4 and st["n_terminals"] == 12


@pytest.mark.parametrize("name,rp,c,v", CASES, ids=[cs[0] for cs in CASES])
def test_builder_matches_oracle(gcs, name, rp, c, v):
    n, m = len(rp) - 1, int(c.max()) + 3
    G = gcs.Grammar(n, m, rp, c, v)
    check_grammar(G, rp, c, v, n, m)


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("block_rows", [0, 7, 64])
def test_blocks_and_orders(gcs, order, block_rows):
    d = gcsynth.genotype_dense(n=150, m=400, founders=6, switch=0.01, mutation=0.005, seed=11)
    rp, c, v = gcsynth.dense_to_csr(d)
    G = gcs.Grammar(150, 400, rp, c, v, block_rows=block_rows, order=order)
    ex = check_grammar(G, rp, c, v, 150, 400, block_rows)
    st = G.stats()
    assert st["n_blocks"] == (1 if block_rows == 0 else -(-150 // block_rows))
    if block_rows:
        # no rule is shared across blocks: each block's rows use its own rules
        og = oracle_grammar(ex)
        owner = {}
        for r, row in enumerate(og["C"]):
            blk = r // block_rows
            stack = [s for s in row if s >= 0]
            while stack:
                s = stack.pop()
                assert owner.setdefault(s, blk) == blk
                stack.extend(int(z) for z in og["R"][s] if z >= 0)


def test_integer_and_boolean_values(gcs):
    # graph-like 0/1 matrix, built with val = NULL (every entry 1)
    rp, col = gcsynth.copy_model_graph(nodes=300, n0=10, d0=12, p_edit=0.1, seed=5)
    G = gcs.Grammar(300, 300, rp, col, None)
    ex = export_all(G)
    assert ex["values"].tolist() == [1.0]
    x = np.random.default_rng(0).integers(0, 2**63, 300, dtype=np.uint64)
    np.testing.assert_array_equal(emulate(ex, x, "or"), direct.matvec_or(rp, col, x))
    xi = np.random.default_rng(1).integers(-1000, 1000, 300)
    np.testing.assert_array_equal(emulate(ex, xi, "i64"),
                                  direct.matvec_i64(rp, col, np.ones(len(col)), xi))
    xf = np.random.default_rng(2).standard_normal(300).astype(np.float32)
    assert np.array_equal(emulate(ex, xf, "minplus"), direct.matvec_minplus(rp, col, np.ones(len(col)), xf))
    for pol in ("f32", "i64", "or", "minplus"):
        lay = G.layout(pol, 1)
        assert lay["arena_bytes"] >= lay["grammar_bytes"] + lay["scratch_bytes"]
    with pytest.raises(gcs.GcError):
        G.layout("f32", 3)
    # the float32 sum takes the batch widths 1, 4, 8, ..., 256; the buffers
    # grow with the width, the grammar does not
    lays = {k: G.layout("f32", k) for k in (1, 4, 8, 16, 32, 64, 128, 256)}
    assert len({lay["grammar_bytes"] for k, lay in lays.items() if k > 1}) == 1
    assert lays[256]["scratch_bytes"] > lays[64]["scratch_bytes"] > lays[16]["scratch_bytes"]
    for bad in (2, 12, 512):
        with pytest.raises(gcs.GcError):
            G.layout("f32", bad)
    for bad in (4, 64):
        with pytest.raises(gcs.GcError):
            G.layout("minplus", bad)


def test_minplus_packed_layout_matches_oracle(gcs):
    # the tropical policy reads the same packed arrays; min is exact, so the
    # packed evaluation equals the direct product bit for bit, k = 1 and 16
    d = gcsynth.genotype_dense(n=120, m=300, founders=5, switch=0.01, mutation=0.005, seed=4)
    rp, c, v = gcsynth.dense_to_csr(d)
    G = gcs.Grammar(120, 300, rp, c, v)
    ex = export_all(G)
    g = np.random.default_rng(9)
    for x in (g.standard_normal(300).astype(np.float32), g.standard_normal((300, 16)).astype(np.float32)):
        assert np.array_equal(emulate(ex, x, "minplus"), direct.matvec_minplus(rp, c, v, x))
    for k_max in (1, 16):
        lay = G.layout("minplus", k_max)
        assert lay == G.layout("f32", k_max)     # same value width as the float32 sum
    with pytest.raises(gcs.GcError):
        G.layout("minplus", 4)


def test_policy_value_checks(gcs):
    rp, c, v, _ = gcsynth.random_sparse(10, 10, 0.5, [0.5, 2.0], 3)
    G = gcs.Grammar(10, 10, rp, c, v)
    with pytest.raises(gcs.GcError, match="UNSUPPORTED"):
        G.layout("i64", 1)
    with pytest.raises(gcs.GcError, match="UNSUPPORTED"):
        G.layout("or", 1)
    rp, c, v, _ = gcsynth.random_sparse(10, 10, 0.5, [1.0, 2.0], 3)
    G = gcs.Grammar(10, 10, rp, c, v)
    G.layout("i64", 1)
    with pytest.raises(gcs.GcError, match="UNSUPPORTED"):
        G.layout("or", 1)


@pytest.mark.parametrize("k_max", [1, 16, 256])
def test_device_plans_pass_host_checks(gcs, k_max):
    # gc_upload builds and checks every device array on the host (node codes,
    # level-emit chunks, references into the narrow top levels) before its
    # first CUDA call; without a GPU it must get that far and stop there
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    cfg = dict(gcsynth.GENO_MEDIUM, n=150, m=20000)
    slice_ = gcs.Grammar(150, 20000, *gcsynth.genotype_csr(**cfg))         # level emit, with a tail
    w = slice_.widths()
    assert slice_.stats()["c_len"] >= 128 * 150 and w[-1] <= 1024 and w[-2] <= 1024
    rp, c, v, _ = gcsynth.random_sparse(40, 3000, 0.4, [1.0, -1.0, 0.5], 8)
    heavy = gcs.Grammar(40, 3000, rp, c, v)                                 # level emit, few levels
    small = gcs.Grammar(1000, 2000, *gcsynth.genotype_csr(**gcsynth.GENO_SMALL))   # row emit
    for G in (slice_, heavy, small):
        for pol in ("f32", "minplus") if k_max <= 16 else ("f32",):
            lay = G.layout(pol, k_max)
            with pytest.raises(gcs.GcError, match="GC_ERR_CUDA"):
                gcs.capi.gc_upload(G._p, pol, k_max, 256, lay["arena_bytes"])
            if k_max == 1:   # the dataflow layout: block plan and its checks
                lay = G.layout(pol, 1, "dataflow")
                with pytest.raises(gcs.GcError, match="GC_ERR_CUDA"):
                    gcs.capi.gc_upload_ex(G._p, pol, 1, "dataflow", 256, lay["arena_bytes"])
            else:
                with pytest.raises(gcs.GcError, match="GC_ERR_UNSUPPORTED"):
                    G.layout(pol, k_max, "dataflow")


def test_dataflow_block_plan(gcs, tmp_path):
    # tests/native/flow_plan_check.cpp builds the dataflow sweep's block plan
    # (blocks, their dependencies, the final block) for 4- and 8-byte values,
    # runs the host checks gc_upload runs, and replays the blocks on the CPU
    # through their child references, against the direct product
    import struct
    import subprocess
    from grammar_compressed_sparse_gb300 import build as gbuild
    gbuild.build()
    objs = [os.path.join(gbuild.BUILD, f + ".o") for f in gbuild.HOST_SOURCES]
    exe = str(tmp_path / "flow_plan_check")
    subprocess.run(["g++", "-O2", "-std=c++17", "-fopenmp", "-I", gbuild.INCLUDE, "-I", gbuild.CSRC,
                    os.path.join(ROOT, "tests", "native", "flow_plan_check.cpp"), *objs, "-o", exe],
                   check=True, capture_output=True)
    files = []

    def dump(name, n, m, rp, c, v):
        path = str(tmp_path / name)
        with open(path, "wb") as f:
            f.write(struct.pack("qqq", n, m, int(rp[-1])))
            f.write(np.asarray(rp, np.int64).tobytes())
            f.write(np.asarray(c, np.int32).tobytes())
            f.write(np.asarray(v, np.float32).tobytes())
        files.append(path)

    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    dump("slice300.bin", 300, cfg["m"], *gcsynth.genotype_csr(**cfg))                  # many blocks a level
    dump("small.bin", 1000, 2000, *gcsynth.genotype_csr(**gcsynth.GENO_SMALL))
    rp, c, v, _ = gcsynth.random_sparse(40, 3000, 0.4, [1.0, -1.0, 0.5], 8)
    dump("heavy.bin", 40, 3000, rp, c, v)                                               # one final block
    rp, col = gcsynth.copy_model_graph(nodes=3000, n0=20, d0=15, p_edit=0.05, seed=1)
    dump("graph.bin", 3000, 3000, rp, col, np.ones(len(col), np.float32))
    d = np.zeros((9, 700), np.float32)
    d[:, ::3] = 1.0
    d[4, 1::3] = 2.0
    dump("dense.bin", 9, 700, *dense_to_csr(d, np.float32))
    dump("one.bin", 1, 1, *dense_to_csr(np.full((1, 1), 3.0, np.float32), np.float32))   # no rules
    out = subprocess.run([exe, *files], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith("OK")
    # the 300-row slice has regular blocks below its final block
    first = [ln for ln in out.stdout.splitlines() if ln.startswith("flow vb=4")][0]
    assert "(final from level 1)" not in first and int(first.split(" blocks ")[1].split()[0]) > 100


def test_slice_plan_and_tile_reduction(gcs, tmp_path):
    # tests/native/slice_plan_check.cpp rebuilds the slice emit's plan for each
    # matrix and replays the device's tile reduction on the CPU (lane runs and
    # the segmented lane scan), against direct row sums over random values
    import struct
    import subprocess
    from grammar_compressed_sparse_gb300 import build as gbuild
    gbuild.build()
    objs = [os.path.join(gbuild.BUILD, f + ".o") for f in gbuild.HOST_SOURCES]
    exe = str(tmp_path / "slice_plan_check")
    subprocess.run(["g++", "-O2", "-std=c++17", "-fopenmp", "-I", gbuild.INCLUDE, "-I", gbuild.CSRC,
                    os.path.join(ROOT, "tests", "native", "slice_plan_check.cpp"), *objs, "-o", exe],
                   check=True, capture_output=True)
    files = []

    def dump(name, n, m, rp, c, v):
        path = str(tmp_path / name)
        with open(path, "wb") as f:
            f.write(struct.pack("qqq", n, m, int(rp[-1])))
            f.write(np.asarray(rp, np.int64).tobytes())
            f.write(np.asarray(c, np.int32).tobytes())
            f.write(np.asarray(v, np.float32).tobytes())
        files.append(path)

    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    dump("slice300.bin", 300, cfg["m"], *gcsynth.genotype_csr(**cfg))                  # long segments
    dump("small.bin", 1000, 2000, *gcsynth.genotype_csr(**gcsynth.GENO_SMALL))         # one or two slices
    rp, c, v, _ = gcsynth.random_sparse(40, 3000, 0.4, [1.0, -1.0, 0.5], 8)
    dump("heavy.bin", 40, 3000, rp, c, v)                                               # bare terminals
    d = np.zeros((9, 700), np.float32)
    d[:, ::3] = 1.0
    d[4, 1::3] = 2.0                                                                     # one row much longer
    dump("dense.bin", 9, 700, *dense_to_csr(d, np.float32))
    out = subprocess.run([exe, *files], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith("OK")


@pytest.mark.parametrize("bad", ["row_ptr", "col_range", "dup", "nan", "inf"])
def test_bad_csr_is_rejected(gcs, bad):
    rp = np.array([0, 2, 3], dtype=np.int64)
    c = np.array([0, 2, 1], dtype=np.int32)
    v = np.array([1.0, 2.0, 3.0], dtype=np.float32)
    if bad == "row_ptr":
        rp = np.array([0, 3, 2], dtype=np.int64)
    elif bad == "col_range":
        c = np.array([0, 5, 1], dtype=np.int32)
    elif bad == "dup":
        c = np.array([1, 1, 1], dtype=np.int32)
    elif bad == "nan":
        v[1] = np.nan
    elif bad == "inf":
        v[1] = np.inf
    with pytest.raises(gcs.GcError, match="GC_ERR_ARG"):
        gcs.Grammar(2, 3, rp, c, v)


def test_zeros_unsorted_and_degenerate(gcs):
    # stored zeros are dropped; unsorted rows are ordered by column
    rp = np.array([0, 3, 3, 5], dtype=np.int64)
    c = np.array([2, 0, 1, 1, 0], dtype=np.int32)
    v = np.array([1.5, 0.0, -0.0, 1.5, 2.0], dtype=np.float32)
    G = gcs.Grammar(3, 3, rp, c, v)
    ex = export_all(G)
    x = np.array([1.0, 2.0, 4.0])
    dense = np.zeros((3, 3))
    for r in range(3):
        for q in range(rp[r], rp[r + 1]):
            dense[r, c[q]] = v[q]
    np.testing.assert_allclose(emulate(ex, x), dense @ x)
    # empty matrix, all-empty rows, a single non-zero, no repetition at all
    for n, m, rp, c, v in [
        (0, 0, np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32)),
        (4, 6, np.zeros(5, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32)),
        (3, 3, np.array([0, 0, 1, 1], np.int64), np.array([2], np.int32), np.array([5.0], np.float32)),
        (2, 4, np.array([0, 2, 4], np.int64), np.array([0, 1, 2, 3], np.int32),
         np.array([1, 2, 3, 4], np.float32)),
    ]:
        G = gcs.Grammar(n, m, rp, c, v)
        st = G.stats()
        assert st["n"] == n
        ex = export_all(G)
        x = np.arange(1, m + 1, dtype=np.float64)
        dense = np.zeros((n, m))
        for r in range(n):
            for q in range(rp[r], rp[r + 1]):
                dense[r, c[q]] = v[q]
        np.testing.assert_allclose(emulate(ex, x), dense @ x)
        assert G.layout("f32", 1)["arena_bytes"] > 0


def test_save_load_roundtrip(gcs, tmp_path):
    d = gcsynth.genotype_dense(n=40, m=120, founders=4, switch=0.02, mutation=0.01, seed=2)
    rp, c, v = gcsynth.dense_to_csr(d)
    G = gcs.Grammar(40, 120, rp, c, v)
    p = str(tmp_path / "g.bin")
    G.save(p)
    H = gcs.Grammar.load(p)
    a, b = export_all(G), export_all(H)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    assert G.stats()["n_nodes"] == H.stats()["n_nodes"]
    with open(p, "r+b") as f:
        f.truncate(100)
    with pytest.raises(gcs.GcError, match="GC_ERR_IO"):
        gcs.Grammar.load(p)
    with pytest.raises(gcs.GcError, match="GC_ERR_IO"):
        gcs.Grammar.load(str(tmp_path / "missing.bin"))


@pytest.mark.parametrize("workers", [1, 3])
def test_streaming_row_blocks_match_block_build(gcs, workers):
    d = gcsynth.genotype_dense(n=130, m=300, founders=5, switch=0.01, mutation=0.005, seed=21)
    rp, c, v = gcsynth.dense_to_csr(d)

    def make_block(r0, r1):
        return rp[r0:r1 + 1] - rp[r0], c[rp[r0]:rp[r1]], v[rp[r0]:rp[r1]]

    S = gcs.Grammar.from_row_blocks(130, 300, 32, make_block, workers=workers)
    B = gcs.Grammar(130, 300, rp, c, v, block_rows=32)
    a, b = export_all(S), export_all(B)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    st = S.stats()
    assert st["n_blocks"] == 5 and st["nnz"] == rp[-1]
    check_grammar(S, rp, c, v, 130, 300, 32)


def test_streaming_builder_rejects_gaps_and_overlaps(gcs):
    capi = gcs.capi
    rp = np.array([0, 1], dtype=np.int64)
    c = np.array([0], dtype=np.int32)
    v = np.array([1.0], dtype=np.float32)
    b = capi.gc_builder_create(3, 2)
    try:
        capi.gc_builder_add_rows(b, 0, rp, c, v)
        with pytest.raises(gcs.GcError, match="overlap"):
            capi.gc_builder_add_rows(b, 0, rp, c, v)
        with pytest.raises(gcs.GcError, match="cover"):
            capi.gc_builder_finish(b)
        with pytest.raises(gcs.GcError, match="outside"):
            capi.gc_builder_add_rows(b, 3, rp, c, v)
    finally:
        capi.gc_builder_free(b)


def test_left_plan_replays_to_the_transpose(gcs, tmp_path):
    # tests/native/left_plan_check.cpp builds the left product's plan, checks
    # it, and replays its warp tasks on the CPU exactly as left_step_kernel
    # runs them (float32 and float64) against a direct M^T y
    import struct
    import subprocess
    from grammar_compressed_sparse_gb300 import build as gbuild
    gbuild.build()
    objs = [os.path.join(gbuild.BUILD, f + ".o") for f in gbuild.HOST_SOURCES]
    exe = str(tmp_path / "left_plan_check")
    subprocess.run(["g++", "-O2", "-std=c++17", "-fopenmp", "-I", gbuild.INCLUDE, "-I", gbuild.CSRC,
                    os.path.join(ROOT, "tests", "native", "left_plan_check.cpp"), *objs, "-o", exe],
                   check=True, capture_output=True)
    files = []

    def dump(name, n, m, rp, c, v):
        path = str(tmp_path / name)
        with open(path, "wb") as f:
            f.write(struct.pack("qqq", n, m, int(rp[-1])))
            f.write(np.asarray(rp, np.int64).tobytes())
            f.write(np.asarray(c, np.int32).tobytes())
            f.write(np.asarray(v, np.float32).tobytes())
        files.append(path)

    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    dump("slice300.bin", 300, cfg["m"], *gcsynth.genotype_csr(**cfg))
    dump("small.bin", 1000, 2000, *gcsynth.genotype_csr(**gcsynth.GENO_SMALL))
    rp, c, v, _ = gcsynth.random_sparse(40, 3000, 0.4, [1.0, -1.0, 0.5], 8)
    dump("heavy.bin", 40, 3000, rp, c, v)
    rp, col = gcsynth.copy_model_graph(nodes=3000, n0=20, d0=15, p_edit=0.05, seed=1)
    dump("graph.bin", 3000, 3000, rp, col, gcsynth.target_lengths(col, 3000, seed=2))
    d = np.zeros((400, 50), np.float32)
    d[:, 7] = 1.0                         # one column in every row: long parent lists
    d[::2, 11] = 2.0
    dump("column.bin", 400, 50, *dense_to_csr(d, np.float32))
    dump("empty.bin", 4, 6, np.zeros(5, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32))
    dump("norules.bin", 2, 4, np.array([0, 2, 4], np.int64), np.array([0, 1, 2, 3], np.int32),
         np.array([1, 2, 3, 4], np.float32))
    out = subprocess.run([exe, *files], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith("OK")


def test_left_layout_sizes(gcs):
    d = gcsynth.genotype_dense(n=120, m=300, founders=5, switch=0.01, mutation=0.005, seed=4)
    G = gcs.Grammar(120, 300, *gcsynth.dense_to_csr(d))
    lay = gcs.capi.gc_left_layout(G._p, "f32")
    st = G.stats()
    # W holds one float per layered node; RS one per root slot and terminal
    assert lay["scratch_bytes"] >= 4 * (st["n_nodes"] + st["n_roots"] + 2 * st["n_terminals"])
    assert lay["arena_bytes"] == lay["grammar_bytes"] + lay["scratch_bytes"] and lay["staging_bytes"] == 0
    # 8-byte policies double the scratch; OR needs a 0/1 pattern
    lay8 = gcs.capi.gc_left_layout(G._p, "i64")
    assert lay8["scratch_bytes"] >= 2 * lay["scratch_bytes"] - 3 * 256
    assert gcs.capi.gc_left_layout(G._p, "minplus")["arena_bytes"] == lay["arena_bytes"]
    with pytest.raises(gcs.GcError, match="UNSUPPORTED"):
        gcs.capi.gc_left_layout(G._p, "or")


def test_corrupted_grammar_file_is_rejected(gcs, tmp_path):
    # a child reference pointed past its level below: gc_load's validation
    # must refuse the file (no device is ever handed such a grammar)
    d = gcsynth.genotype_dense(n=40, m=120, founders=4, switch=0.02, mutation=0.01, seed=2)
    rp, c, v = gcsynth.dense_to_csr(d)
    G = gcs.Grammar(40, 120, rp, c, v)
    ex = export_all(G)
    p = str(tmp_path / "g.bin")
    G.save(p)
    raw = bytearray(open(p, "rb").read())
    nodes = ex["nodes"].astype(np.int32)
    at = bytes(raw).find(nodes.tobytes())
    assert at >= 0 and ex["lvl_off"][-2] > ex["lvl_off"][2]     # found, and there is a level >= 2
    k2 = int(ex["lvl_off"][2])                                  # first node of level 2
    bad = nodes.copy()
    bad[2 * k2] = 1 << 30                                       # its first child: far outside level 1
    raw[at:at + len(nodes.tobytes())] = bad.tobytes()
    q = str(tmp_path / "bad.bin")
    open(q, "wb").write(bytes(raw))
    with pytest.raises(gcs.GcError, match="GC_ERR_INVALID_GRAMMAR"):
        gcs.Grammar.load(q)
    raw2 = bytearray(open(p, "rb").read())
    raw2[0] ^= 0xFF                                             # not the file's magic
    open(q, "wb").write(bytes(raw2))
    with pytest.raises(gcs.GcError, match="GC_ERR_IO"):
        gcs.Grammar.load(q)


def test_cpu_grammar_sweep_on_the_builders_grammar(gcs):
    # the CPU baseline's W-array sweep reads the library's exported raw
    # grammar: it must give the direct product
    from baselines.wsweep import GrammarSweep
    cfg = dict(gcsynth.GENO_MEDIUM, n=300)
    rp, c, v = gcsynth.genotype_csr(**cfg)
    G = gcs.Grammar(300, cfg["m"], rp, c, v)
    sw = GrammarSweep.from_grammar(G)
    x = gcsynth.beta(cfg["m"], seed=2).astype(np.float64)
    y_ref, b = direct.matvec_f64(rp, c, v, x)
    y = sw(x, 1)
    assert direct.within_tolerance(y, y_ref, b, 1e-12)[0]
    assert np.array_equal(sw(x, 4), y)


@pytest.mark.parametrize("name,rp,c,v", CASES, ids=[cs[0] for cs in CASES])
def test_balanced_grammar(gcs, name, rp, c, v):
    """Sec. 4.2 pre-balancing (an AVL grammar): same decompression, same
    products, children's heights within one of each other, and depth within
    the AVL bound 1.4405 log2(len + 2) of the longest expansion."""
    n, m = len(rp) - 1, int(c.max()) + 3
    G = gcs.Grammar(n, m, rp, c, v)
    B = G.balanced()
    ex = check_grammar(B, rp, c, v, n, m, repair_end_state=False)
    og = oracle_grammar(ex)
    lvl = grammar.levels(og["R"])
    h = lambda s: 0 if s < 0 else int(lvl[s])
    assert all(abs(h(a) - h(b)) <= 1 for a, b in og["R"])
    lens = np.zeros(len(og["R"]), np.int64)
    for i, (a, b) in enumerate(og["R"]):
        lens[i] = (1 if a < 0 else lens[a]) + (1 if b < 0 else lens[b])
    longest = int(lens.max()) if len(lens) else 1
    assert B.stats()["depth"] <= 1.4405 * np.log2(longest + 2)
    assert B.stats()["depth"] <= G.stats()["depth"]
    # balancing a balanced grammar changes nothing
    ex2 = export_all(B.balanced())
    for key in ("nodes", "lvl_off", "c_ref"):
        np.testing.assert_array_equal(ex2[key], ex[key])


def test_balanced_degenerate_grammars(gcs):
    # no rules at all, all rows empty, a 1 x 1 matrix, one long repeated row
    # (a deep right comb that balancing must flatten to about log2 of its
    # length): the same products and a valid packed grammar
    cases = [
        (2, 4, np.array([0, 2, 4], np.int64), np.array([0, 1, 2, 3], np.int32), np.array([1, 2, 3, 4], np.float32)),
        (3, 5, np.zeros(4, np.int64), np.zeros(0, np.int32), np.zeros(0, np.float32)),
        (1, 1, np.array([0, 1], np.int64), np.array([0], np.int32), np.array([-2.5], np.float32)),
    ]
    m = 4096
    row = np.arange(m, dtype=np.int32)
    rep = 6
    cases.append((rep, m, np.arange(rep + 1, dtype=np.int64) * m, np.tile(row, rep),
                  np.tile(np.where(row % 3 == 0, 1.0, 2.0).astype(np.float32), rep)))
    for n, m, rp, c, v in cases:
        G = gcs.Grammar(n, m, rp, c, v)
        B = G.balanced()
        check_grammar(B, rp, c, v, n, m, repair_end_state=False)
        assert B.stats()["depth"] <= max(1, G.stats()["depth"])
    assert B.stats()["depth"] <= 1.4405 * np.log2(m + 2)
