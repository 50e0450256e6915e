"""bench.py's output contract, on the CPU: the reference arm (the CPU oracle)
prints one JSON line with the keys the driver reads, and our arm refuses to
run without a CUDA device (the product path has no CPU fallback)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, cwd=ROOT)


@pytest.mark.parametrize("workload", ["geno_1k_2k", "geno_10k_50k_left"])
def test_reference_arm_prints_one_json_line(workload):
    r = _bench("--impl", "reference", "--workload", workload, "--steps", "2", "--warmup", "1", "--cpu-seconds", "2")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["workload"] == workload and d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_our_arm_needs_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    r = _bench("--steps", "1", "--warmup", "1", "--no-cpu-baseline")
    assert r.returncode != 0
    assert "CUDA" in (r.stdout + r.stderr)


def test_traffic_record_follows_the_kernel_code():
    # the bench line's DRAM traffic comes from profiles/traffic.json only while
    # engine.cu's code (comments aside) is the code the counters were taken on
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    src = 'int f(int a) { // add one\n  return a + 1; /* done */ }\nconst char* s = "x // y";\n'
    h = b.engine_code_hash(src)
    assert b.engine_code_hash(src.replace("// add one", "// plus one")) == h
    assert b.engine_code_hash(src + "\n\n// trailing note\n") == h
    assert b.engine_code_hash(src.replace("a + 1", "a + 2")) != h
    assert b.engine_code_hash(src.replace('"x // y"', '"x // z"')) != h   # strings are code
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    with open(os.path.join(ROOT, "grammar_compressed_sparse_gb300", "csrc", "engine.cu"), encoding="utf-8") as f:
        cur = b.engine_code_hash(f.read())
    for key, rec in recs.items():
        assert rec["dram_bytes_per_launch"] > 0 and os.path.exists(os.path.join(ROOT, rec["source"]))
        got = b.profile_traffic(key)
        assert got == (rec["dram_bytes_per_launch"] if rec["engine_code_sha"] == cur else None)
