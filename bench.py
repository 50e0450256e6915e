#!/usr/bin/env python
"""Benchmark: single-vector genotype right product y = G beta on one GB300.

Workload (default): 10,000 individuals x 50,000 variants, genotypes in
{0,1,2} from a 100-founder mosaic (switch = mutation = 1e-3, seed 0), one
grammar built once (RePair, then height-balanced: --grammar repair keeps
RePair's grammar as built), then K timed products with fresh beta ~ N(0,1)
float32. A step is one whole product (leaf gather, every level, row emit).

Timing: W warm-up steps, then K steps, each timed with CUDA events on the
launching stream; the L2 cache (129 MB) is flushed by writing a 512 MB buffer
before every step, outside the events. value = K / (sum of step times). The
same K products back to back without flushes are reported as "hot".
e2e: the same products through gc_matvec_host (pinned host beta in, y out,
copies inside the timed region, wall clock per call).

Multi-GPU (torchrun): every rank runs an independent replica of the
workload (replicas only: the product needs no exchange); value = all
products / the slowest rank's time.

--impl reference times the CPU oracle (float64 direct product over the CSR
rows, one BLAS thread) on the same workload; each step is a bounded sample
of rows, scaled to products per second.

Other workloads (--workload): the same matrix with 16, 64 or 256 right-hand sides, the
small and the row-blocked 50,000 x 200,000 genotype matrices, the
2,000,000-node copy-model graph under the Boolean policy (with the
reachability fixpoint) and, with the "_minplus" suffix, the tropical policy
on the genotype matrix and on the graph (with the shortest-path fixpoint,
unit edge lengths), and the left product x = M^T y on the genotype matrix
("_left": a step is one left product; its algorithmic bytes are the plan's
arrays, each read once, plus y and x); with the "_dataflow" suffix, the genotype
product and the graph under the dataflow schedule (per-block ready flags
instead of grid barriers; its own layout).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gcsynth  # noqa: E402

METRIC = "matvecs/s and effective HBM GB/s (% of roofline) for y=Gβ on one GB300"
# k = 1 products run over the height-balanced grammar (faster on every one
# measured); the wide batches keep RePair's (the balanced grammar has more
# rules, and their values dominate a wide product's traffic)
WORKLOADS = {
    "geno_10k_50k": dict(gen=gcsynth.GENO_MEDIUM, k=1, grammar="balanced"),
    "geno_10k_50k_k16": dict(gen=gcsynth.GENO_MEDIUM, k=16),
    "geno_10k_50k_k64": dict(gen=gcsynth.GENO_MEDIUM, k=64),
    "geno_10k_50k_k256": dict(gen=gcsynth.GENO_MEDIUM, k=256),
    "geno_1k_2k": dict(gen=gcsynth.GENO_SMALL, k=1, grammar="balanced"),
    "geno_50k_200k": dict(gen=gcsynth.GENO_LARGE, k=1, grammar="balanced"),
    "graph_2m": dict(graph=gcsynth.GRAPH, k=1, grammar="balanced"),
    # tropical (min, +): one Bellman-Ford relaxation per product
    "geno_10k_50k_minplus": dict(gen=gcsynth.GENO_MEDIUM, k=1, policy="minplus", grammar="balanced"),
    # the left product x = M^T y (float32, one vector)
    "geno_10k_50k_left": dict(gen=gcsynth.GENO_MEDIUM, k=1, op="left", grammar="balanced"),
    "graph_2m_minplus": dict(graph=gcsynth.GRAPH, k=1, policy="minplus", grammar="balanced"),
    # the same products under the dataflow schedule (its own layout)
    "geno_10k_50k_dataflow": dict(gen=gcsynth.GENO_MEDIUM, k=1, schedule="dataflow"),
    "graph_2m_dataflow": dict(graph=gcsynth.GRAPH, k=1, schedule="dataflow"),
}
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="geno_10k_50k", choices=sorted(WORKLOADS))
    ap.add_argument("--grammar", default=None, choices=["repair", "balanced"],
                    help="RePair's grammar as built, or its AVL height-balanced form (default: the workload's)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the CPU-oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def make_csr(gen):
    rp, c, v = gcsynth.genotype_csr(**gen)
    return gen["n"], gen["m"], rp, c, v


def make_blocked(gcs, gen):
    """Streaming build of a row-blocked genotype matrix: each block of
    ``block_rows`` rows is generated and compressed on its own, several at a
    time (a block's CSR and RePair peak near 22 bytes per matrix entry)."""
    mem = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    per_block = 22 * gen["block_rows"] * gen["m"]
    workers = max(1, min(os.cpu_count() or 1, int(0.75 * mem // per_block), 8))
    return gcs.Grammar.from_row_blocks(gen["n"], gen["m"], gen["block_rows"],
                                       lambda r0, r1: gcsynth.genotype_csr(**gen, r0=r0, r1=r1),
                                       workers=workers)


def make_graph(gp):
    rp, col = gcsynth.copy_model_graph(**gp)
    return gp["nodes"], gp["nodes"], rp, col, None


def compulsory_bytes(st, k, elem=4):
    """Algorithmic bytes of one product: every array the sweep must read or
    write once -- child pairs of all layered nodes (8 B), one leaf code per
    terminal (4 B), the level table, C offsets and references (4 B), x and y."""
    L = st["depth"]
    return (8 * st["n_nodes"] + 4 * st["n_terminals"] + 4 * 8 * (L + 2) + 4 * (st["n"] + 1)
            + 4 * st["c_len"] + elem * k * (st["m"] + st["n"]))


class ClockSampler:
    """SM clock and throttle reasons sampled DURING the timed region.

    Reads NVML directly (libnvidia-ml, read-only queries) from a thread about
    every millisecond, because a timed region of a few milliseconds is far
    shorter than nvidia-smi's sampling period; nvidia-smi is the fallback.
    """

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.max_mhz = None
        self._stop = False
        self._thread = None
        self._nvml = None
        self._smi = None

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        return lib, h, get_reasons

    def _loop(self):
        import ctypes
        lib, h, get_reasons = self._nvml
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        try:
            self._nvml = self._open_nvml()
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
            while not self.samples and self._thread.is_alive():   # first sample before timing starts
                time.sleep(0.0005)
        except (OSError, AttributeError):
            self._nvml = None
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.index}", "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._smi = None
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            time.sleep(0.002)   # one more sample at the end of the region
            self._stop = True
            self._thread.join(timeout=2)
        if self._smi is not None:
            self._smi.terminate()
            try:
                out, _ = self._smi.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
                out, _ = self._smi.communicate()
            for r in out.strip().splitlines():
                f = [x.strip() for x in r.split(",")]
                try:
                    self.samples.append((int(float(f[0])), int(f[2], 16)))
                    self.max_mhz = int(float(f[1]))
                except (ValueError, IndexError):
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        mhz = [c for c, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(name for bit, name in self.REASONS.items() if bits & bit)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "nvml" if self._nvml else "nvidia-smi"}


ORACLE_SAMPLE_ROWS = 2000


def _oracle_sample(workload, seconds, steps):
    """Runs in a child process whose BLAS is limited to one thread. Generates
    the first ORACLE_SAMPLE_ROWS rows of the workload's matrix once, then for
    each of ``steps`` steps runs the oracle's float64 direct product over
    blocks of 250 of those rows until ``seconds`` pass; prints, per step, the
    rows done and the time, as JSON."""
    from oracle import direct
    wl = WORKLOADS[workload]
    k = wl["k"]
    minplus = wl.get("policy") == "minplus"
    if "graph" in wl:
        gp = wl["graph"]
        rp, c = gcsynth.copy_model_graph(**gp)
        rows = min(gp["nodes"], ORACLE_SAMPLE_ROWS * 100)
        rp, c = rp[:rows + 1], c[:rp[rows]]
        if minplus:
            x = gcsynth.beta(gp["nodes"], seed=0)
            ones = np.ones(len(c), np.float32)
            product = lambda a, b: direct.matvec_minplus(rp[a:b + 1] - rp[a], c[rp[a]:rp[b]], ones[rp[a]:rp[b]], x)
        else:
            x = np.random.default_rng(0).integers(0, 2**63, gp["nodes"], dtype=np.uint64)
            product = lambda a, b: direct.matvec_or(rp[a:b + 1] - rp[a], c[rp[a]:rp[b]], x)
        block = 25000
    else:
        gen = wl["gen"]
        rows = min(gen["n"], ORACLE_SAMPLE_ROWS)
        rp, c, v = gcsynth.genotype_csr(**dict(gen, r1=rows))
        x = gcsynth.beta(gen["m"], seed=0, k=k)
        if minplus:
            product = lambda a, b: direct.matvec_minplus(rp[a:b + 1] - rp[a], c[rp[a]:rp[b]], v[rp[a]:rp[b]], x)
        elif wl.get("op") == "left":
            yv = gcsynth.beta(gen["n"], seed=0)
            product = lambda a, b: direct.left_matvec_f64(rp[a:b + 1] - rp[a], c[rp[a]:rp[b]], v[rp[a]:rp[b]],
                                                          yv[a:b], gen["m"])
        else:
            product = lambda a, b: direct.matvec_f64(rp[a:b + 1] - rp[a], c[rp[a]:rp[b]], v[rp[a]:rp[b]], x)
        block = 250
    out = []
    for _ in range(steps):
        done_rows = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            a = done_rows % rows
            b = min(rows, a + block)
            product(a, b)
            done_rows += b - a
        out.append({"rows": done_rows, "seconds": time.perf_counter() - t0})
    print(json.dumps(out), flush=True)


def cpu_oracle_rates(workload, seconds, steps=1):
    """Products per second of the CPU oracle, one figure per step, each step
    a bounded sample (``seconds``) of the workload's rows; timed in a child
    process with one BLAS / OpenMP thread."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample",
                          "--workload", workload, "--cpu-seconds", str(seconds), "--steps", str(steps)],
                         env=env, capture_output=True, text=True, check=True).stdout
    recs = json.loads(out.strip().splitlines()[-1])
    wl = WORKLOADS[workload]
    n = wl["graph"]["nodes"] if "graph" in wl else wl["gen"]["n"]
    return [(r["rows"] / n) / r["seconds"] for r in recs], recs


def cpu_oracle_all_cores(workload, seconds):
    """The same oracle sample on every host core the process may use: one
    child process per core (one BLAS thread each), all running at once for
    ``seconds``; products per second summed over the children."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload,
           "--cpu-seconds", str(seconds), "--steps", "1"]
    procs = [subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
             for _ in range(cores)]
    wl = WORKLOADS[workload]
    n = wl["graph"]["nodes"] if "graph" in wl else wl["gen"]["n"]
    rows = secs = 0.0
    total = 0.0
    for p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("oracle sample child failed")
        r = json.loads(out.strip().splitlines()[-1])[0]
        total += (r["rows"] / n) / r["seconds"]
        rows += r["rows"]
        secs = max(secs, r["seconds"])
    return total, cores, rows


def grammar_sweep_rates(G, gen, seconds):
    """Theorem 2.3's W-array sweep over the same grammar on the host cores
    (baselines/wsweep.c, float64), sequential and on every core the process may
    use: the CPU grammar baseline, reported beside the oracle; and the direct
    CSR product of the same matrix the same two ways."""
    from baselines.wsweep import CsrProduct, GrammarSweep
    t0 = time.perf_counter()
    sw = GrammarSweep.from_grammar(G)
    prep = time.perf_counter() - t0
    x = gcsynth.beta(gen["m"], seed=0).astype(np.float64)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    seq = sw.rate(x, 1, seconds / 4)
    par = sw.rate(x, cores, seconds / 4)
    out = {"kind": "grammar sweep (Theorem 2.3 W-array over the same grammar, float64, C + OpenMP)",
           "unit": "matvec/s", "sequential": seq, "parallel": par, "cores": cores, "prepare_seconds": round(prep, 2)}
    del sw
    csr = CsrProduct(*make_csr(gen)[2:5])
    out["csr"] = {"kind": "direct CSR product of the same matrix (float64, C + OpenMP)",
                  "sequential": csr.rate(x, 1, seconds / 4), "parallel": csr.rate(x, cores, seconds / 4)}
    return out


def oracle_sample_text(workload):
    wl = WORKLOADS[workload]
    minplus = wl.get("policy") == "minplus"
    if "graph" in wl:
        what = "float32 min-plus product" if minplus else "Boolean OR product"
        return (f"{what} of the first {min(wl['graph']['nodes'], ORACLE_SAMPLE_ROWS * 100)} rows "
                + ("" if minplus else "(64 sources per word) ") + "in blocks of 25,000")
    what = ("float32 min-plus" if minplus else "float64 direct left (M^T y)" if wl.get("op") == "left"
            else "float64 direct")
    return f"{what} product over the first {ORACLE_SAMPLE_ROWS} rows in blocks of 250"


def workload_policy(wl):
    """(policy, element bytes, dtype name) of a workload."""
    pol = wl.get("policy", "or" if "graph" in wl else "f32")
    return pol, (8 if pol in ("or", "i64") else 4), {"or": "u64", "i64": "i64", "f32": "f32", "minplus": "f32"}[pol]


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    k = wl["k"]
    gen = dict(n=wl["graph"]["nodes"], m=wl["graph"]["nodes"]) if "graph" in wl else wl["gen"]
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    rates, _ = cpu_oracle_rates(args.workload, per_step, args.warmup + args.steps)
    rates = rates[args.warmup:]
    value = len(rates) / sum(1.0 / r for r in rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "matvec/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if wl.get("policy") == "minplus" else ("u64" if "graph" in wl else "f64"),
        "data": "synthetic",
        "config": {"workload": args.workload, "n": gen["n"], "m": gen["m"], "k": k},
        "cpu_baseline": {"value": value, "unit": "matvec/s", "cores": 1, "kind": "oracle",
                         "sample": f"{oracle_sample_text(args.workload)}, {per_step:.1f} s per step, "
                                   "scaled to whole products"},
        "e2e": {"value": value, "unit": "matvec/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def engine_code_hash(text: str) -> str:
    """sha256 prefix of a CUDA/C++ source with its comments, blank lines and
    trailing spaces removed: equal exactly when the code is equal."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':   # string literal: kept whole (a "//" inside is not a comment)
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).split("\n")]
    code = "\n".join(ln for ln in lines if ln)
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def profile_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel code (comments aside; else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "grammar_compressed_sparse_gb300", "csrc", "engine.cu")
    try:
        with open(src, encoding="utf-8") as f:
            h = engine_code_hash(f.read())
    except (OSError, UnicodeDecodeError):
        return None
    return rec.get("dram_bytes_per_launch") if rec.get("engine_code_sha") == h else None


class LeftAdapter:
    """The left product behind the calls the timing loop makes: input y
    (n values), output x (m values); the host-buffer form copies pinned y in
    and x out around gc_left_matvec and synchronises."""

    def __init__(self, gcs, G, dev, torch):
        self.eng = gcs.LeftEngine(G, device=dev)
        self.layout = self.eng.layout
        self._torch = torch
        self._yd = torch.empty(self.eng.n, dtype=torch.float32, device=dev)
        self._xd = torch.empty(self.eng.m, dtype=torch.float32, device=dev)

    def matvec(self, y, x, stream=None):
        self.eng.matvec(y, x, stream=stream)

    def matvec_host(self, yh, xh, stream=None):
        torch = self._torch
        with torch.cuda.stream(stream):
            self._yd.copy_(torch.from_numpy(yh), non_blocking=True)
            self.eng.matvec(self._yd, self._xd, stream=stream)
            torch.from_numpy(xh).copy_(self._xd, non_blocking=True)
        stream.synchronize()

    def launch_count(self):
        return self.eng.launch_count()


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from grammar_compressed_sparse_gb300 import build as gbuild
    gbuild.build()
    import grammar_compressed_sparse_gb300 as gcs

    wl = WORKLOADS[args.workload]
    k = wl["k"]
    graph = "graph" in wl
    t0 = time.perf_counter()
    if graph:
        gp = wl["graph"]
        gen = dict(n=gp["nodes"], m=gp["nodes"])
        key = f"graph:{sorted(gp.items())}"
        load = lambda: gcs.cached_grammar(key, lambda: make_graph(gp))  # noqa: E731
    else:
        gen = wl["gen"]
        key = f"genotype:{sorted(gen.items())}"
        if "block_rows" in gen:
            load = lambda: gcs.cached_grammar(key, None, build=lambda: make_blocked(gcs, gen))  # noqa: E731
        else:
            load = lambda: gcs.cached_grammar(key, lambda: make_csr(gen))  # noqa: E731
    balanced = (args.grammar or wl.get("grammar", "repair")) == "balanced"
    if balanced:
        G = gcs.cached_grammar(key + ":balanced", None, build=lambda: load().balanced(),
                               extra_sources=("balance.cpp",))
    else:
        G = load()
    build_s = time.perf_counter() - t0
    st = G.stats()
    policy, elem, dtype_name = workload_policy(wl)
    minplus = policy == "minplus"
    left = wl.get("op") == "left"
    stream = torch.cuda.current_stream(dev)
    eng = LeftAdapter(gcs, G, dev, torch) if left else gcs.Engine(G, policy, k, device=dev,
                                                                  schedule=wl.get("schedule", "persistent"))
    # the left product reads n values and writes m
    n_in, n_out = (gen["n"], gen["m"]) if left else (gen["m"], gen["n"])

    nvec = args.warmup + args.steps
    if graph and not minplus:
        xs = [torch.from_numpy(np.random.default_rng(rank * 1000 + i).integers(
            0, 2**63, gen["m"], dtype=np.int64)).to(dev) for i in range(min(nvec, 8))]
        y = torch.empty(gen["n"], dtype=torch.int64, device=dev)
    else:
        xs = [torch.from_numpy(gcsynth.beta(n_in, seed=(rank * 1000 + i) % 100, k=k)).to(dev)
              for i in range(min(nvec, 100))]
        y = torch.empty((n_out,) if k == 1 else (n_out, k), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(i, timed_events=None):
        flush.fill_(i & 0xff)
        if timed_events is not None:
            timed_events[0].record(stream)
        eng.matvec(xs[i % len(xs)], y, stream=stream)
        if timed_events is not None:
            timed_events[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    launches_per_step = eng.launch_count()

    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            step(args.warmup + i, events[i])
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    times_ms = [a.elapsed_time(b) for a, b in events]
    total_s = sum(times_ms) / 1e3
    if world > 1:
        t = torch.tensor([total_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_s = float(t.item())
    value = world * args.steps / total_s

    # hot: the same products back to back, no flush between them (the
    # grammar of the 10,000 x 50,000 matrix is about the size of L2), timed
    # as one stretch; reported beside the cold figure, not as the value
    # (into a buffer of their own: y keeps the last timed product, which the
    # parity check below reads)
    y_hot = torch.empty_like(y)
    hot0, hot1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    hot0.record(stream)
    for i in range(args.steps):
        eng.matvec(xs[i % len(xs)], y_hot, stream=stream)
    hot1.record(stream)
    torch.cuda.synchronize(dev)
    hot_ms = hot0.elapsed_time(hot1) / args.steps

    # end to end through the host-buffer entry point (pinned x in, y out)
    xh = [xx.cpu().pin_memory().numpy() for xx in xs[:8]]
    yh = torch.empty(y.shape, dtype=y.dtype).pin_memory().numpy()
    for i in range(args.warmup):
        eng.matvec_host(xh[i % len(xh)], yh, stream=stream)
    e2e_t = 0.0
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        eng.matvec_host(xh[i % len(xh)], yh, stream=stream)
        e2e_t += time.perf_counter() - t1
    e2e = world * args.steps / e2e_t if world == 1 else None
    if world > 1:
        t = torch.tensor([e2e_t], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e = world * args.steps / float(t.item())

    # graph workloads: the reachability (Boolean) or shortest-path (min-plus)
    # fixpoint from 64 sources, timed once
    fixpoint = None
    if graph:
        srcs = gcsynth.sources(gen["n"], gp["sources"], gp["seed"])
        if minplus:
            x0d = torch.from_numpy(gcsynth.frontier_distances(gen["n"], srcs)).to(dev)
        else:
            x0d = torch.from_numpy(gcsynth.frontier(gen["n"], srcs).view(np.int64)).to(dev)
        run = gcs.capi.gc_sssp if minplus else gcs.capi.gc_reach
        xfp = torch.empty_like(x0d)
        itd = torch.zeros(1, dtype=torch.int32, device=dev)
        run(eng._h, x0d, xfp, 1000, itd, stream)    # once untimed (first-call set-up)
        torch.cuda.synchronize(dev)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t1 = time.perf_counter()
        f0.record(stream)
        rc = run(eng._h, x0d, xfp, 1000, itd, stream)
        f1.record(stream)   # after every kernel the call enqueued, early-return ones included
        torch.cuda.synchronize(dev)
        wall_fp = time.perf_counter() - t1
        dev_ms = f0.elapsed_time(f1)
        iters = int(itd.item())
        fixpoint = {"kind": "shortest paths, unit lengths" if minplus else "reachability, 64-bit source bitsets",
                    "iterations": iters, "seconds": round(wall_fp, 5), "device_ms": round(dev_ms, 4),
                    "per_iteration_ms": round(dev_ms / max(1, iters), 4),
                    "vs_iterations_x_product": round(dev_ms / max(1e-9, iters * 1e3 * total_s / args.steps), 3),
                    "vs_iterations_x_hot_product": round(dev_ms / max(1e-9, iters * hot_ms), 3),
                    "status": rc}

    if rank != 0:
        return
    # parity spot check of the last product against the oracle, 200 rows
    from oracle import direct
    y_last = y.cpu().numpy()
    if graph and minplus:
        x_last = xs[(args.warmup + args.steps - 1) % len(xs)].cpu().numpy()
        rp, col = gcsynth.copy_model_graph(**gp)
        rp, col = rp[:201], col[:rp[200]]
        y_ref = direct.matvec_minplus(rp, col, np.ones(len(col), np.float32), x_last)
        ok = bool(np.array_equal(y_last[:200].view(np.uint32), y_ref.view(np.uint32)))
        worst = 0.0 if ok else float("inf")
    elif graph:
        x_last = xs[(args.warmup + args.steps - 1) % len(xs)].cpu().numpy().view(np.uint64)
        rp, col = gcsynth.copy_model_graph(**gp)
        y_ref = direct.matvec_or(rp, col, x_last)
        ok = bool(np.array_equal(y_last.view(np.uint64), y_ref))
        worst = 0.0 if ok else float("inf")
    elif left:
        # one more product with y zero past the first 200 rows: x is then the
        # left product of those rows alone
        rp, c, v = gcsynth.genotype_csr(**dict(gen, r1=200))
        y200 = np.zeros(gen["n"], np.float32)
        y200[:200] = gcsynth.beta(200, seed=123)
        xd = torch.empty(gen["m"], dtype=torch.float32, device=dev)
        eng.matvec(torch.from_numpy(y200).to(dev), xd, stream=stream)
        torch.cuda.synchronize(dev)
        x_ref, bnd = direct.left_matvec_f64(rp, c, v, y200[:200], gen["m"])
        ok, worst = direct.within_tolerance(xd.cpu().numpy(), x_ref, bnd, 1e-4)
    elif minplus:
        rp, c, v = gcsynth.genotype_csr(**dict(gen, r1=200))
        xl = gcsynth.beta(gen["m"], seed=(args.warmup + args.steps - 1) % len(xs) % 100, k=k)
        y_ref = direct.matvec_minplus(rp, c, v, xl)
        ok = bool(np.array_equal(y_last[:200].view(np.uint32), y_ref.view(np.uint32)))
        worst = 0.0 if ok else float("inf")
    else:
        rp, c, v = gcsynth.genotype_csr(**dict(gen, r1=200))
        xl = gcsynth.beta(gen["m"], seed=(args.warmup + args.steps - 1) % len(xs) % 100, k=k)
        y_ref, bnd = direct.matvec_f64(rp, c, v, xl)
        ok, worst = direct.within_tolerance(y_last[:200], y_ref, bnd, 1e-4)

    peak, peak_src = peaks()
    bytes_step = (eng.layout["grammar_bytes"] + 4 * (gen["n"] + gen["m"])) if left else compulsory_bytes(st, k, elem)
    mean_s = total_s / args.steps
    achieved = bytes_step / mean_s / 1e9
    lay = eng.layout
    footprint = lay["grammar_bytes"] + lay["scratch_bytes"] + elem * k * (gen["m"] + gen["n"])
    if left:
        kernel_name = "whole left product: left_step_kernel x (depth + 3)"
    elif eng.schedule == "dataflow":
        kernel_name = "whole product: flow_kernel + " + ("slice_kernel" if not graph else "emit_kernel (rows)")
    else:
        kernel_name = "whole product: sweep_kernel" + (" + slice_kernel" if launches_per_step == 2 else "")
    cpu = cpu_all = None
    if not args.no_cpu_baseline:
        rates, recs = cpu_oracle_rates(args.workload, args.cpu_seconds)
        cpu = {"value": rates[0], "unit": "matvec/s", "cores": 1, "kind": "oracle",
               "sample": f"{recs[0]['rows']} rows ({recs[0]['rows'] / gen['n']:.3f} products) of the same "
                         f"matrix in {recs[0]['seconds']:.1f} s: {oracle_sample_text(args.workload)}, "
                         "one BLAS thread"}
        # the same oracle on every host core (one process a core), reported beside it
        try:
            v_all, cores_all, rows_all = cpu_oracle_all_cores(args.workload, max(2.0, args.cpu_seconds / 3))
            cpu_all = {"value": v_all, "unit": "matvec/s", "cores": cores_all, "kind": "oracle",
                       "sample": f"{int(rows_all)} rows in all over {cores_all} processes, each "
                                 f"{max(2.0, args.cpu_seconds / 3):.1f} s of {oracle_sample_text(args.workload)}, "
                                 "one BLAS thread each; products per second summed"}
        except Exception as e:  # noqa: BLE001
            cpu_all = {"error": f"{type(e).__name__}: {e}"[:200]}
    # the CPU grammar sweep (genotype workloads, float32 sum, one vector);
    # reported only, and never allowed to cost the line
    cpu_sweep = None
    if not args.no_cpu_baseline and not graph and not left and policy == "f32" and k == 1:
        try:
            cpu_sweep = grammar_sweep_rates(G, gen, max(2.0, args.cpu_seconds / 2))
        except Exception as e:  # noqa: BLE001
            cpu_sweep = {"error": f"{type(e).__name__}: {e}"[:200]}
    line = {
        "metric": METRIC, "value": value, "unit": "matvec/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_name, "data": "synthetic",
        "config": {"workload": args.workload, "n": gen["n"], "m": gen["m"], "k": k,
                   "policy": policy, **({"op": "left: x = M^T y"} if left else {}),
                   **({"graph": "copy model, unit edge lengths" if minplus else "copy model, 64-bit source bitsets"}
                      if graph else
                      {"founders": gen["founders"], "switch": gen["switch"], "mutation": gen["mutation"]}),
                   "grammar": "RePair, AVL height-balanced" if balanced else "RePair",
                   "l2": "flushed before every step (512 MB write, outside the events)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "traffic": profile_traffic(f"sweep:{args.workload}" + (":balanced" if balanced else "")),
                     "kernel": kernel_name,
                     "algorithmic_bytes_per_launch": bytes_step},
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "cpu_grammar_sweep": cpu_sweep,
        "e2e": {"value": e2e, "unit": "matvec/s", "h2d_bytes_per_step": elem * k * n_in,
                "d2h_bytes_per_step": elem * k * n_out},
        "vectors_per_s": value * k,
        "fixpoint": fixpoint,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "grammar": {"depth": st["depth"], "max_width": st["max_width"], "rules": st["n_rules"],
                    "pass_through": st["n_pass"], "nodes": st["n_nodes"], "c_len": st["c_len"],
                    "roots": st["n_roots"], "completion_overhead": st["n_pass"] / max(1, st["n_rules"]),
                    "build_seconds": round(build_s, 2), "repair_seconds": round(st["repair_seconds"], 2)},
        "footprint": {"engine_bytes": footprint, "csr_bytes": lay["csr_bytes"],
                      "ratio": lay["csr_bytes"] / footprint},
        "parity": {"rows_checked": 200, "max_scaled_error": worst, "ok": ok},
        "wall_s": round(wall, 4),
        "step_ms": {"median": statistics.median(times_ms), "min": min(times_ms), "max": max(times_ms)},
        "hot": {"ms_per_step": hot_ms, "value": 1e3 / hot_ms,
                "note": "back-to-back products without the L2 flush (the headline value is flushed)"},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.oracle_sample:
        _oracle_sample(args.workload, args.cpu_seconds, args.steps)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
