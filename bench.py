#!/usr/bin/env python
"""Benchmark: single-vector genotype right product y = G beta on one GB300.

Workload (default): 10,000 individuals x 50,000 variants, genotypes in
{0,1,2} from a 100-founder mosaic (switch = mutation = 1e-3, seed 0), one
grammar built once, then K timed products with fresh beta ~ N(0,1) float32.
A step is one whole product (leaf gather, every level, row emit).

Timing: W warm-up steps, then K steps, each timed with CUDA events on the
launching stream; the L2 cache (129 MB) is flushed by writing a 512 MB buffer
before every step, outside the events. value = K / (sum of step times).
e2e: the same products through gc_matvec_host (pinned host beta in, y out,
copies inside the timed region, wall clock per call).

Multi-GPU (torchrun): every rank runs an independent replica of the
workload (replicas only: the product needs no exchange); value = all
products / the slowest rank's time.

--impl reference times the CPU oracle (float64 direct product over the CSR
rows, one BLAS thread) on the same workload; each step is a bounded sample
of rows, scaled to products per second.
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
WORKLOADS = {
    "geno_10k_50k": dict(gen=gcsynth.GENO_MEDIUM, k=1),
    "geno_10k_50k_k16": dict(gen=gcsynth.GENO_MEDIUM, k=16),
    "geno_1k_2k": dict(gen=gcsynth.GENO_SMALL, k=1),
}
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="geno_10k_50k", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the CPU-oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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


def compulsory_bytes(st, k, alpha):
    """Algorithmic bytes of one product: every array the sweep must read or
    write once -- child pairs of all layered nodes (8 B), leaf records (col +
    value, 8 B), level tables, C offsets and references (4 B), x and y."""
    L = st["depth"]
    return (8 * st["n_nodes"] + 8 * alpha + 3 * 8 * (L + 2) + 4 * (st["n"] + 1)
            + 4 * st["c_len"] + 4 * k * (st["m"] + st["n"]))


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_oracle_rate(gen, k, seconds, rows_cap=None):
    """Products per second of the CPU oracle on a bounded sample of rows."""
    from threadpoolctl import threadpool_limits

    from oracle import direct
    rp, c, v = gcsynth.genotype_csr(**dict(gen, r1=rows_cap or gen["n"]))
    x = gcsynth.beta(gen["m"], seed=0, k=k)
    n = len(rp) - 1
    done_rows = 0
    t0 = time.perf_counter()
    with threadpool_limits(limits=1):
        while time.perf_counter() - t0 < seconds:
            a = done_rows % n
            b = min(n, a + 250)
            direct.matvec_f64(rp[a:b + 1] - rp[a], c[rp[a]:rp[b]], v[rp[a]:rp[b]], x)
            done_rows += b - a
    el = time.perf_counter() - t0
    products = done_rows / gen["n"]
    return products / el, {"rows": done_rows, "seconds": round(el, 3), "cores": 1}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    gen, k = wl["gen"], wl["k"]
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    rates = []
    for i in range(args.warmup + args.steps):
        r, info = cpu_oracle_rate(gen, k, per_step)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.mean(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "matvec/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "n": gen["n"], "m": gen["m"], "k": k},
        "cpu_baseline": {"value": value, "unit": "matvec/s", "cores": 1, "kind": "oracle",
                         "sample": f"float64 CSR rows in blocks of 250, about {per_step:.1f} s per step"},
        "e2e": {"value": value, "unit": "matvec/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def profile_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "grammar_compressed_sparse_gb300", "csrc", "engine.cu")
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    return rec.get("dram_bytes_per_launch") if rec.get("engine_sha") == h else None


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
    gen, k = wl["gen"], wl["k"]
    t0 = time.perf_counter()
    G = gcs.cached_grammar(f"genotype:{sorted(gen.items())}", lambda: make_csr(gen))
    build_s = time.perf_counter() - t0
    st = G.stats()
    alpha = st["n_terminals"]
    eng = gcs.Engine(G, "f32", k, device=dev)
    stream = torch.cuda.current_stream(dev)

    nvec = args.warmup + args.steps
    xs = [torch.from_numpy(gcsynth.beta(gen["m"], seed=(rank * 1000 + i) % 100, k=k)).to(dev)
          for i in range(min(nvec, 100))]
    y = torch.empty((gen["n"],) if k == 1 else (gen["n"], k), dtype=torch.float32, device=dev)
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

    # end to end through the host-buffer entry point (pinned beta in, y out)
    xh = [torch.from_numpy(gcsynth.beta(gen["m"], seed=i % 100, k=k)).pin_memory().numpy()
          for i in range(min(nvec, 8))]
    yh = torch.empty(y.shape, dtype=torch.float32).pin_memory().numpy()
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

    if rank != 0:
        return
    # parity spot check of the last product against the oracle, 200 rows
    from oracle import direct
    y_last = y.cpu().numpy()
    rp, c, v = gcsynth.genotype_csr(**dict(gen, r1=200))
    xl = gcsynth.beta(gen["m"], seed=(args.warmup + args.steps - 1) % len(xs) % 100, k=k)
    y_ref, bnd = direct.matvec_f64(rp, c, v, xl)
    ok, worst = direct.within_tolerance(y_last[:200], y_ref, bnd, 1e-4)

    peak, peak_src = peaks()
    bytes_step = compulsory_bytes(st, k, alpha)
    mean_s = total_s / args.steps
    achieved = bytes_step / mean_s / 1e9
    lay = eng.layout
    footprint = lay["grammar_bytes"] + lay["scratch_bytes"] + 4 * k * (gen["m"] + gen["n"])
    cpu = None
    if not args.no_cpu_baseline:
        r, info = cpu_oracle_rate(gen, k, args.cpu_seconds)
        cpu = {"value": r, "unit": "matvec/s", "cores": info["cores"], "kind": "oracle",
               "sample": f"{info['rows']} rows ({info['rows'] / gen['n']:.2f} products) of the same "
                         f"matrix in {info['seconds']} s, float64, one BLAS thread"}
    line = {
        "metric": METRIC, "value": value, "unit": "matvec/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "n": gen["n"], "m": gen["m"], "k": k,
                   "founders": gen["founders"], "switch": gen["switch"], "mutation": gen["mutation"],
                   "l2": "flushed before every step (512 MB write, outside the events)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "traffic": profile_traffic(f"sweep:{args.workload}"),
                     "kernel": "whole product (leaf gather + level combines + row emit)",
                     "algorithmic_bytes_per_launch": bytes_step},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e, "unit": "matvec/s", "h2d_bytes_per_step": 4 * k * gen["m"],
                "d2h_bytes_per_step": 4 * k * gen["n"]},
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
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
