"""Benchmark: batch-1 block-quantized decode (tok/s) and quant-GEMV HBM GB/s.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A "step" is one pass of the hot path over one
batch of synthetic input: one decode token for the decode workloads, one
GEMV launch for the GEMV workloads.  Inputs are seeded and synthetic (random
weights of the named shape; no checkpoint exists here).  Multi-GPU runs are
independent replicas ("scaling": "weak"): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "batch-1 decode tok/s (8B/70B shapes); quant-GEMV HBM GB/s and % of GB300 peak"


# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def profile_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary for this kernel and
    workload, if its recorded source hash still matches the kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    src = os.path.join(ROOT, "block_quantized_gemv_nt_gb300", "csrc", "qgemv.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    got = {}
    for ln in open(path):
        if ":" in ln:
            k, v = ln.split(":", 1)
            got[k.strip().strip("-* `")] = v.strip().strip("`")
    if got.get("source_sha256_16") != sha:
        return None
    try:
        return float(got["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# GEMV workloads: Q8_0 4096x4096 (seed 0) and the format sweep shapes
def parse_gemv(name):
    """gemv_<fmt>_<rows>x<cols>, e.g. gemv_q8_0_4096x4096, gemv_q4_k_8192x28672"""
    import synth
    parts = name.split("_")
    fmt = synth.FMT_BY_NAME[(parts[1] + "_" + parts[2]).upper()]
    rows, cols = (int(v) for v in parts[3].split("x"))
    return fmt, rows, cols


def bench_gemv(args, rank, world):
    import torch

    import synth
    from block_quantized_gemv_nt_gb300 import nt

    fmt, rows, cols = parse_gemv(args.workload)
    seed = 0 if (fmt == synth.Q8_0 and rows == 4096 and cols == 4096) else 100 + fmt
    W = synth.quant_matrix(fmt, rows, cols, seed=seed, stream=0)
    x = synth.normal_f32(cols, seed=seed, stream=1)
    ctx = nt.Context(torch.cuda.current_device())
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    wbytes = W.nbytes
    ncopy = max(1, -(-4 * l2 // wbytes))          # rotate copies so the set is >= 4x L2
    Wd = [torch.from_numpy(W).cuda() for _ in range(ncopy)]
    xd = torch.from_numpy(x).cuda()
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()
    algo = wbytes + 4 * cols + 4 * rows
    with torch.cuda.stream(st):
        for i in range(max(3, args.warmup)):
            nt.nt_gemv_q(ctx, fmt, Wd[i % ncopy], xd, y, rows, cols)
        st.synchronize()
        # CUDA graph of K launches over the rotating copies (launch overhead out of the way)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(args.steps):
                nt.nt_gemv_q(ctx, fmt, Wd[i % ncopy], xd, y, rows, cols)
        g.replay()
        st.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            torch.cuda.synchronize()
            e0.record(st)
            g.replay()
            e1.record(st)
            e1.synchronize()
        ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    per_launch_s = ms / 1e3 / args.steps
    gbs = algo / per_launch_s / 1e9
    peak, peak_kind = measured_peaks()

    # e2e through the C ABI with host buffers: x from pinned host in, y back to pinned host
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.empty(rows, dtype=torch.float32).pin_memory()
    xdev = torch.empty_like(xd)
    with torch.cuda.stream(st):
        for i in range(3):
            xdev.copy_(xh, non_blocking=True)
            nt.nt_gemv_q(ctx, fmt, Wd[i % ncopy], xdev, y, rows, cols)
            yh.copy_(y, non_blocking=True)
        st.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(st)
        for i in range(args.steps):
            xdev.copy_(xh, non_blocking=True)
            nt.nt_gemv_q(ctx, fmt, Wd[i % ncopy], xdev, y, rows, cols)
            yh.copy_(y, non_blocking=True)
        f1.record(st)
        f1.synchronize()
    e2e_s = max_over_ranks(f0.elapsed_time(f1), world) / 1e3 / args.steps
    ctx.sync()

    line = {
        "metric": METRIC, "value": round(gbs * world, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_launch_s * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (block-quantized weights)",
        "data": "synthetic seeded blocks", "impl": "ours",
        "config": {"workload": args.workload, "fmt": synth.FMT_NAMES[fmt], "rows": rows, "cols": cols,
                   "seed": seed, "l2": f"rotating {ncopy} weight copies ({ncopy * wbytes / 2**20:.0f} MiB >= 4x L2)"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": profile_traffic("qgemv", args.workload), "algo_bytes_per_launch": algo},
        "e2e": {"value": round(algo / e2e_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": 4 * cols,
                "d2h_bytes_per_step": 4 * rows},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_gemv(fmt, W, x, rows, cols, algo)
    return line


def cpu_gemv(fmt, W, x, rows, cols, algo, budget_s=10.0):
    import oracle
    xd = x.astype(np.float64)
    n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or n == 0:
        oracle.gemv(fmt, W, xd, rows, cols)
        n += 1
    dt = (time.perf_counter() - t0) / n
    return {"value": round(algo / dt / 1e9, 3), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} full oracle GEMVs ({rows}x{cols}) in {n * dt:.1f} s"}


# ---------------------------------------------------------------------------
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reference_arm(args, rank, world):
    """The oracle, as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    import synth
    if args.workload.startswith("gemv"):
        fmt, rows, cols = parse_gemv(args.workload)
        seed = 0 if (fmt == synth.Q8_0 and rows == 4096 and cols == 4096) else 100 + fmt
        W = synth.quant_matrix(fmt, rows, cols, seed=seed, stream=0)
        x = synth.normal_f32(cols, seed=seed, stream=1)
        algo = W.nbytes + 4 * cols + 4 * rows
        import oracle
        for _ in range(max(1, min(args.warmup, 2))):
            oracle.gemv(fmt, W, x.astype(np.float64), rows, cols)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.gemv(fmt, W, x.astype(np.float64), rows, cols)
        dt = (time.perf_counter() - t0) / args.steps
        v = round(algo / dt / 1e9, 3)
        return {"metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic seeded blocks",
                "impl": "reference", "config": {"workload": args.workload},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                                 "sample": f"{args.steps} full oracle GEMVs"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return {"impl": "reference", "unavailable": f"no reference arm for workload {args.workload}"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gemv_q8_0_4096x4096")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.workload.startswith("gemv"):
        line = bench_gemv(args, rank, world)
    else:
        raise SystemExit(f"unknown workload {args.workload}")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
