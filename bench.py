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
import atexit
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
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
    """nvidia-smi clocks and throttle reasons sampled every 50 ms; each line is
    stamped with the host time it arrived, so the summary can keep the samples
    taken inside the timed region (mark_start / mark_end around it)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)
        self.n0 = len(self.lines)

    def wait_one_more(self, timeout=1.0):
        t0 = time.time()
        n = len(self.lines)
        while self.proc and len(self.lines) == n and time.time() - t0 < timeout:
            time.sleep(0.02)

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
        inside = [ln for t, ln in self.lines if self.t0 is not None and self.t1 is not None and self.t0 <= t <= self.t1]
        # the samples taken inside the timed region; the ones around it when the region is shorter than a sample
        use = inside if inside else [ln for _, ln in self.lines]
        for ln in use:
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
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_timed_region": len(inside), "sample_ms": 50}


def kernel_source_sha() -> str:
    """First 16 hex digits of the SHA-256 of the quant-GEMV sources (the
    kernel file and the block-format header it includes)."""
    h = hashlib.sha256()
    for f in ("qgemv.cu", "qformats.cuh"):
        h.update(open(os.path.join(ROOT, "block_quantized_gemv_nt_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary for this kernel and
    workload, if its recorded source hash still matches the kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha()
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
    """gemv_<fmt>_<rows>x<cols>, e.g. gemv_q8_0_4096x4096, gemv_q4_k_8192x28672;
    gemm_<fmt>_<rows>x<cols>_m<M> for the M-vector verify GEMM.  Returns
    (fmt, rows, cols, M)."""
    import synth
    parts = name.split("_")[1:]
    # the format name is one or two parts: q8_0, q4_k, f16, ...
    nf = 2 if (parts[0] + "_" + parts[1]).upper() in synth.FMT_BY_NAME else 1
    fmt = synth.FMT_BY_NAME["_".join(parts[:nf]).upper()]
    rows, cols = (int(v) for v in parts[nf].split("x"))
    M = int(parts[nf + 1][1:]) if len(parts) > nf + 1 else 1
    return fmt, rows, cols, M


def bench_gemv(args, rank, world):
    import torch

    import synth
    from block_quantized_gemv_nt_gb300 import nt

    fmt, rows, cols, M = parse_gemv(args.workload)
    gemm = args.workload.startswith("gemm")
    seed = 0 if (fmt == synth.Q8_0 and rows == 4096 and cols == 4096) else 100 + fmt
    W = synth.quant_matrix(fmt, rows, cols, seed=seed, stream=0)
    x = synth.normal_f32(M * cols, seed=seed, stream=1)
    ctx = nt.Context(torch.cuda.current_device())
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    wbytes = W.nbytes
    ncopy = max(1, -(-4 * l2 // wbytes))          # rotate copies so the set is >= 4x L2
    Wd = [torch.from_numpy(W).cuda() for _ in range(ncopy)]
    xd = torch.from_numpy(x).cuda()
    y = torch.empty(M * rows, dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()
    algo = wbytes + 4 * M * (cols + rows)

    def launch(i, xin):
        if gemm:
            nt.nt_gemm_q(ctx, fmt, Wd[i % ncopy], xin, y, rows, cols, M)
        else:
            nt.nt_gemv_q(ctx, fmt, Wd[i % ncopy], xin, y, rows, cols)

    with torch.cuda.stream(st):
        for i in range(max(3, args.warmup)):
            launch(i, xd)
        st.synchronize()
        # CUDA graph of K launches over the rotating copies (launch overhead out of the way)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(args.steps):
                launch(i, xd)
        g.replay()
        st.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            clk.wait_first()
            torch.cuda.synchronize()
            clk.mark_start()
            e0.record(st)
            g.replay()
            e1.record(st)
            e1.synchronize()
            clk.mark_end()
            clk.wait_one_more()
        ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    per_launch_s = ms / 1e3 / args.steps
    gbs = algo / per_launch_s / 1e9
    peak, peak_kind = measured_peaks()

    # e2e through the C ABI with host buffers: x from pinned host in, y back to pinned host
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.empty(M * rows, dtype=torch.float32).pin_memory()
    xdev = torch.empty_like(xd)
    with torch.cuda.stream(st):
        for i in range(3):
            xdev.copy_(xh, non_blocking=True)
            launch(i, xdev)
            yh.copy_(y, non_blocking=True)
        st.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(st)
        for i in range(args.steps):
            xdev.copy_(xh, non_blocking=True)
            launch(i, xdev)
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
        "config": {"workload": args.workload, "fmt": synth.FMT_NAMES[fmt], "rows": rows, "cols": cols, "M": M,
                   "seed": seed, "l2": f"rotating {ncopy} weight copies ({ncopy * wbytes / 2**20:.0f} MiB >= 4x L2)"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": profile_traffic("qgemv", args.workload), "algo_bytes_per_launch": algo},
        "e2e": {"value": round(algo / e2e_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": 4 * M * cols,
                "d2h_bytes_per_step": 4 * M * rows},
        "gpu_launches": args.steps * (2 if gemm else 1),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_gemv(fmt, W, x.reshape(M, cols), rows, cols, algo)
    return line


def cpu_gemv(fmt, W, X, rows, cols, algo, budget_s=10.0):
    """The oracle's GEMV over the same inputs (M vectors: M oracle GEMVs),
    with all host cores and, on a shorter sample, one thread."""
    import oracle
    Xd = X.astype(np.float64)

    def rate(budget):
        n = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget or n == 0:
            for xv in Xd:
                oracle.gemv(fmt, W, xv, rows, cols)
            n += 1
        return (time.perf_counter() - t0) / n, n

    dt, n = rate(budget_s)
    cores = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        dt1, n1 = rate(budget_s / 4)
    finally:
        oracle.set_num_threads(cores)
    return {"value": round(algo / dt / 1e9, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "value_1_thread": round(algo / dt1 / 1e9, 3),
            "sample": f"{n} full oracle passes ({len(Xd)} x {rows}x{cols}) in {n * dt:.1f} s; "
                      f"{n1} on one thread in {n1 * dt1:.1f} s"}


# ---------------------------------------------------------------------------
# Attention workload attn_<n_qh>x<n_kvh>x<n_pos>: one decode attention over an
# f16 KV cache of n_pos positions per step, rotating over enough caches to
# exceed 4x L2.
def bench_attn(args, rank, world):
    import torch

    import synth
    from block_quantized_gemv_nt_gb300 import nt

    H, G, P = (int(v) for v in args.workload.split("_")[1].split("x"))
    hd, stride = 128, P
    ctx = nt.Context(torch.cuda.current_device())
    kv_bytes = 2 * G * stride * hd * 2
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    ncopy = max(1, -(-4 * l2 // kv_bytes))
    K = torch.from_numpy(synth.normal_f16(G * stride * hd, 5, 1)).cuda()
    V = torch.from_numpy(synth.normal_f16(G * stride * hd, 5, 2)).cuda()
    Ks = [K.clone() for _ in range(ncopy)]
    Vs = [V.clone() for _ in range(ncopy)]
    q = torch.from_numpy(synth.normal_f32(H * hd, 5, 3)).cuda()
    out = torch.empty(H * hd, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for i in range(max(3, args.warmup)):
            nt.nt_attn_decode(ctx, q, Ks[i % ncopy], Vs[i % ncopy], out, H, G, hd, P, stride)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for i in range(args.steps):
                nt.nt_attn_decode(ctx, q, Ks[i % ncopy], Vs[i % ncopy], out, H, G, hd, P, stride)
        g.replay()
        st.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            clk.wait_first()
            clk.mark_start()
            e0.record(st)
            g.replay()
            e1.record(st)
            e1.synchronize()
            clk.mark_end()
            clk.wait_one_more()
    per = e0.elapsed_time(e1) / 1e3 / args.steps
    gbs = kv_bytes / per / 1e9
    peak, kind = measured_peaks()
    ctx.sync()
    return {"metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(per * 1e3, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 KV, f32 math", "data": "synthetic N(0,1) KV", "impl": "ours",
            "config": {"workload": args.workload, "l2": f"rotating {ncopy} KV caches"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind, "traffic": None,
                         "algo_bytes_per_launch": kv_bytes},
            "gpu_launches": 2 * args.steps, "clocks": clk.summary()}  # split + combine per call


# ---------------------------------------------------------------------------
# Decode workloads: the synthetic Llama shapes, one token per step
def gemv_plan(spec, skip=None):
    """The quant-GEMV launches of one decode step, in order: (fmt, [(W, rows)], cols, x-tag, norm-tag, kind)."""
    plan = []
    for li in range(spec.n_layers):
        if skip is not None and skip[li]:
            continue
        f = spec.fmt
        by = {}
        for t in ("wq", "wk", "wv"):
            by.setdefault(f[t], []).append(t)
        for fm, ts in by.items():
            plan.append((fm, [(li, t) for t in ts], spec.d_model, "x", ("attn_norm", li), "plain"))
        plan.append((f["wo"], [(li, "wo")], spec.n_qh * spec.head_dim, "ao", None, "resid"))
        plan.append((f["wg"], [(li, "wg"), (li, "wu")], spec.d_model, "x", ("ffn_norm", li), "swiglu"))
        plan.append((f["wd"], [(li, "wd")], spec.ffn, "h", None, "resid"))
    plan.append((spec.fmt["out"], [(-1, "out")], spec.d_model, "x", ("out_norm", -1), "plain"))
    return plan


def gemm_launches(fmt, cols, normed):
    """Kernel launches of one verify GEMM: the GEMM and its epilogue, plus the
    RMSNorm scalars' kernel when a normed launch takes the tensor-core form
    (Q8_0 / Q4_K / Q6_K rows of a multiple of 16 bytes)."""
    import synth
    wide = (os.environ.get("NT_GEMM_MMA", "1") != "0" and fmt in (synth.Q8_0, synth.Q4_K, synth.Q6_K)
            and synth.row_bytes(fmt, cols) % 16 == 0)
    return 2 + (1 if normed and wide else 0)


def verify_layer_launches(spec):
    """Launches of one layer of a verify (or prefill) pass: the Q/K/V GEMMs (one
    per format), attention (split, combine), O, gate/up and down."""
    nq = spec.n_qh * spec.head_dim
    qkv = sum(gemm_launches(f, spec.d_model, True) for f in {spec.fmt[t] for t in ("wq", "wk", "wv")})
    return (qkv + 2 + gemm_launches(spec.fmt["wo"], nq, False) + gemm_launches(spec.fmt["wg"], spec.d_model, True)
            + gemm_launches(spec.fmt["wd"], spec.ffn, False))


def bench_prefill(args, rank, world):
    """<model>_prefill<N>: one N-token prompt through nt_prefill (chunks of 16
    tokens, or 8, through the verify GEMMs), repeated; tokens/s of prompt."""
    import torch

    import synth
    from block_quantized_gemv_nt_gb300 import engine, nt

    base, n = args.workload.rsplit("_prefill", 1)
    n = int(n)
    spec = synth.model_spec(base)
    hm = synth.make_host_model(spec)
    ctx = nt.Context(torch.cuda.current_device())
    gm = engine.DeviceModel(ctx, spec, hm)
    raw = synth.random_bytes(4 * n, seed=spec.seed, stream=777).view(np.uint32)
    prompt = (raw % spec.vocab).astype(np.int32)
    pos0 = max(0, min(spec.n_prefill, spec.kv_cap - n))
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(max(1, min(args.warmup, 2))):
            gm.prefill(prompt, pos0, stream=st)
        st.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            clk.wait_first()
            clk.mark_start()
            e0.record(st)
            for _ in range(args.steps):
                gm.prefill(prompt, pos0, stream=st)
            e1.record(st)
            e1.synchronize()
            clk.mark_end()
            clk.wait_one_more()
    ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    chunk = nt.nt_model_prefill_chunk(ctx, gm.handle)
    chunks = -(-n // chunk)
    wbytes = spec.layer_bytes() * spec.n_layers
    gbs = chunks * wbytes / (ms / 1e3) / 1e9
    peak, kind = measured_peaks()
    # e2e: the prompt from host memory (read by the call), the last logits back to pinned host memory
    out_h = torch.empty(spec.vocab, dtype=torch.float32).pin_memory()
    n_e2e = max(1, min(args.steps, 3))
    with torch.cuda.stream(st):
        st.synchronize()
        h0 = time.perf_counter()
        for _ in range(n_e2e):
            lg = gm.prefill(prompt, pos0, stream=st)
            out_h.copy_(lg, non_blocking=True)
            st.synchronize()
        e2e_s = max_over_ranks((time.perf_counter() - h0) / n_e2e, world)
    ctx.sync()
    gm.close()
    # launches per prompt: per chunk its setup, the embedding rows and the layers; after the last chunk the
    # LM head, the state update and the argmax
    launches = (chunks * (2 + spec.n_layers * verify_layer_launches(spec))
                + gemm_launches(spec.fmt["out"], spec.d_model, True) + 2)
    return {"metric": METRIC, "value": round(n / (ms / 1e3) * world, 2), "unit": "prompt tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (block-quantized weights, f16 KV)",
            "data": "synthetic: random weights of the named shape, seeded", "impl": "ours",
            "config": {"workload": args.workload, "prompt_tokens": n, "chunk_tokens": chunk, "chunks": chunks,
                       "pos0": pos0,
                       "l2": f"inputs larger than L2 ({wbytes / 1e9:.2f} GB of weights per chunk)"},
            "roofline": {"bound": "hbm", "kernel": f"qgemm (M <= {chunk}; issue-bound, far from the HBM bound)",
                         "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "peak_kind": kind, "traffic": None,
                         "algo_bytes_per_launch": wbytes},
            "e2e": {"value": round(n / e2e_s * world, 2), "unit": "prompt tok/s", "h2d_bytes_per_step": 4 * n,
                    "d2h_bytes_per_step": 4 * spec.vocab},
            "gpu_launches": args.steps * launches, "clocks": clk.summary()}


SAMPLER = (0.8, 0.9)  # temperature, top-p of the "_sample" workloads

# The pages' own decode throughput for a workload, where they print one: Llama
# 8B Q8_0 with custom CUDA kernels on an RTX 3090 ("Ntransformer",
# en.unwiki.net, roadmap: phase 1).  Another machine's number, so vs_baseline
# is context, not a target.
PAGE_TOK_S = {"llama8b_q8_0": 48.9}


def decode_kernels_per_step(spec, n_exec, sampled=False):
    """Kernel launches of one decode step: the embedding row and the LM head;
    per executed layer one Q/K/V GEMV per distinct format, attention (split,
    combine), O, gate/up and down; then the argmax, or the six sampler
    launches."""
    return 2 + n_exec * (5 + len({spec.fmt[t] for t in ("wq", "wk", "wv")})) + (6 if sampled else 1)


def parse_decode(name):
    """<model>[_skip<N>][_spec<K>][_sample][_file]: a synthetic model, optionally
    decoding with the N layers of highest calibration cosine skipped, or
    self-speculatively with K drafted tokens per step; "_sample" draws tokens
    with the sampler (SAMPLER) instead of the argmax (speculative sampling
    with _spec); "_file" streams a streamed model's layers from a model file
    (bench_streamed).  Returns (spec, n_skip, k, sampled)."""
    import synth
    n_skip = k = 0
    if name.endswith("_file"):
        name = name[:-len("_file")]
    sampled = name.endswith("_sample")
    if sampled:
        name = name[:-len("_sample")]
    if "_spec" in name:
        name, n = name.rsplit("_spec", 1)
        k = int(n)
    if "_skip" in name:
        name, n = name.rsplit("_skip", 1)
        n_skip = int(n)
    return synth.model_spec(name), n_skip, k, sampled


def bench_decode(args, rank, world):
    import torch

    import synth
    from block_quantized_gemv_nt_gb300 import engine, nt

    spec, n_skip, _, sampled = parse_decode(args.workload)
    t0 = time.perf_counter()
    hm = synth.make_host_model(spec)
    t_gen = time.perf_counter() - t0
    ctx = nt.Context(torch.cuda.current_device())
    gm = engine.DeviceModel(ctx, spec, hm)
    if sampled:
        gm.set_sampler(*SAMPLER, seed=spec.seed)
    st = torch.cuda.Stream()
    P = spec.n_prefill
    window = spec.n_gen
    skip = None
    with torch.cuda.stream(st):
        if n_skip:
            # calibration on the first token (all layers run), then the mask is frozen
            skip, _ = gm.calibrate(spec.first_token, P, n_skip, stream=st)
        gm.step(spec.first_token, P, skip, stream=st)
        for _ in range(max(3, args.warmup) - 1):
            gm.step(-1, 0, skip, stream=st)
        st.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            clk.wait_first()
            torch.cuda.synchronize()
            clk.mark_start()
            e0.record(st)
            for i in range(args.steps):
                if i % window == 0:
                    gm.step(spec.first_token, P, skip, stream=st)  # restart the generation window
                else:
                    gm.step(-1, 0, skip, stream=st)
            e1.record(st)
            e1.synchronize()
            clk.mark_end()
            clk.wait_one_more()
        ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    tok_s = args.steps / (ms / 1e3)

    # the step's quant-GEMV launches, same arguments, timed on their own (dominant kernel)
    plan = gemv_plan(spec, skip)
    W = lambda li, t: gm.out if li < 0 else gm.layers[li][t]  # noqa: E731
    norm = lambda tag: None if tag is None else (gm.out_norm if tag[1] < 0 else gm.layers[tag[1]][tag[0]])  # noqa
    xbuf = {"x": torch.randn(spec.d_model, device="cuda"), "ao": torch.randn(spec.n_qh * spec.head_dim, device="cuda"),
            "h": torch.randn(spec.ffn, device="cuda") * 0.01}
    ybuf = torch.empty(max(spec.vocab, 3 * spec.ffn), device="cuda")
    algo = 0
    for fm, ws, cols, xt, nt_, kind in plan:
        for li, t in ws:
            algo += W(li, t).numel()
        algo += 4 * cols
    rows_out = sum(sum(W(li, t).shape[0] for li, t in ws) // (2 if kind == "swiglu" else 1) for _, ws, *_r in plan)
    algo += 4 * rows_out

    def run_plan():
        for fm, ws, cols, xt, ntag, kind in plan:
            g = norm(ntag)
            if kind == "swiglu":
                (li, tg), (_, tu) = ws
                nt.nt_gemv_q_swiglu(ctx, fm, W(li, tg), W(li, tu), xbuf[xt], ybuf, W(li, tg).shape[0], cols,
                                    norm_g=g, eps=spec.eps, stream=st)
            else:
                jobs, off = [], 0
                for li, t in ws:
                    r = W(li, t).shape[0]
                    jobs.append((W(li, t), ybuf[off:], ybuf[off:] if kind == "resid" else None, r))
                    off += ((r + 63) // 64) * 64
                nt.nt_gemv_q_multi(ctx, fm, jobs, xbuf[xt], cols, norm_g=g, eps=spec.eps, stream=st)

    with torch.cuda.stream(st):
        run_plan()
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            run_plan()
        g.replay()
        st.synchronize()
        k_reps = max(1, min(args.steps, 32))
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(st)
        for _ in range(k_reps):
            g.replay()
        f1.record(st)
        f1.synchronize()
    gemv_ms = f0.elapsed_time(f1) / k_reps
    n_launch = len(plan)
    gemv_gbs = algo / (gemv_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()

    # e2e: host-driven loop through the C ABI: token in by value, logits + next token back to pinned host
    logits_h = torch.empty(spec.vocab, dtype=torch.float32).pin_memory()
    tok_h = torch.empty(1, dtype=torch.int32).pin_memory()
    n_e2e = min(args.steps, window)
    with torch.cuda.stream(st):
        tok, pos = spec.first_token, P
        st.synchronize()
        h0 = time.perf_counter()
        for i in range(n_e2e):
            gm.step(tok, pos, skip, stream=st)
            logits_h.copy_(gm.logits, non_blocking=True)
            tok_h.copy_(gm.next_token, non_blocking=True)
            st.synchronize()
            tok, pos = int(tok_h[0]), pos + 1
        e2e_s = (time.perf_counter() - h0) / n_e2e
    e2e_s = max_over_ranks(e2e_s, world)
    ctx.sync()

    per_step_bytes = step_bytes(spec, skip)
    n_exec = spec.n_layers - (int(np.sum(skip)) if skip is not None else 0)
    kernels_per_step = decode_kernels_per_step(spec, n_exec, sampled)
    page = PAGE_TOK_S.get(args.workload)
    line = {
        "metric": METRIC, "value": round(tok_s * world, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": round(tok_s * world / page, 3) if page else None,
        "dtype": "f32 (block-quantized weights, f16 KV)",
        "data": "synthetic: random weights of the named shape, seeded", "impl": "ours",
        "config": {"workload": args.workload, "layers": spec.n_layers, "layers_executed": n_exec,
                   "d_model": spec.d_model, "ffn": spec.ffn,
                   "vocab": spec.vocab, "kv_prefill": P, "batch": 1, "seed": spec.seed,
                   "weights": {k: synth.FMT_NAMES[v] for k, v in spec.fmt.items()},
                   "decode": "sampled (temperature %g, top-p %g)" % SAMPLER if sampled else "greedy",
                   "l2": f"inputs larger than L2 ({per_step_bytes / 1e9:.2f} GB read per token)",
                   "step_bytes": per_step_bytes,
                   "step_hbm_gbs": round(per_step_bytes * tok_s / 1e9, 1),
                   "step_frac_of_peak": round(per_step_bytes * tok_s / 1e9 / peak, 4)},
        "roofline": {"bound": "hbm", "kernel": "qgemv", "achieved": round(gemv_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gemv_gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": profile_traffic("qgemv", args.workload),
                     "algo_bytes_per_launch": int(algo / n_launch), "launches_per_step": n_launch,
                     "avg_launch_us": round(gemv_ms * 1e3 / n_launch, 3)},
        "e2e": {"value": round(1.0 / e2e_s, 2), "unit": "tok/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4 * spec.vocab + 4},
        "gpu_launches": args.steps * kernels_per_step + (args.steps + window - 1) // window,
        "clocks": clk.summary(),
        "host_generation_s": round(t_gen, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_decode(spec, hm, budget_s=args.cpu_budget, skip=skip)
    gm.close()
    return line


def h2d_peak(src, nbytes, reps=5):
    """Best pinned host -> HBM copy bandwidth (GB/s) of one nbytes copy."""
    import torch
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            e0.record(st)
            dst.copy_(src[:nbytes], non_blocking=True)
            e1.record(st)
        e1.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del dst
    return best


def bench_streamed(args, rank, world):
    """Decode of a model whose layers n_resident.. stream from page-locked
    host memory each pass; greedy, or self-speculative with k drafts (the
    resident layers draft, all layers verify)."""
    import torch

    import synth
    from block_quantized_gemv_nt_gb300 import engine, nt

    spec, n_skip, k, sampled = parse_decode(args.workload)
    assert n_skip == 0, "layer skip is not combined with streaming here"
    from_file = args.workload.endswith("_file")
    t0 = time.perf_counter()
    blobs = engine.HostBlobs(spec)
    hm = synth.make_host_model(spec, out_view=blobs.view)
    t_gen = time.perf_counter() - t0
    ctx = nt.Context(torch.cuda.current_device())
    mf = fpath = None
    ram_blobs = blobs  # the pinned-RAM copy of the streamed layers: also the copy-peak reference
    if from_file:
        # the host-file tier: the model written to a file (RAM-backed /dev/shm when present), its
        # streamed layers page-locked in the mapping where the OS allows, else copied once
        from block_quantized_gemv_nt_gb300 import modelfile
        fdir = "/dev/shm" if os.path.isdir("/dev/shm") else tempfile.gettempdir()
        fpath = os.path.join(fdir, f"nt_bench_{os.getpid()}_{rank}.ntq")
        atexit.register(lambda p=fpath: os.path.exists(p) and os.unlink(p))  # removed however the run ends
        modelfile.write_model(fpath, spec, hm)
        mf = modelfile.ModelFile(fpath)
        hm = synth.HostModel(mf.spec, mf.layers, mf.embd, mf.out, mf.out_norm, hm.kcache, hm.vcache)
        blobs = modelfile.FileBlobs(ctx, mf, spec.n_resident)
    slots = args.stream_slots
    if slots <= 0:
        # greedy: double buffering (per-layer compute is far below a layer copy);
        # speculative: as many slots as the weight cap allows (2..8), so copies
        # run ahead during the drafts and the resident part of the verify pass
        r, c = spec.tensor_shape("out")
        fixed = spec.n_resident * spec.layer_bytes() + r * synth.row_bytes(spec.fmt["out"], c)
        slots = int(max(2, min(8, (args.hbm_weight_cap * 1e9 - fixed) // blobs.nbytes))) if k else 2
    gm = engine.DeviceModel(ctx, mf.spec if from_file else spec, hm, blobs=blobs, stream_slots=slots)
    if sampled:
        gm.set_sampler(*SAMPLER, seed=spec.seed)
    st = torch.cuda.Stream()
    P = spec.n_prefill
    n_streamed = len(blobs.layers)
    # one step emits up to k + 1 tokens: restart the window before the KV capacity runs out
    window = max(1, spec.n_gen // (k + 1)) if k else spec.n_gen
    counts = torch.zeros(max(1, args.steps), dtype=torch.int32, device="cuda")

    def one(i, timed):
        first = i % window == 0
        if k:
            _, cnt, _ = gm.spec_step(spec.first_token if first else -1, P, k, stream=st)
            if timed:
                counts[i:i + 1].copy_(cnt, non_blocking=True)
        else:
            gm.step(spec.first_token if first else -1, P, stream=st)

    with torch.cuda.stream(st):
        for i in range(max(3, args.warmup)):
            one(i, False)
        st.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            clk.wait_first()
            torch.cuda.synchronize()
            clk.mark_start()
            e0.record(st)
            for i in range(args.steps):
                one(i, True)
            e1.record(st)
            e1.synchronize()
            clk.mark_end()
            clk.wait_one_more()
        ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    n_tok = int(counts[:args.steps].sum().item()) if k else args.steps
    tok_s = n_tok / (ms / 1e3)
    pass_s = ms / 1e3 / args.steps
    link_bytes = n_streamed * blobs.nbytes          # host -> HBM bytes of one pass
    b_h2d = h2d_peak(ram_blobs.blob[ram_blobs.layers[0]], ram_blobs.nbytes)
    link_gbs = link_bytes / pass_s / 1e9

    # e2e: host-driven loop through the C ABI, results back to pinned host memory each step
    n_e2e = min(args.steps, 4)
    out_h = torch.empty(spec.vocab, dtype=torch.float32).pin_memory()
    tok_h = torch.empty(8, dtype=torch.int32).pin_memory()
    cnt_h = torch.empty(1, dtype=torch.int32).pin_memory()
    with torch.cuda.stream(st):
        st.synchronize()
        tok, pos, got = spec.first_token, P, 0
        h0 = time.perf_counter()
        for i in range(n_e2e):
            if k:
                toks, cnt, _ = gm.spec_step(tok, pos, k, stream=st)
                tok_h.copy_(toks, non_blocking=True)
                cnt_h.copy_(cnt, non_blocking=True)
                st.synchronize()
                n = int(cnt_h[0])
                tok, pos, got = int(tok_h[n - 1]), pos + n, got + n
            else:
                gm.step(tok, pos, stream=st)
                out_h.copy_(gm.logits, non_blocking=True)
                tok_h[:1].copy_(gm.next_token, non_blocking=True)
                st.synchronize()
                tok, pos, got = int(tok_h[0]), pos + 1, got + 1
        e2e_s = time.perf_counter() - h0
    e2e_tok_s = got / max_over_ranks(e2e_s, world)
    ctx.sync()
    hbm_w = gm.hbm_weight_bytes()
    peak, peak_kind = measured_peaks()
    per_pass = n_tok / args.steps
    line = {
        "metric": METRIC, "value": round(tok_s * world, 3), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(pass_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (block-quantized weights, f16 KV)",
        "data": "synthetic: random weights of the named shape, seeded", "impl": "ours",
        "config": {"workload": args.workload, "layers": spec.n_layers, "resident_layers": spec.n_resident,
                   "streamed_layers": n_streamed, "stream_slots": gm.n_slots, "layer_blob_bytes": blobs.nbytes,
                   "hbm_weight_bytes": hbm_w, "hbm_weight_cap_gb": args.hbm_weight_cap, "d_model": spec.d_model, "ffn": spec.ffn, "vocab": spec.vocab,
                   "kv_prefill": P, "batch": 1, "seed": spec.seed,
                   "weights": {kk: synth.FMT_NAMES[v] for kk, v in spec.fmt.items()},
                   "decode": (f"self-speculative, k={k} drafts by the resident layers" if k else "greedy")
                   + (", sampled (temperature %g, top-p %g)" % SAMPLER if sampled else ""),
                   "tokens_per_pass": round(per_pass, 3),
                   "draft_acceptance": round((per_pass - 1) / k, 4) if k else None,
                   "l2": f"inputs larger than L2 ({link_bytes / 1e9:.1f} GB streamed per pass)"},
        "roofline": {"bound": "h2d", "kernel": "host-to-HBM layer copies", "achieved": round(link_gbs, 1),
                     "peak": round(b_h2d, 1), "unit": "GB/s", "frac": round(link_gbs / b_h2d, 4),
                     "peak_kind": "measured in this run: best pinned copy of one layer blob",
                     "traffic": None, "algo_bytes_per_launch": link_bytes, "hbm_peak": peak},
        "e2e": {"value": round(e2e_tok_s, 3), "unit": "tok/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4 * (k + 2) if k else 4 * spec.vocab + 4},
        "gpu_launches": None,
        "clocks": clk.summary(),
        "host_generation_s": round(t_gen, 1),
    }
    n_exec = spec.n_layers
    per_layer = 5 + len({spec.fmt[t] for t in ("wq", "wk", "wv")})  # Q/K/V, attention (2), O, gate/up, down
    if k:
        # per pass: setup, k drafts (resident layers), verify (GEMM + epilogue per GEMV, attention), accept
        n_res = spec.n_resident
        draft = 2 + n_res * per_layer + (6 if sampled else 1)
        verify = (1 + n_exec * verify_layer_launches(spec) + gemm_launches(spec.fmt["out"], spec.d_model, True)
                  + (6 if sampled else k + 1))
        line["gpu_launches"] = args.steps * (2 + k * draft + verify)
    else:
        line["gpu_launches"] = (args.steps * (2 + n_exec * per_layer + (6 if sampled else 1))
                                + (args.steps + window - 1) // window)
    if from_file:
        rungs = {}
        for r in blobs.rung_of.values():
            rungs[r] = rungs.get(r, 0) + 1
        line["config"]["host_source"] = {"model_file": fpath, "tier": blobs.tier, "ranges_by_rung": rungs}
        line["roofline"]["peak_kind"] = "measured in this run: best pinned-RAM copy of one layer blob"
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_decode(spec, hm, budget_s=args.cpu_budget)
    gm.close()
    if from_file:
        blobs.close()
        mf.close()
        os.unlink(fpath)
    return line


def step_bytes(spec, skip=None):
    """Algorithmic HBM bytes of one decode token: every executed weight byte once,
    the KV cache of the executed layers read (mean context of the window) and
    written, activations ignored (they stay in L2)."""
    import synth
    n_exec = spec.n_layers - (int(np.sum(skip)) if skip is not None else 0)
    w = spec.layer_bytes() * n_exec
    r, c = spec.tensor_shape("out")
    w += r * synth.row_bytes(spec.fmt["out"], c)
    w += synth.row_bytes(spec.fmt["embd"], spec.d_model)
    ctxlen = spec.n_prefill + spec.n_gen / 2
    kv = n_exec * 2 * spec.n_kvh * spec.head_dim * 2 * (ctxlen + 1)
    return int(w + kv)


def cpu_decode(spec, hm, budget_s=15.0, skip=None):
    import oracle
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    tok, pos, n = spec.first_token, spec.n_prefill, 0
    t0 = time.perf_counter()
    while n == 0 or time.perf_counter() - t0 < budget_s:
        logits = om.step(tok, pos, skip)
        tok, pos, n = int(np.argmax(logits)), pos + 1, n + 1
    dt = time.perf_counter() - t0
    what = "the full model" if skip is None else f"the model with {int(np.sum(skip))} layers skipped"
    return {"value": round(n / dt, 4), "unit": "tok/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} greedy oracle decode step{'' if n == 1 else 's'} of {what} in {dt:.1f} s"}


# ---------------------------------------------------------------------------
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The largest of every rank's v (the slowest rank's time); the tensor
    lives where the process group's backend reduces (GPU for NCCL)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reference_arm(args, rank, world):
    """The oracle, as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    import synth
    if args.workload.startswith("gem"):
        fmt, rows, cols, M = parse_gemv(args.workload)
        seed = 0 if (fmt == synth.Q8_0 and rows == 4096 and cols == 4096) else 100 + fmt
        W = synth.quant_matrix(fmt, rows, cols, seed=seed, stream=0)
        X = synth.normal_f32(M * cols, seed=seed, stream=1).reshape(M, cols).astype(np.float64)
        algo = W.nbytes + 4 * M * (cols + rows)
        import oracle
        for _ in range(max(1, min(args.warmup, 2))):
            oracle.gemv(fmt, W, X[0], rows, cols)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            for xv in X:
                oracle.gemv(fmt, W, xv, rows, cols)
        dt = (time.perf_counter() - t0) / args.steps
        v = round(algo / dt / 1e9, 3)
        return {"metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic seeded blocks",
                "impl": "reference", "config": {"workload": args.workload},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                                 "sample": f"{args.steps} full oracle GEMVs"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if args.workload.startswith("attn_"):
        import oracle
        H, G, P = (int(v) for v in args.workload.split("_")[1].split("x"))
        hd = 128
        K = synth.normal_f16(G * P * hd, 5, 1)
        V = synth.normal_f16(G * P * hd, 5, 2)
        q = synth.normal_f32(H * hd, 5, 3).astype(np.float64)
        kv_bytes = 2 * G * P * hd * 2
        oracle.attn_decode(q, K, V, H, G, hd, P, P)
        n = max(1, min(args.steps, args.ref_max_steps))
        t0 = time.perf_counter()
        for _ in range(n):
            oracle.attn_decode(q, K, V, H, G, hd, P, P)
        dt = (time.perf_counter() - t0) / n
        v = round(kv_bytes / dt / 1e9, 3)
        return {"metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": n,
                "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic N(0,1) KV",
                "impl": "reference", "config": {"workload": args.workload},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                                 "sample": f"{n} full oracle attention calls"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    prefill_n, sampled = 0, False
    if "_prefill" in args.workload:
        base, n = args.workload.rsplit("_prefill", 1)
        spec, n_skip, prefill_n = synth.model_spec(base), 0, int(n)
    else:
        spec, n_skip, _, sampled = parse_decode(args.workload)
    hm = synth.make_host_model(spec)
    import oracle
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, hm.kcache, hm.vcache)
    tok, pos = spec.first_token, spec.n_prefill
    skip = None
    if n_skip:
        # calibration step (all layers), then the frozen mask
        _, cos_l = om.step(tok, pos, want_cos=True)
        skip = oracle.layer_skip_select(cos_l, n_skip)
    for _ in range(max(0, min(args.warmup, 1))):
        om.step(tok, pos, skip)
    t0 = time.perf_counter()
    n = max(1, min(args.steps, args.ref_max_steps))
    for _ in range(n):
        logits = om.step(tok, pos, skip)
        # a prompt is fed token by token (teacher-forced); decoding feeds back the argmax
        if prefill_n:
            nxt = (tok * 7 + 3) % spec.vocab
        elif sampled:
            nxt = oracle.sample(logits, *SAMPLER, oracle.sample_uniform(spec.seed, pos))[0]
        else:
            nxt = int(np.argmax(logits))
        tok, pos = nxt, pos + 1
    dt = (time.perf_counter() - t0) / n
    v = round(1.0 / dt, 4)
    unit = "prompt tok/s" if prefill_n else "tok/s"
    what = ("prompt tokens fed to the oracle one by one" if prefill_n else
            "sampled oracle decode steps" if sampled else "greedy oracle decode steps")
    return {"metric": METRIC, "value": v, "unit": unit, "n_gpus": world, "steps": n, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 1), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic: random weights of the named shape, seeded", "impl": "reference",
            "config": {"workload": args.workload, "batch": 1},
            "cpu_baseline": {"value": v, "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{n} {what} (bounded sample of the workload)"},
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama8b_q8_0")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-max-steps", type=int, default=8, help="oracle steps per reference-arm run")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stream-slots", type=int, default=0,
                    help="HBM slots for streamed layers (0: 2 for greedy decoding; for speculative decoding as "
                         "many as --hbm-weight-cap allows, 2..8)")
    ap.add_argument("--hbm-weight-cap", type=float, default=24.0, help="GB of HBM for weights, streamed models")
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
    if args.workload.startswith("gemv") or args.workload.startswith("gemm"):
        line = bench_gemv(args, rank, world)
    elif args.workload.startswith("attn"):
        line = bench_attn(args, rank, world)
    elif "_prefill" in args.workload:
        line = bench_prefill(args, rank, world)
    elif parse_decode(args.workload)[0].n_resident >= 0:
        line = bench_streamed(args, rank, world)
    else:
        line = bench_decode(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
