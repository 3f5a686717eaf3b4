#!/usr/bin/env python
"""Benchmark of the WhiteMatter cross-layer KV pool path on one B300.

One step is one whole prefill of a batch: a zeroed k-channel cache, three
cyclic Gauss-Seidel passes with g = 16 over B x T tokens (the cache updated
after every group), and the last-position logits in the final pass, all
through the C ABI (``wm_cyclic_pass``). The default workload is the 1.3B-scale
half-cache model (L=28, D=1792, k=14, p=2, Hq=14, Hkv=2, d=128, F=4608,
V=151936) at B=64, T=2048. After the timed steps, 256 decode steps of that
model run from the prefilled cache (Tmax = 2304) and are reported as
``decode``: replayed from one CUDA graph of ``wm_decode_batch`` (positions on
the device), with the direct ``wm_decode_step`` calls as ``decode.eager``.
Inputs are seeded and synthetic; weights are N(0, 0.02) with unit norm gains.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--kernel mixer|attention`` instead times one kernel of the path alone, through
the C ABI (``wm_pool_mix`` on ``--rows`` token rows of the 1.3B pool, or
``wm_channel_attn`` on one prefill group of ``--batch`` sequences), and prints
one JSON line with its CUDA-event time and roofline fraction; the profiles
under profiles/ capture these invocations.

``--kernel decode`` times one decode step (``wm_decode_batch``, 64 sequences at
position 2048) against the bytes it must move. ``--sweep convergence`` runs
the fixed-point residual per pass of the prefill schedules g in {1, 4, 16, 64}
on the full-cache small model. ``--workload half_small|full_small|tiny_fp32``
runs the other configurations through the same step.

Under torchrun each rank runs an independent replica on its own GPU (the
path has no exchange step); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from cross_layer_kv_pool_b300 import synth  # noqa: E402

METRIC = "prefill tok/s (3 cyclic passes, g=16) at 1.3B k=14"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
# DRAM bytes (read + written) per tcgen05 GEMM launch of the prefill step.
# None: the GEMM kernel gained its entry check of the flag word (control path
# only) after the last counter capture (98.5 MB per launch, launch-weighted
# over the 335 gemm_tc_kernel launches among the first 600 of the timed step),
# and a capture of the full-size step with DRAM counters holds more device
# memory than such captures may; set it again from a capture of the current
# kernel.
GEMM_DRAM_BYTES_PER_LAUNCH = None
GEMM_DRAM_SOURCE = ("null: the kernel changed (entry flag check) after the last DRAM counter "
                    "capture of the full-size step, which is not repeated at that size")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_1p3b",
                    choices=["prefill_1p3b", "half_small", "full_small", "tiny_fp32"])
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the tiny / half-small / full-small prefill lines")
    ap.add_argument("--k", type=int, default=None, help="override the channel count k")
    ap.add_argument("--kernel", choices=["mixer", "attention", "pool_backward", "decode"],
                    default=None,
                    help="time one kernel of the path alone (1.3B shapes)")
    ap.add_argument("--rows", type=int, default=8192, help="--kernel mixer: token rows")
    ap.add_argument("--seqs", type=int, default=None,
                    help="sequences of the prefill workload (default: the workload's own; "
                         "a smaller count gives the small case a profiler captures)")
    ap.add_argument("--batch", type=int, default=64, help="--kernel attention: sequences")
    ap.add_argument("--group", type=int, default=15, help="--kernel attention: group index q")
    ap.add_argument("--sweep", choices=["convergence"], default=None,
                    help="fixed-point residual per pass for g in {1, 4, 16, 64} (full-small model)")
    ap.add_argument("--passes", type=int, default=32, help="--sweep convergence: passes per g")
    ap.add_argument("--variant", choices=["feedback_free"], default=None,
                    help="time the feedback-free variant (k = L, one pass) at the workload's shape")
    ap.add_argument("--chunk", type=int, default=8,
                    help="--variant feedback_free: sequences per workspace chunk")
    return ap.parse_args()


def workload(args):
    wl = dict(synth.WORKLOADS[args.workload])
    if args.k is not None:
        wl["shape"] = wl["shape"].replace(k=args.k)
    if getattr(args, "seqs", None):
        wl["B"] = args.seqs
    return wl


def peaks():
    try:
        with open(PEAKS_PATH) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_weights(shape, seed: int = 0):
    W = synth.make_weights(shape, seed=seed, device="cpu")
    return {n: t.float().numpy() for n, t in W.items()}


def cpu_sample(shape, rows: int, Wn, seed: int = 0):
    """Time the CPU oracle on ``rows`` token rows of one cyclic group: the
    layer stack plus the pool, against a cache of the workload's length.
    Returns (seconds, rows, threads)."""
    import oracle.whitematter as O
    from types import SimpleNamespace
    import dataclasses
    oc = SimpleNamespace(**dataclasses.asdict(shape))
    oc.storage = "bf16"
    T, g = 2048, 16
    q = g - 1
    # rows spread over the sequence (first and last of the group, then the
    # middle), so that the sample's attention sees ~T/2 keys on average
    allp = np.arange(q, T, g)
    pick = np.unique(np.linspace(0, len(allp) - 1, rows).round().astype(int))
    pos = allp[pick]
    rows = len(pos)
    toks = np.random.default_rng(seed).integers(0, shape.V, size=rows)
    ck, cv = O.new_cache(oc, 1, T)
    threads = torch.get_num_threads()
    t0 = time.perf_counter()
    O.run_rows(oc, Wn, toks, np.zeros(rows, dtype=np.int64), pos, ck, cv, want_logits=False)
    return time.perf_counter() - t0, rows, threads


def cpu_decode_record(shape, pos: int, Tmax: int):
    """The CPU oracle on one decode step of one sequence at ``pos`` (stack,
    LM head and pool against a zero cache of Tmax positions)."""
    import oracle.whitematter as O
    from types import SimpleNamespace
    import dataclasses
    oc = SimpleNamespace(**dataclasses.asdict(shape))
    oc.storage = "bf16"
    Wn = oracle_weights(shape)
    ck, cv = O.new_cache(oc, 1, Tmax)
    tok = np.random.default_rng(0).integers(0, shape.V, size=1)
    threads = torch.get_num_threads()
    t0 = time.perf_counter()
    O.decode_batch(oc, Wn, tok, np.array([pos]), ck, cv)
    secs = time.perf_counter() - t0
    return {"value": 1.0 / secs, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": f"one decode step of one sequence at position {pos} (fp64 NumPy, {secs:.1f} s)"}


def cpu_baseline_record(shape, passes: int, rows: int):
    secs, n, threads = cpu_sample(shape, rows, oracle_weights(shape))
    tok_s = n / secs / passes
    return {"value": tok_s, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": (f"{n} token rows of one cyclic group (positions 15 and 2047 of a "
                       f"2048-token sequence) through the {shape.L}-layer stack and the pool, "
                       f"fp64 NumPy, {secs:.1f} s; tok/s = rows / time / {passes} passes")}


def run_reference(args, ws, rank):
    """The CPU oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    wl = workload(args)
    shape = wl["shape"]
    rows = 2
    samples = []
    Wn = oracle_weights(shape)
    for i in range(args.warmup + args.steps):
        secs, n, threads = cpu_sample(shape, rows, Wn, seed=i)
        if i >= args.warmup:
            samples.append(n / secs / wl["passes"])
    value = statistics.mean(samples)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * rows / (value * wl["passes"]),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_dict(args, wl),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step {rows} token rows of one cyclic group through the "
                                   f"{shape.L}-layer stack and pool (fp64 NumPy), extrapolated "
                                   f"to {wl['passes']} passes"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(args, wl):
    s = wl["shape"]
    return {"workload": f"{args.workload}: 3 cyclic passes g={wl['g']} + last-position logits",
            "L": s.L, "D": s.D, "k": s.k, "p": s.p, "Hq": s.Hq, "Hkv": s.Hkv, "d": s.d,
            "F": s.F, "V": s.V, "global_batch": wl["B"] * args.gpus, "seq_len": wl["T"],
            "g": wl["g"], "passes": wl["passes"], "parallelism": f"replicas x{args.gpus}",
            "l2": "inputs larger than L2 (weights 2.9 GB, 0.8 GB layer-state stash per group)"
                  if args.workload == "prefill_1p3b" else "inputs larger than L2"}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def run_ours(args, ws, rank, local):
    from cross_layer_kv_pool_b300 import wm

    wl = workload(args)
    s = wl["shape"]
    B, T, g, passes = wl["B"], wl["T"], wl["g"], wl["passes"]
    nd = args.decode_steps
    Tmax = T + nd
    dev = torch.device("cuda", torch.cuda.current_device())
    W = synth.make_weights(s, seed=0, device=dev)
    m = wm.Model(s, W)
    tok = synth.make_tokens(s, B, T, seed=1 + rank, device=dev)
    dec_tok = synth.make_tokens(s, B, max(nd, 1), seed=2 + rank, device=dev)
    ck, cv = m.new_cache(B, Tmax)
    wsp = m.workspace(max(wm.rows_for_pass(B, T, g), B), Tmax)
    lg = torch.empty((B, s.V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(tokens):
        ck.zero_()
        cv.zero_()
        for n in range(passes):
            last = n == passes - 1
            wm.wm_cyclic_pass(m, tokens, g, ck, cv, wsp, logits=lg if last else None,
                              logits_mode="last" if last else "none")

    for _ in range(args.warmup):
        step(tok)
    torch.cuda.synchronize()
    if wm.wm_check_flags(wsp) != 0:
        raise RuntimeError("device-side checks failed during warm-up")

    # ---- timed region: K steps; per-kernel events on three of them ----
    tracers = [wm.Tracer(wm.WM_TRACE_GEMM, 512), wm.Tracer(wm.WM_TRACE_MIX, 64),
               wm.Tracer(wm.WM_TRACE_ATTN, 256)]
    launches = wm.Tracer(wm.WM_TRACE_GEMM, 1)  # launch counting only
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    torch.cuda.nvtx.range_push("timed")   # lets a profiler select the timed steps
    for i in range(args.steps):
        tr = tracers[i] if i < len(tracers) else launches
        tr.attach(m)
        step(tok)
        wm.Tracer.detach(m)
    torch.cuda.nvtx.range_pop()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(ws)
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, ws)
    gpu_launches = int(sum(t.t.launches for t in tracers[:args.steps]) + launches.t.launches)
    value = ws * B * T / (ms / 1e3)

    # ---- end to end through the C ABI with host buffers ----
    tok_host = tok.cpu().pin_memory()
    lg_host = torch.empty((B, s.V), dtype=torch.float32).pin_memory()
    tok_dev = torch.empty_like(tok)
    for _ in range(max(1, args.warmup // 2)):
        tok_dev.copy_(tok_host, non_blocking=True)
        step(tok_dev)
        lg_host.copy_(lg, non_blocking=True)
    torch.cuda.synchronize()
    barrier(ws)
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(args.steps):
        tok_dev.copy_(tok_host, non_blocking=True)
        step(tok_dev)
        lg_host.copy_(lg, non_blocking=True)
    x1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(x0.elapsed_time(x1) / args.steps, ws)
    e2e = {"value": ws * B * T / (ms_e2e / 1e3), "unit": "tok/s",
           "h2d_bytes_per_step": tok_host.numel() * 4, "d2h_bytes_per_step": lg_host.numel() * 4}

    # ---- decode from the prefilled cache ----
    decode = None
    if nd > 0:
        dlg = torch.empty((B, s.V), dtype=torch.float32, device=dev)
        step(tok)
        for t in range(3):  # warm-up, overwritten below
            wm.wm_decode_step(m, dec_tok[:, t].contiguous(), T + t, ck, cv, dlg, wsp)
        cols = [dec_tok[:, t].contiguous() for t in range(nd)]
        torch.cuda.synchronize()
        barrier(ws)
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for t in range(nd):
            wm.wm_decode_step(m, cols[t], T + t, ck, cv, dlg, wsp)
        d1.record(stream)
        torch.cuda.synchronize()
        dms_eager = max_over_ranks(d0.elapsed_time(d1), ws)
        # The same steps replayed from one CUDA graph per step: the step's
        # tokens gathered on the device, wm_decode_batch (positions on the
        # device), then the position and step counters advanced, so that each
        # step is a single graph launch. The entries rewritten at
        # T .. T + nd - 1 get the values they already hold.
        dec_all = dec_tok[:, :nd].t().contiguous()
        tok_buf = torch.empty(B, dtype=torch.int32, device=dev)
        pos_buf = torch.full((B,), T, dtype=torch.int32, device=dev)
        step_idx = torch.zeros(1, dtype=torch.long, device=dev)

        def one_step():
            torch.index_select(dec_all, 0, step_idx, out=tok_buf.view(1, B))
            wm.wm_decode_batch(m, tok_buf, pos_buf, ck, cv, dlg, wsp)
            pos_buf.add_(1)
            step_idx.add_(1)

        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            one_step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_step()
        for _ in range(3):
            pos_buf.fill_(T)
            step_idx.zero_()
            graph.replay()
        pos_buf.fill_(T)
        step_idx.zero_()
        torch.cuda.synchronize()
        barrier(ws)
        d0.record(stream)
        for t in range(nd):
            graph.replay()
        d1.record(stream)
        torch.cuda.synchronize()
        dms = max_over_ranks(d0.elapsed_time(d1), ws)
        # per-kernel shares of one decode step (separate, traced steps)
        dtr = {}
        for kind, name in ((wm.WM_TRACE_GEMM, "gemm"), (wm.WM_TRACE_ATTN, "attention"),
                           (wm.WM_TRACE_MIX, "mixer")):
            tr = wm.Tracer(kind, 256)
            tr.attach(m)
            wm.wm_decode_step(m, cols[0], T, ck, cv, dlg, wsp)
            wm.Tracer.detach(m)
            torch.cuda.synchronize()
            res = tr.results()
            dtr[name] = {"launches": len(res), "total_ms": sum(r[0] for r in res),
                         "launches_per_step_traced": tr.t.launches}
            if kind == wm.WM_TRACE_GEMM:
                by = {}
                for ms_, w_ in res:
                    d_ = by.setdefault(f"{w_:.4g}", [0, 0.0])
                    d_[0] += 1
                    d_[1] += ms_
                dtr[name]["by_flops"] = {k: [v[0], v[1] / v[0]] for k, v in by.items()}
        cache_bytes = 2 * B * s.k * s.Hkv * Tmax * s.d * 2
        # bytes the steps must move, averaged over their positions T .. T + nd - 1
        step_bytes = sum(decode_step_bytes(s, B, T + t) for t in range(nd)) / nd
        hbm_peak = peaks()[0]["hbm_gbs"]
        decode = {"value": ws * B * nd / (dms / 1e3), "unit": "tok/s", "steps": nd, "batch": B,
                  "prefix": T, "ms_per_step": dms / nd, "replay": "cuda_graph",
                  "eager": {"value": ws * B * nd / (dms_eager / 1e3), "ms_per_step": dms_eager / nd},
                  "hbm": {"bytes_per_step": step_bytes, "achieved": step_bytes / (dms / nd) / 1e6,
                          "unit": "GB/s", "peak": hbm_peak,
                          "frac": step_bytes / (dms / nd) / 1e6 / hbm_peak,
                          "what": "weights once and the visible cache entries once per step, "
                                  "averaged over the steps' positions; peak = measured HBM copy"},
                  "peak_cache_bytes": cache_bytes,
                  "cache_bytes_L_channels": cache_bytes // s.k * s.L, "kernels": dtr}
        if rank == 0 and not args.no_cpu_baseline:
            decode["cpu_baseline"] = cpu_decode_record(s, T, Tmax)
    if wm.wm_check_flags(wsp) != 0:
        raise RuntimeError("device-side checks failed")

    # ---- per-kernel rooflines from the traced launches ----
    pk, pk_kind = peaks()

    def summarise(tr, unit):
        res = tr.results()
        if not res:
            return None
        tot_ms = sum(r[0] for r in res)
        tot_w = sum(r[1] for r in res)
        return {"launches": len(res), "avg_ms": tot_ms / len(res), "work_per_launch": tot_w / len(res),
                "achieved": tot_w / (tot_ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)}

    gemm = summarise(tracers[0], "TFLOP/s") if args.steps >= 1 else None
    shapes = {}
    for ms_, w_ in tracers[0].results():
        d = shapes.setdefault(f"{w_:.4g}", [0, 0.0])
        d[0] += 1
        d[1] += ms_
    gemm_shapes = {k: {"launches": v[0], "avg_ms": v[1] / v[0],
                       "tflops": float(k) / (v[1] / v[0] / 1e3) / 1e12} for k, v in shapes.items()}
    mix = summarise(tracers[1], "GB/s") if args.steps >= 2 else None
    attn = summarise(tracers[2], "TFLOP/s") if args.steps >= 3 else None
    tc_peak = pk.get("bf16_tflops_sustained", 1400.0)
    roofline = None
    if gemm:
        roofline = {"kernel": "gemm_tc_kernel (tcgen05 GEMM engine, all stack/router/projection/"
                              "LM-head contractions)",
                    "bound": "tensor", "achieved": gemm["achieved"], "peak": tc_peak,
                    "unit": "TFLOP/s", "frac": gemm["achieved"] / tc_peak,
                    "traffic": GEMM_DRAM_BYTES_PER_LAUNCH, "traffic_source": GEMM_DRAM_SOURCE,
                    "peak_source": f"{pk_kind} bf16_tflops_sustained",
                    "launches_timed": gemm["launches"], "avg_launch_ms": gemm["avg_ms"],
                    "flops_per_launch": gemm["work_per_launch"], "by_flops_per_launch": gemm_shapes}
    mixer = None
    if mix:
        hbm = pk.get("hbm_gbs", 6400.0)
        mixer = {"bound": "hbm", "achieved": mix["achieved"], "peak": hbm, "unit": "GB/s",
                 "frac": mix["achieved"] / hbm, "peak_source": f"{pk_kind} hbm_gbs",
                 "launches_timed": mix["launches"], "avg_launch_ms": mix["avg_ms"],
                 "bytes_per_launch": mix["work_per_launch"]}
    attention = None
    if attn:
        attention = {"bound": "tensor", "achieved": attn["achieved"], "peak": tc_peak,
                     "unit": "TFLOP/s", "frac": attn["achieved"] / tc_peak,
                     "flops": "causal only (4*Hq*d per visible key)",
                     "launches_timed": attn["launches"], "avg_launch_ms": attn["avg_ms"]}

    # cache writes of the K/V projections (their epilogue scatters the new
    # channel entries): bytes written per launch over the launch's time
    cache_write = None
    kv_flops = 2.0 * wm.rows_for_pass(B, T, g) * s.Hkv * s.d * s.D * s.k
    kv = [(ms_, w_) for ms_, w_ in tracers[0].results() if abs(w_ - kv_flops) < 0.5]
    if kv:
        kv_ms = statistics.mean(r[0] for r in kv)
        kv_bytes = wm.rows_for_pass(B, T, g) * s.k * s.Hkv * s.d * 2
        hbm = pk.get("hbm_gbs", 6400.0)
        cache_write = {"kernel": "gemm_tc_kernel EPI_KV (K or V projection + K-norm + RoPE + "
                                 "cache scatter)",
                       "launches_timed": len(kv), "avg_launch_ms": kv_ms,
                       "bytes_written_per_launch": kv_bytes,
                       "achieved": kv_bytes / (kv_ms * 1e-3) / 1e9, "unit": "GB/s",
                       "frac_of_hbm": kv_bytes / (kv_ms * 1e-3) / 1e9 / hbm,
                       "note": "the launch is a tensor-core product; the cache write is its "
                               "output stream, not its bound",
                       "tflops": kv_flops / (kv_ms * 1e-3) / 1e12}

    others = None
    if args.workload == "prefill_1p3b" and not args.no_other_configs:
        others = other_configs(args, dev)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_record(s, passes, rows=2)

    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if s.dtype == "f32" else "bf16",
        "data": "synthetic (seeded tokens, N(0,0.02) weights)",
        "config": config_dict(args, wl), "e2e": e2e, "gpu_launches": gpu_launches,
        "roofline": roofline, "mixer": mixer, "attention": attention, "decode": decode,
        "cache_write": cache_write, "configs": others, "cpu_baseline": cpu, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def other_configs(args, dev):
    """Prefill tok/s of the other workloads through the same step (CUDA events
    around ``steps`` whole steps after ``warmup``): the tiny fp32 model (3
    cyclic passes g = 4, and 64 Jacobi passes), the half-cache and the
    full-cache small models (3 cyclic passes g = 16, B = 8, T = 2048)."""
    from cross_layer_kv_pool_b300 import wm
    out = {}
    for name, sched in (("tiny_fp32", ((4, 3), (1, 64))), ("half_small", ((16, 3),)),
                        ("full_small", ((16, 3),))):
        wl = synth.WORKLOADS[name]
        s, B, T = wl["shape"], wl["B"], wl["T"]
        m = wm.Model(s, synth.make_weights(s, seed=0, device=dev))
        tok = synth.make_tokens(s, B, T, seed=1, device=dev)
        ck, cv = m.new_cache(B, T)
        lg = torch.empty((B, s.V), dtype=torch.float32, device=dev)
        res = {}
        for g, passes in sched:
            wsp = m.workspace(wm.rows_for_pass(B, T, g), T)

            def step():
                ck.zero_()
                cv.zero_()
                for n in range(passes):
                    last = n == passes - 1
                    wm.wm_cyclic_pass(m, tok, g, ck, cv, wsp, logits=lg if last else None,
                                      logits_mode="last" if last else "none")
            for _ in range(2):
                step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(3):
                step()
            e1.record()
            torch.cuda.synchronize()
            if wm.wm_check_flags(wsp) != 0:
                raise RuntimeError(f"device-side checks failed ({name})")
            ms = e0.elapsed_time(e1) / 3
            res["jacobi" if g == 1 else "cyclic"] = {
                "g": g, "passes": passes, "ms_per_step": ms, "tok_s": B * T / (ms / 1e3)}
            del wsp
        out[name] = {"L": s.L, "D": s.D, "k": s.k, "B": B, "T": T, "dtype": s.dtype,
                     "tok_s": res["cyclic"]["tok_s"], **res}
        del m, ck, cv
        torch.cuda.empty_cache()
    return out


def decode_step_bytes(s, B, pos):
    """Bytes a decode step must move at least: every weight it multiplies by
    (layer stack, LM head, router, channel projections; the B embedding rows),
    the visible K and V entries of each layer's channel, and the new entries."""
    Hd, kv = s.Hq * s.d, s.Hkv * s.d
    layer = Hd * s.D + s.D * Hd + 2 * s.F * s.D + s.D * s.F + 2 * s.D + s.d
    weights = s.L * layer + s.V * s.D + s.D + 2 * s.k * s.L * s.nR * s.D + 2 * s.k * kv * s.D
    cache = s.L * B * 2 * kv * pos + 2 * B * s.k * kv
    return 2 * (weights + B * s.D + cache)


def run_kernel(args):
    """One kernel alone at 1.3B shapes, timed by the library's CUDA events on
    its stream (warm-up launches first; inputs above L2 size for the mixer)."""
    from cross_layer_kv_pool_b300 import wm

    # the pool and attention do not read the vocabulary; a decode step does
    s = synth.HALF_1P3B if args.kernel == "decode" else synth.HALF_1P3B.replace(V=1024)
    dev = torch.device("cuda", torch.cuda.current_device())
    m = wm.Model(s, synth.make_weights(s, seed=0, device=dev, gain_jitter=0.1))
    pk, pk_src = peaks()
    if args.kernel == "mixer":
        N, B, Tmax = args.rows, 4, max(2048, -(-args.rows // 4))
        flat = torch.randperm(B * Tmax, generator=torch.Generator().manual_seed(0))[:N]
        seq = (flat // Tmax).to(torch.int32).to(dev)
        pos = (flat % Tmax).to(torch.int32).to(dev)
        states = synth.make_normal((N, s.L, s.D), 31, dev, 1.0, s.torch_dtype)
        ck, cv = m.new_cache(B, Tmax)
        wsp = m.workspace(N, Tmax)
        kind = wm.WM_TRACE_MIX

        def call():
            wm.wm_pool_mix(m, states, seq, pos, ck, cv, wsp)
        work = N * (s.L * s.D * 2 + 2 * s.k * s.L * 4 + s.L * 4 + 2 * s.k * s.D * 2)
        unit, peak, bound = "GB/s", pk["hbm_gbs"], "hbm"
        desc = f"wm_pool_mix, {N} rows of the 1.3B pool (L=28, D=1792, k=14)"
    elif args.kernel == "pool_backward":
        N = args.rows
        states = synth.make_normal((N, s.L, s.D), 31, dev, 1.0, s.torch_dtype)
        pos = torch.randint(0, 2048, (N,), generator=torch.Generator().manual_seed(0),
                            dtype=torch.int32).to(dev)
        dK = synth.make_normal((N, s.k, s.Hkv, s.d), 32, dev, 1.0, s.torch_dtype)
        dV = synth.make_normal((N, s.k, s.Hkv, s.d), 33, dev, 1.0, s.torch_dtype)
        dst = torch.empty((N, s.L, s.D), dtype=torch.float32, device=dev)
        grads = wm.pool_grads(m)
        wsp = wm.wm_pool_backward(m, states, pos, dK, dV, dst, grads)
        kind = None

        def call():
            wm.wm_pool_backward(m, states, pos, dK, dV, dst, grads, ws=wsp)
        kL, w, nRD = s.k * s.L, s.Hkv * s.d, s.nR * s.D
        # products per branch: router forward, mix forward, key projection (keys
        # only), dW and dc, mix backward (da and dn), router dW_R and dx
        per_branch = (2.0 * N * kL * nRD + 2.0 * N * kL * s.D + 4.0 * N * w * s.D * s.k
                      + 4.0 * N * kL * s.D + 4.0 * N * kL * nRD)
        work = 2 * per_branch + 2.0 * N * w * s.D * s.k
        # the products run on the tensor cores as bf16 hi/lo splits, three
        # bf16 products per fp32-accurate one: their ceiling is a third of
        # the measured bf16 peak, in fp32-equivalent FLOP/s
        unit, peak, bound = "TFLOP/s", pk["bf16_tflops"] / 3.0, "tensor"
        desc = (f"wm_pool_backward, {N} rows of the 1.3B pool, fp32-accurate products "
                "(bf16 hi/lo splits on the tensor cores); peak = measured bf16 burst / 3")
    elif args.kernel == "decode":
        # one decode step of B sequences at position 2048 over a random prefix
        B, T, Tmax = args.batch, 2048, 2304
        ck, cv = m.new_cache(B, Tmax)
        ck.copy_(synth.make_normal(tuple(ck.shape), 4, dev, 1.0, torch.bfloat16))
        cv.copy_(synth.make_normal(tuple(cv.shape), 5, dev, 1.0, torch.bfloat16))
        wsp = m.workspace(B, Tmax)
        tok = synth.make_tokens(s, B, 1, seed=7, device=dev)[:, 0].contiguous()
        pos = torch.full((B,), T, dtype=torch.int32, device=dev)
        lg = torch.empty((B, s.V), dtype=torch.float32, device=dev)
        kind = None

        def call():
            wm.wm_decode_batch(m, tok, pos, ck, cv, lg, wsp)
        work = decode_step_bytes(s, B, T)
        unit, peak, bound = "GB/s", pk["hbm_gbs"], "hbm"
        desc = (f"wm_decode_batch, {B} sequences at position {T} of the 1.3B model "
                "(weights and visible cache entries read once)")
    else:
        B, T, g, Tmax = args.batch, 2048, 16, 2048
        nq = T // g
        pos = torch.arange(args.group, T, g, dtype=torch.int32).repeat(B).to(dev)
        seq = torch.arange(B, dtype=torch.int32).repeat_interleave(nq).to(dev)
        N = B * nq
        q = synth.make_normal((N, s.Hq, s.d), 3, dev, 1.0, torch.bfloat16)
        ck, cv = m.new_cache(B, Tmax)
        ck.copy_(synth.make_normal(tuple(ck.shape), 4, dev, 1.0, torch.bfloat16))
        cv.copy_(synth.make_normal(tuple(cv.shape), 5, dev, 1.0, torch.bfloat16))
        out = torch.empty_like(q)
        wsp = m.workspace(N, Tmax)
        kind = wm.WM_TRACE_ATTN

        def call():
            wm.wm_channel_attn(m.cfg, q, seq, pos, 3, ck, cv, out, wsp, rows_per_seq=nq)
        work = 4.0 * s.Hq * s.d * float(pos.double().sum())
        unit, peak, bound = "TFLOP/s", pk["bf16_tflops"], "tensor"
        desc = f"wm_channel_attn, group {args.group} of {B} sequences of 2048 (1.3B heads)"
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    if kind is None:  # a whole entry point: events around the call on the current stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("timed")
        e0.record()
        for _ in range(args.steps):
            call()
        e1.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / max(args.steps, 1)
    else:
        tr = wm.Tracer(kind, max(args.steps, 1))
        tr.attach(m)
        for _ in range(args.steps):
            call()
        torch.cuda.synchronize()
        wm.Tracer.detach(m)
        ms = statistics.mean(r[0] for r in tr.results())
        if wm.wm_check_flags(wsp) != 0:
            raise RuntimeError("device-side checks failed")
    achieved = work / (ms * 1e-3) / (1e9 if unit == "GB/s" else 1e12)
    print(json.dumps({"kernel": args.kernel, "call": desc, "ms": ms, "achieved": achieved,
                      "unit": unit, "bound": bound, "peak": peak, "frac": achieved / peak,
                      "peak_source": ("fp32 FMA pipes, 148 SMs x 128 lanes x 2 flop x 2.032 GHz"
                                      if bound == "alu" else
                                      f"{pk_src} {'hbm_gbs' if unit == 'GB/s' else 'bf16_tflops (burst)'}"),
                      "work_per_launch": work, "launches": args.steps, "warmup": args.warmup}),
          flush=True)


def run_variant(args):
    """The feedback-free variant ([PL 5 ANALYSIS, "Deep-to-shallow feedback"])
    at the workload's model shape with k = L: one exact layer-by-layer pass
    over B x T tokens through ``wm_feedforward_pass``, last-position logits;
    the workspace holds ``--chunk`` sequences at a time."""
    from cross_layer_kv_pool_b300 import wm

    wl = workload(args)
    s = wl["shape"].replace(k=wl["shape"].L)
    B, T = wl["B"], wl["T"]
    dev = torch.device("cuda", torch.cuda.current_device())
    m = wm.Model(s, synth.make_weights(s, seed=0, device=dev))
    tok = synth.make_tokens(s, B, T, seed=1, device=dev)
    ck, cv = m.new_cache(B, T)
    chunk = max(1, min(args.chunk, B))
    wsp = m.workspace(chunk * T, T)
    lg = torch.empty((B, s.V), dtype=torch.float32, device=dev)

    def step():
        ck.zero_()
        cv.zero_()
        wm.wm_feedforward_pass(m, tok, ck, cv, wsp, logits=lg, logits_mode="last")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if wm.wm_check_flags(wsp) != 0:
        raise RuntimeError("device-side checks failed during warm-up")
    tr = [wm.Tracer(wm.WM_TRACE_GEMM, 4096), wm.Tracer(wm.WM_TRACE_MIX, 512),
          wm.Tracer(wm.WM_TRACE_ATTN, 512)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    # one more step with the per-kernel events on
    kinds = {}
    for t, name in zip(tr, ("gemm", "mixer", "attention")):
        t.attach(m)
        step()
        torch.cuda.synchronize()
        wm.Tracer.detach(m)
        res = t.results()
        kinds[name] = {"launches": len(res), "total_ms": sum(r[0] for r in res),
                       "work": sum(r[1] for r in res)}
    pk, pk_src = peaks()
    kinds["gemm"]["tflops"] = kinds["gemm"]["work"] / (kinds["gemm"]["total_ms"] * 1e9)
    kinds["attention"]["tflops_causal"] = kinds["attention"]["work"] / (kinds["attention"]["total_ms"] * 1e9)
    kinds["mixer"]["gbs"] = kinds["mixer"]["work"] / (kinds["mixer"]["total_ms"] * 1e6)
    print(json.dumps({
        "metric": "prefill tok/s (feedback-free variant, k = L, one pass)", "value": B * T / (ms / 1e3),
        "unit": "tok/s", "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded tokens, N(0,0.02) weights)",
        "config": {"workload": f"{args.workload} shape with k = L = {s.L}, one feedback-free pass",
                   "global_batch": B, "seq_len": T, "chunk_sequences": chunk},
        "kernels": kinds, "peaks": {"source": pk_src, **pk},
        "cache_bytes": 2 * B * s.k * T * s.Hkv * s.d * 2}), flush=True)


def run_convergence(args):
    """Fixed-point convergence of the prefill schedules on the full-cache small
    model (L=16, D=512, k=16, B=8, T=2048): for g in {1 (Jacobi), 4, 16, 64},
    up to ``--passes`` whole passes from a zero cache, each followed by the
    relative residual r_n = ||KV_n - KV_{n-1}||_F / ||KV_n||_F over the cache
    and its CUDA-event time per sequence; then the passes (and milliseconds per
    sequence) needed to reach r <= 1e-1, 3e-2 and 1e-2. Random weights: the
    counts say how contractive this model is, not what a trained one needs."""
    from cross_layer_kv_pool_b300 import wm

    wl = synth.WORKLOADS["full_small"]
    s, B, T = wl["shape"], wl["B"], wl["T"]
    dev = torch.device("cuda", torch.cuda.current_device())
    m = wm.Model(s, synth.make_weights(s, seed=0, device=dev))
    tok = synth.make_tokens(s, B, T, seed=1, device=dev)
    thresholds = (1e-1, 3e-2, 1e-2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {}
    for g in (1, 4, 16, 64):
        ck, cv = m.new_cache(B, T)
        wsp = m.workspace(wm.rows_for_pass(B, T, g), T)
        pk, pv = ck.clone(), cv.clone()
        r, ms = [], []
        for n in range(args.passes):
            torch.cuda.synchronize()
            e0.record()
            wm.wm_cyclic_pass(m, tok, g, ck, cv, wsp)
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1) / B)
            num = (ck.float() - pk.float()).square().sum() + (cv.float() - pv.float()).square().sum()
            den = ck.float().square().sum() + cv.float().square().sum()
            r.append(float((num / den).sqrt()) if float(den) > 0 else 0.0)
            pk.copy_(ck)
            pv.copy_(cv)
        if wm.wm_check_flags(wsp) != 0:
            raise RuntimeError("device-side checks failed")
        reach = {}
        for thr in thresholds:
            n = next((i + 1 for i, v in enumerate(r) if v <= thr), None)
            reach[f"{thr:g}"] = None if n is None else {"passes": n, "ms_per_seq": sum(ms[:n])}
        out[str(g)] = {"residual": r, "ms_per_seq_per_pass": statistics.mean(ms[1:] or ms),
                       "reach": reach, "passes_for_exactness": -(-T // g)}
        del ck, cv, pk, pv, wsp
    print(json.dumps({"sweep": "convergence", "workload": "full_small (L=16, D=512, k=16, B=8, T=2048)",
                      "data": "synthetic", "passes": args.passes, "schedules": out}), flush=True)


def main():
    args = parse()
    if args.kernel:
        run_kernel(args)
        return
    if args.sweep == "convergence":
        run_convergence(args)
        return
    if args.variant:
        run_variant(args)
        return
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
