#!/usr/bin/env python
"""Benchmark of the Mamba-2 chunked SSD forward pass on GB300.

One step = one ssd_forward over one batch of the workload (seeded synthetic
inputs already resident in HBM).  Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--skip-cpu-baseline] [--skip-e2e]

Timing: W untimed warm-up steps, then exactly K timed steps bracketed by a
barrier and torch.cuda.synchronize() on both sides.  Each step is timed with
CUDA events recorded by the library between its own launches on the
launching stream; L2 is flushed (a 256 MB write, outside the events) before
every step.  Under torchrun every rank runs the whole workload on its own GPU
(independent batches: weak scaling, no data-path collective) and the slowest
rank's time is reported.

--impl reference times the float64 CPU oracle on the host cores instead, on
a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mamba_ssd_forward_gb300 import inputs as W  # noqa: E402

METRIC = "SSD forward tokens/s at 1 GB300; achieved TFLOP/s + HBM GB/s vs roofline"
# The headline workload: the largest single-GPU configuration (long context,
# S 256, 8 groups), where the method's gain over other implementations is
# said to grow with sequence length and state size.
DEFAULT_WORKLOAD = W.LONG_32K
# Launch sequence of ssd_forward: bf16 I/O runs the chunk-jump kernel, the
# state pass and the output pass; fp32 I/O runs the cumsum, chunk-state and
# state-passing steps and an output pass (fwd_out_tf32 where it applies).
KERNEL_NAMES = {"bf16": ["fwd_chunk_state", "fwd_state_pass", "fwd_scan"],
                "fp32": ["chunk_cumsum", "chunk_state", "state_passing", "chunk_scan"]}
KERNEL_SOURCES = {"chunk_cumsum": "chunk_cumsum.cu", "chunk_state": "chunk_state.cu",
                  "state_passing": "state_passing.cu", "chunk_scan": "chunk_scan.cu",
                  "fwd_chunk_state": "fwd_chunk_state.cu", "fwd_state_pass": "fwd_state_pass.cu",
                  "fwd_scan": "fwd_scan.cu", "fwd_scan_chunk": "fwd_scan_chunk.cu",
                  "fwd_out": "fwd_out.cu", "fwd_out_tf32": "fwd_out_tf32.cu",
                  "fwd_chunk_state_tf32": "fwd_chunk_state_tf32.cu"}
FALLBACK_HBM_GBS = 6800.0


def workload_by_name(name: str) -> W.Workload:
    for w in W.NAMED + W.sweep():
        if w.name == name or w.name.startswith(name):
            return w
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def io_bytes(w: W.Workload) -> int:
    return 2 if w.dtype == "bf16" else 4


def compulsory_bytes(w: W.Workload) -> int:
    """Bytes the forward pass must move at least once: read x, dt, B, C, A, D
    (and h0), write y and the final state."""
    e = io_bytes(w)
    tok = w.batch * w.seqlen
    n = tok * w.nheads * w.headdim * e * 2            # x in, y out
    n += tok * w.nheads * e                             # dt
    n += 2 * tok * w.ngroups * w.dstate * e             # B, C
    n += 2 * w.nheads * 4                               # A, D
    st = w.batch * w.nheads * w.headdim * w.dstate * 4
    n += st * (2 if w.has_h0 else 1)                    # h0, final state
    return n


def algorithmic_flops(w: W.Workload) -> float:
    """Tensor-core flops per token-head: 4 S P (C h and the chunk state)
    + (T+1) P (causal interaction times X) + (T+1) S / hpg (C B^T, once per
    group), times the token-heads."""
    hpg = w.nheads // w.ngroups
    per = 4 * w.dstate * w.headdim + (w.chunk + 1) * w.headdim + (w.chunk + 1) * w.dstate / hpg
    return per * w.batch * w.seqlen * w.nheads


def kernel_names(w: W.Workload, plan: dict | None = None) -> list:
    """Labels of the kernels ssd_forward launches for this workload, in
    launch order.  The bf16 output pass is the plan's output kernel:
    fwd_out (scan_kernel 3), fwd_scan_chunk (1, or 2: one row tile per CTA)
    or fwd_scan (0)."""
    names = list(KERNEL_NAMES[w.dtype])
    if w.dtype == "fp32" and w.headdim == 64 and w.chunk in (128, 256):
        # the warp-specialised fp32 kernels where the shape allows (the
        # chunk-jump one forms the cumsum itself: one launch less)
        if w.dstate % 32 == 0 and w.dstate <= 256:
            names[3] = "fwd_out_tf32"
        if w.dstate % 64 == 0:
            names = ["fwd_chunk_state_tf32"] + names[2:]
    if w.dtype == "bf16" and plan is not None:
        names[2] = {0: "fwd_scan", 1: "fwd_scan_chunk", 2: "fwd_scan_chunk",
                    3: "fwd_out"}[plan["scan_kernel"]]
    return names


def kernel_method_bytes(w: W.Workload) -> dict:
    """The method's own compulsory bytes that each kernel moves (x, dt, B, C
    read and y written once, h0 read and the final state written), without
    the intermediate per-chunk states or jump terms the kernel split adds."""
    e = io_bytes(w)
    tok = w.batch * w.seqlen
    x = tok * w.nheads * w.headdim * e
    dt = tok * w.nheads * e
    bc = tok * w.ngroups * w.dstate * e
    fin = w.batch * w.nheads * w.headdim * w.dstate * 4
    h0 = fin if w.has_h0 else 0
    out = {"fwd_chunk_state": x + bc + dt + w.nheads * 4,
           "fwd_state_pass": h0 + fin,
           "chunk_cumsum": dt + w.nheads * 4,
           "chunk_state": x + bc + dt,
           "fwd_chunk_state_tf32": x + bc + dt + w.nheads * 4,
           "state_passing": h0 + fin,
           "chunk_scan": 2 * x + 2 * bc + dt + 2 * w.nheads * 4}
    for k in ("fwd_scan", "fwd_scan_chunk", "fwd_out", "fwd_out_tf32"):
        out[k] = out["chunk_scan"]
    return out


def kernel_bytes(w: W.Workload) -> dict:
    """Algorithmic bytes of one launch of each kernel: its own inputs read
    once and outputs written once."""
    e = io_bytes(w)
    tok = w.batch * w.seqlen
    x = tok * w.nheads * w.headdim * e
    dt = tok * w.nheads * e
    bc = tok * w.ngroups * w.dstate * e
    G = w.batch * w.nheads * w.nchunks * w.chunk * 4
    st = w.batch * w.nheads * w.nchunks * w.headdim * w.dstate * 4
    fin = w.batch * w.nheads * w.headdim * w.dstate * 4
    st16 = w.batch * w.nheads * w.nchunks * w.headdim * w.dstate * 2
    # per (batch, head, chunk): (decay, start-state scale) and (anchor, path)
    # float2 pairs; per token and head the fp32 factors u and v of the
    # factored output pass
    gam = w.batch * w.nheads * w.nchunks * 8
    anc = w.batch * w.nheads * w.nchunks * 8
    uv = 2 * w.batch * w.nheads * w.nchunks * w.chunk * 4
    h0 = fin if w.has_h0 else 0
    return {
        "fwd_chunk_state": x + bc + dt + w.nheads * 4 + st16 + gam + anc + uv,
        "fwd_state_pass": 2 * st16 + gam + h0 + fin,
        "fwd_scan": 2 * x + 2 * bc + dt + 2 * w.nheads * 4 + st16,
        "fwd_scan_chunk": 2 * x + 2 * bc + dt + 2 * w.nheads * 4 + st16,
        "fwd_out": 2 * x + 2 * bc + dt + 2 * w.nheads * 4 + st16 + anc + uv,
        "chunk_cumsum": dt + G + w.nheads * 4,
        "chunk_state": x + bc + dt + G + st,
        "fwd_chunk_state_tf32": x + bc + dt + w.nheads * 4 + G + st,
        "state_passing": 2 * st + w.batch * w.nheads * w.nchunks * 4 + fin * (2 if w.has_h0 else 1),
        "chunk_scan": 2 * x + 2 * bc + dt + G + st + w.nheads * 4,
        "fwd_out_tf32": 2 * x + 2 * bc + dt + G + st + 2 * w.nheads * 4,
    }


# ---------------------------------------------------------------------------
# peaks, traffic, clocks
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(kernel: str) -> str:
    path = os.path.join(ROOT, "mamba_ssd_forward_gb300", "csrc", KERNEL_SOURCES[kernel])
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel: str, w: W.Workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel and this workload; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(f"{kernel}@{w.name}")
    except Exception:
        return None
    if not rec or rec.get("source_sha256_16") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.lines = []

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def time_oracle(w: W.Workload, inp, target_s: float, threads: int | None = None):
    """Time the float64 oracle on as many (batch, head) pairs of the workload
    as fit in about target_s seconds, on `threads` OpenMP threads (default:
    all).  Returns (tokens/s, threads, sample, seconds per repetition)."""
    import oracle
    oracle.build()
    oracle.set_threads(threads or os.cpu_count() or 1)
    threads = oracle.max_threads()
    total = w.batch * w.nheads
    t = time.perf_counter()
    oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"],
                      chunk=w.chunk, bh=[0])
    one = max(time.perf_counter() - t, 1e-4)
    n = int(max(1, min(total, target_s / one * threads)))
    if n >= threads:
        n = (n // threads) * threads
    bh = list(range(n))
    t = time.perf_counter()
    oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"],
                      chunk=w.chunk, bh=bh)
    dt_s = time.perf_counter() - t
    reps = 1
    if n == total:
        # the whole workload fits the budget: repeat it for a steadier number
        while dt_s < min(target_s, 5.0) and reps < 64:
            t = time.perf_counter()
            oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["h0"], chunk=w.chunk, bh=bh)
            dt_s += time.perf_counter() - t
            reps += 1
    tok_per_s = reps * n * w.seqlen / w.nheads / dt_s
    what = f"{n} of {total} (batch, head) pairs at full length L={w.seqlen}"
    if reps > 1:
        what += f", whole workload repeated {reps} times"
    return tok_per_s, threads, what, dt_s / reps


def host_inputs(w):
    inp = W.make_inputs(w, seed=0)
    return inp


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_throughput(ms_local: float, tokens_per_rank: int, world: int, device=None):
    """Whole-job step time and tokens/s of `world` replicas: the slowest
    rank's step time (max over ranks, one all-reduce) and every rank's
    tokens.  world == 1 needs no process group."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_per_rank / (ms / 1e3)


def run_reference(args, w):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    inp = host_inputs(w)
    # each step: a bounded sample sized so that W + K steps take a few minutes
    budget = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    times, vals = [], []
    threads = sample = None
    for i in range(args.warmup + args.steps):
        v, threads, sample, secs = time_oracle(w, inp, budget)
        if i >= args.warmup:
            vals.append(v)
            times.append(secs)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import mamba_ssd_forward_gb300 as ssd
    from mamba_ssd_forward_gb300 import build

    world, rank, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()

    inp = host_inputs(w)
    d = {k: (None if v is None else v.to(dev).contiguous()) for k, v in inp.items()}
    ws = ssd.new_workspace(ssd.workspace_size(d["x"], d["B"], w.chunk), dev)
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
    # L2 flush between steps: write a 256 MB buffer, then read another 256 MB
    # one, so that L2 holds neither the workload's data nor dirty lines whose
    # write-back would land inside the next timed step.
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    flush_sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        if args.flush == "write+read":
            torch.sum(flush_r, dim=0, keepdim=True, out=flush_sink)

    nev = 8

    # launch plan: the timing autotuner's choice for this shape (once, before
    # the warm-up; every candidate timed from a cold L2, as the timed steps
    # run; passed to every later call), or the cost model's
    plan, tuned = None, False
    if w.dtype == "bf16":
        dims = ssd.dims_of(d["x"], d["B"], w.chunk)
        if args.tune:
            plan, _, _ = ssd.tune(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                                  chunk=w.chunk, reps=5, workspace=ws, flush=flush_w)
            tuned = True
        else:
            plan = ssd.default_plan(dims)

    def step(events):
        return ssd.forward_profiled(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                                    w.chunk, ws, y, fin, events, plan=plan)

    warm_ev = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
    for _ in range(args.warmup):
        flush()
        step(warm_ev)
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    launches = 0
    n_l = 0
    for i in range(args.steps):
        flush()
        if args.kernel_events == "separate":
            ev[i][0].record()
            n_l = step([])
            for j in range(1, n_l + 1):
                ev[i][j].record()  # all after the step: step time = ev[0] -> ev[n_l]
        else:
            n_l = step(ev[i])
        launches += n_l
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if sampler:
        sampler.mark_end()
    clocks = sampler.stop() if sampler else None
    ssd.workspace_error(ws)  # no bounded device-side wait gave up in the timed steps

    step_ms = [ev[i][0].elapsed_time(ev[i][n_l]) for i in range(args.steps)]
    names = kernel_names(w, plan)
    kern_ms = {names[j]: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1])
                                                for i in range(args.steps))
               for j in range(n_l)}
    if args.kernel_events == "separate":
        # the timed steps above recorded only their first and last events;
        # the per-kernel split comes from as many steps again with an event
        # between launches (events between launches serialise them)
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)]
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            step(ev2[i])
        torch.cuda.synchronize()
        kern_ms = {names[j]: statistics.mean(ev2[i][j].elapsed_time(ev2[i][j + 1])
                                                    for i in range(args.steps))
                   for j in range(n_l)}
    ms, value = job_throughput(statistics.mean(step_ms), w.batch * w.seqlen, world, dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    # roofline of the dominant kernel
    dom = max(kern_ms, key=kern_ms.get)
    kb = kernel_bytes(w)
    peak, peak_src = hbm_peak()
    achieved = kb[dom] / (kern_ms[dom] / 1e3) / 1e9
    mb = kernel_method_bytes(w)
    method_gbs = mb[dom] / (kern_ms[dom] / 1e3) / 1e9
    roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": kb[dom], "traffic": ncu_traffic(dom, w),
            # the same kernel counted by the method's compulsory bytes only
            # (its x, dt, B, C reads and y writes; no per-chunk states)
            "method_bytes_per_launch": mb[dom], "method_achieved": method_gbs,
            "method_frac": method_gbs / peak,
            "kernel_ms": kern_ms,
            "kernel_share": {k: v / sum(kern_ms.values()) for k, v in kern_ms.items()}}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded, distributions of the layer; no dataset)",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen,
                   "nheads": w.nheads, "headdim": w.headdim, "dstate": w.dstate,
                   "ngroups": w.ngroups, "chunk": w.chunk, "h0": w.has_h0,
                   "l2": ("flushed before every step outside the timed events: 256 MB write"
                          + (" then 256 MB read (clean L2)" if args.flush == "write+read" else "")),
                   "parallelism": f"replicas x{world} (independent batches per GPU)",
                   "plan": plan, "plan_source": "timing autotuner" if tuned else "cost model"},
        "achieved_tflops": algorithmic_flops(w) / (ms / 1e3) / 1e12,
        "achieved_gbs_compulsory": compulsory_bytes(w) / (ms / 1e3) / 1e9,
        "roofline_forward": {"bound": "hbm", "frac": compulsory_bytes(w) / (ms / 1e3) / 1e9 / peak,
                             "compulsory_bytes": compulsory_bytes(w)},
        "roofline": roof,
        "gpu_launches": launches,
        "clocks": clocks,
    }

    if not args.skip_e2e:
        line["e2e"] = e2e(args, w, inp, dev, overlapped=True, plan=plan)
        line["e2e_serial"] = e2e(args, w, inp, dev, overlapped=False, plan=plan)
    if not args.skip_cpu_baseline and world == 1:
        v, threads, sample, _ = time_oracle(w, inp, 15.0)
        v1, _, sample1, _ = time_oracle(w, inp, 5.0, threads=1)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle", "sample": sample,
                                "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                                                  "sample": sample1}}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def e2e(args, w, inp, dev, overlapped=True, plan=None):
    """Same metric through the host-buffer API: pinned host inputs copied in,
    forward, y and the final state copied out, every step.  overlapped:
    ssd_forward_host_overlapped (the copies of up to --e2e-slices slices overlap the
    computation on two extra streams); else ssd_forward_host (serial)."""
    import torch

    import mamba_ssd_forward_gb300 as ssd
    h = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}
    y = torch.empty_like(h["x"]).pin_memory()
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32).pin_memory()
    n_slices = args.e2e_slices
    if overlapped:
        ws = ssd.new_workspace(ssd.host_overlapped_workspace_size(
            h["x"], h["B"], w.chunk, n_slices, True, h["h0"] is not None, True), dev)
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def call():
            ssd.forward_host_overlapped(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["h0"],
                                        w.chunk, ws, y, fin, n_slices=n_slices, h2d_stream=s_in,
                                        d2h_stream=s_out, plan=plan)
    else:
        ws = ssd.new_workspace(ssd.host_workspace_size(h["x"], h["B"], w.chunk, has_D=True,
                                                       has_h0=h["h0"] is not None), dev)

        def call():
            ssd.forward_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["h0"], w.chunk,
                             ws, y, fin, plan=plan)
    h2d = sum(v.numel() * v.element_size() for v in h.values() if v is not None)
    d2h = y.numel() * y.element_size() + fin.numel() * fin.element_size()
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    n = max(args.steps, 3)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(n):
        call()
    e.record()
    torch.cuda.synchronize()
    ssd.workspace_error(ws)
    ms = s.elapsed_time(e) / n
    out = {"value": w.batch * w.seqlen / (ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
           "api": "ssd_forward_host_overlapped" if overlapped else "ssd_forward_host"}
    if overlapped:
        out["n_slices"] = n_slices
    out["copy_ceiling"] = copy_ceiling(h2d, d2h, dev, n)
    out["copy_ceiling"]["frac"] = out["copy_ceiling"]["ms_floor"] / ms
    return out


def copy_ceiling(h2d: int, d2h: int, dev, reps: int) -> dict:
    """The host link's own limit for the e2e step: one pinned host-to-device
    copy of the step's input bytes and one device-to-host copy of its output
    bytes, each timed alone (CUDA events, best of reps) and both at once on
    two streams.  ms_floor = the concurrent time, the least any call moving
    those bytes can take."""
    import torch
    hs = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    hd = torch.empty(h2d, dtype=torch.uint8, device=dev)
    ds = torch.empty(d2h, dtype=torch.uint8, device=dev)
    dd = torch.empty(d2h, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(f):
        best = float("inf")
        for _ in range(max(3, reps)):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            f()
            torch.cuda.synchronize()
            best = min(best, (time.perf_counter() - t0) * 1e3)
        return best

    def up():
        with torch.cuda.stream(s1):
            hd.copy_(hs, non_blocking=True)

    def down():
        with torch.cuda.stream(s2):
            dd.copy_(ds, non_blocking=True)

    t_up, t_down = timed(up), timed(down)
    t_both = timed(lambda: (up(), down()))
    return {"h2d_gbs": h2d / t_up / 1e6, "d2h_gbs": d2h / t_down / 1e6,
            "ms_h2d": t_up, "ms_d2h": t_down, "ms_floor": t_both,
            "how": "pinned copies of the step's bytes, host-timed around a synchronize, best of "
                   f"{max(3, reps)}"}


def run_decode(args, w):
    """The single-token decode step (ssd_decode_step) on the workload's layer
    shape with --decode-batch sequences: one token for every (batch, head)
    state per step, the state resident in HBM and L2 flushed between steps.
    Prints its own JSON line (mode "decode"); not the headline metric."""
    import torch

    import mamba_ssd_forward_gb300 as ssd
    from mamba_ssd_forward_gb300 import build

    build.build()
    dev = torch.device("cuda", 0)
    b = args.decode_batch or w.batch
    dw = W.Workload(w.name + "_decode", b, 1, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk,
                    w.dtype, True)
    inp = host_inputs(dw)
    d = {k: (None if v is None else v.to(dev).contiguous()) for k, v in inp.items()}
    x, dt, Bm, Cm = (d[k][:, 0].clone() for k in ("x", "dt", "B", "C"))
    state = d["h0"].clone()
    y = torch.empty_like(x)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        flush_w.zero_()
        ssd.decode_step(x, dt, d["A"], Bm, Cm, d["D"], state, y)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for e0, e1 in ev:
        flush_w.zero_()
        e0.record()
        ssd.decode_step(x, dt, d["A"], Bm, Cm, d["D"], state, y)
        e1.record()
    torch.cuda.synchronize()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    e = io_bytes(dw)
    st_bytes = 2 * b * w.nheads * w.headdim * w.dstate * 4
    io = b * w.nheads * (2 * w.headdim + 1) * e + 2 * b * w.ngroups * w.dstate * e
    peak, peak_src = hbm_peak()
    gbs = (st_bytes + io) / (ms / 1e3) / 1e9
    line = {
        "metric": "SSD decode step tokens/s (one token for each of batch sequences)",
        "mode": "decode", "value": b / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": dw.name, "batch": b, "nheads": w.nheads, "headdim": w.headdim,
                   "dstate": w.dstate, "ngroups": w.ngroups,
                   "l2": "flushed before every step (256 MB write), outside the events"},
        "roofline": {"kernel": "decode_step", "bound": "hbm", "achieved": gbs, "peak": peak,
                     "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": st_bytes + io, "traffic": None},
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


# fp32 CUDA-core peak of one GB300: 152 SMs x 128 fp32 lanes x 2 flop per FMA
# x the 2070 MHz maximum SM clock (the ALU roofline of the backward kernels)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
BWD_KERNELS = ["chunk_cumsum", "bwd_scale", "jump GEMM (x~, B)", "state_passing",
               "jump GEMM (gy~, C)", "state_passing(reverse)", "Kcb GEMM (c . B)",
               "state GEMMs (dx, ysm)", "bwd_main", "bwd_finish", "bwd_reduce",
               "state GEMMs (dB, dC)"]
GEMM_STEPS = ["jump GEMM (x~, B)", "jump GEMM (gy~, C)", "Kcb GEMM (c . B)",
              "state GEMMs (dx, ysm)", "state GEMMs (dB, dC)"]


def backward_macs(w: W.Workload) -> dict:
    """Multiply-adds the backward needs (the algorithmic count, with the
    causal triangle of each chunk counted once and C . B shared by a group's
    heads), split into the per-token kernel's share and the rest."""
    P, S, T = w.headdim, w.dstate, w.chunk
    main = gemm = jump = rest = 0
    for k in range(w.nchunks):
        v = min(T, w.seqlen - k * T)
        npair = v * (v + 1) // 2
        # per head: the scores gy_i . x_j and the P-wide masked products
        # (ysm, dx).  Per group: the S-wide masked products (dB, dC), whose
        # weights add up over the group's heads before they meet B or C
        main += w.batch * w.nheads * npair * 3 * P
        main += w.batch * w.ngroups * npair * 2 * S
        # the four state terms of every token (R B, h c, R^T x~, h^T g~y):
        # two GEMM launches of two products each
        gemm += w.batch * w.nheads * 4 * v * P * S
        jump += w.batch * w.nheads * 2 * v * P * S  # the two jump terms
        jump += w.batch * w.ngroups * npair * S  # c_i . B_j, once per group (Kcb)
        rest += w.batch * w.nheads * P * S  # <R_k, h_k+1>
    return {"bwd_main": main, "gemms": gemm + jump, "total": main + gemm + jump + rest}


def state_gemm_bytes(w: W.Workload) -> int:
    """HBM bytes the five GEMM steps must move (fp32): the jump terms read x~,
    g~y, B, C and write two state-sized buffers; Kcb reads B and C and writes
    the lower triangle of every chunk's T x T block; the state terms read R_k
    and h_k twice, B and C, x~ and g~y once, write dx~S and ysm~S, and read
    and write dB and dC."""
    f = 4
    states = 2 * w.batch * w.nchunks * w.nheads * w.headdim * w.dstate * f
    bc = 2 * w.batch * w.seqlen * w.ngroups * w.dstate * f
    xp = 2 * w.batch * w.seqlen * w.nheads * w.headdim * f
    jump = xp + bc + states            # read x~, g~y, B, C; write dH, dR
    T = w.chunk
    kcb = bc + w.batch * w.ngroups * w.nchunks * T * (T + 1) // 2 * f
    before = states + bc + xp          # read R, h, B, C; write dxS, ysmS
    after = states + xp + 2 * bc       # read R, h, x~, g~y; read and write dB, dC
    return jump + kcb + before + after


def time_oracle_backward(w: W.Workload, inp, gy, gfinal, target_s: float):
    """Time the oracle's chunked backward (numpy float64) on the first
    (batch, head) pair, over as many tokens as fit in about target_s seconds.
    Returns (tokens/s of the whole workload's heads, sample)."""
    import oracle
    g = 0
    L = w.seqlen
    sl = lambda t, n: t[:1, :n, :1].contiguous() if t.dim() == 4 else t[:1, :n, :1]
    def run(n):
        t0 = time.perf_counter()
        oracle.backward_chunked(sl(inp["x"], n), sl(inp["dt"], n), inp["A"][:1],
                                inp["B"][:1, :n, g:g + 1], inp["C"][:1, :n, g:g + 1],
                                inp["D"][:1], None if inp["h0"] is None else inp["h0"][:1, :1],
                                gy[:1, :n, :1], gfinal[:1, :1], chunk=w.chunk)
        return time.perf_counter() - t0
    n = min(L, 4 * w.chunk)
    secs = run(n)
    if secs < target_s and n < L:
        n = min(L, max(n, int(n * target_s / max(secs, 1e-3)) // w.chunk * w.chunk))
        secs = run(n)
    return n / secs / w.nheads, f"1 (batch, head) pair, the first {n} of L={L} tokens"


def run_backward(args, w):
    """The backward pass (ssd_backward, fp32 I/O) on the workload's shape in
    fp32, with seeded dL/dy and dL/dfinal_state; L2 flushed before every
    step.  Prints its own JSON line (mode "backward"); not the headline."""
    import torch

    import mamba_ssd_forward_gb300 as ssd
    from mamba_ssd_forward_gb300 import build

    build.build()
    dev = torch.device("cuda", 0)
    wf = w if w.dtype == "fp32" else W.Workload(w.name.replace("bf16", "fp32"), w.batch,
                                                 w.seqlen, w.nheads, w.headdim, w.dstate,
                                                 w.ngroups, w.chunk, "fp32", w.has_h0)
    inp = host_inputs(wf)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(1)
    gy = torch.randn((wf.batch, wf.seqlen, wf.nheads, wf.headdim), generator=gen)
    gfinal = torch.randn((wf.batch, wf.nheads, wf.headdim, wf.dstate), generator=gen)
    d = {k: (None if v is None else v.to(dev).contiguous()) for k, v in inp.items()}
    gyd, gfd = gy.to(dev), gfinal.to(dev)
    ws = ssd.new_workspace(ssd.backward_workspace_size(d["x"], d["B"], wf.chunk), dev)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    nk = len(BWD_KERNELS)
    out = None

    def step(events):
        return ssd.backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], gyd, gfd,
                            chunk=wf.chunk, workspace=ws, out=out, events=events)

    warm = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
    for _ in range(max(3, args.warmup)):
        flush_w.zero_()
        out = step(warm)
    torch.cuda.synchronize()
    ssd.workspace_error(ws)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(0)
    time.sleep(0.3)
    torch.cuda.synchronize()
    sampler.mark_start()
    launches = 0
    for evs in ev:
        flush_w.zero_()
        launches += step(evs)["n_launches"]
    torch.cuda.synchronize()
    sampler.mark_end()
    clocks = sampler.stop()
    ssd.workspace_error(ws)
    ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in ev)
    per = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ev)
           for i, n in enumerate(BWD_KERNELS)}
    macs = backward_macs(wf)
    tf_main = 2 * macs["bwd_main"] / (per["bwd_main"] / 1e3) / 1e12
    tf_all = 2 * macs["total"] / (ms / 1e3) / 1e12
    ms_gemm = sum(per[n] for n in GEMM_STEPS)
    tf_gemm = 2 * macs["gemms"] / (ms_gemm / 1e3) / 1e12
    gemm_bytes = state_gemm_bytes(wf)
    tokens = wf.batch * wf.seqlen
    cpu = None
    if not args.skip_cpu_baseline:
        v, sample = time_oracle_backward(wf, inp, gy.double(), gfinal.double(), 10.0)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": sample + " (numpy float64, chunked backward)"}
    line = {
        "metric": "SSD backward tokens/s at 1 GB300 (fp32 I/O, gradients of every input)",
        "mode": "backward", "value": tokens / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wf.name, "batch": wf.batch, "seqlen": wf.seqlen,
                   "nheads": wf.nheads, "headdim": wf.headdim, "dstate": wf.dstate,
                   "ngroups": wf.ngroups, "chunk": wf.chunk,
                   "l2": "flushed before every step (256 MB write), outside the events"},
        "kernels_ms": per,
        "roofline": {"kernel": "bwd_main", "bound": "alu", "achieved": tf_main,
                     "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s",
                     "frac": tf_main / FP32_ALU_TFLOPS,
                     "peak_source": "152 SMs x 128 fp32 lanes x 2 x 2070 MHz",
                     "algorithmic_flops_per_launch": 2 * macs["bwd_main"], "traffic": None},
        "whole_pass": {"achieved_tflops": tf_all, "frac": tf_all / FP32_ALU_TFLOPS,
                       "algorithmic_flops": 2 * macs["total"]},
        "gemms": {"steps": GEMM_STEPS, "achieved_tflops": tf_gemm, "ms": ms_gemm,
                  "algorithmic_flops": 2 * macs["gemms"], "hbm_bytes": gemm_bytes,
                  "hbm_frac": gemm_bytes / (ms_gemm / 1e3) / 1e9 / hbm_peak()[0],
                  "kernel": "bwd_state_gemm (split-TF32 tcgen05)"},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": launches, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD.name)
    ap.add_argument("--kernel-events", choices=["inline", "separate"], default="inline",
                    help="inline: CUDA events between the launches of every timed step; "
                         "separate: timed steps carry only start/end events and the "
                         "per-kernel split is taken from extra steps after the timed region")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--no-tune", dest="tune", action="store_false",
                    help="use the cost-model launch plan instead of timing the candidates")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--e2e-slices", type=int, default=8,
                    help="slices of the host-buffer path (copies overlap the computation)")
    ap.add_argument("--flush", choices=["write+read", "write"], default="write+read",
                    help="L2 flush between steps (default: write a buffer, then read another)")
    ap.add_argument("--decode", action="store_true",
                    help="time the single-token decode step instead of the forward pass")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (fp32 I/O) instead of the forward pass")
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="sequences per decode step (default: the workload's batch)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    w = workload_by_name(args.workload)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.decode:
        return run_decode(args, w)
    if args.backward:
        return run_backward(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
