"""Attention-forward benchmark: device-timed TFLOPS on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--path fwd|mask|bwd|fp8] [--no-cpu-baseline] [--no-e2e]

A step is one attention forward (the whole path: every kernel attn_fwd
launches) over one batch of the workload's seeded synthetic inputs, already
resident in HBM.  Between timed steps a 512 MiB buffer is rewritten to flush
L2, outside the per-step CUDA events.  FLOPs = 4*B*Hq*Nq*Nkv*D, halved when
causal.  Under torchrun every rank runs the full workload on its own GPU
(weak scaling, no data-path collective); the reported time is the max over
ranks and the value is the FLOPs of all ranks over that time.

``--path`` selects what a step runs besides the default forward: the forward
with an additive mask, the backward (FLOPs 2.5x the forward's), or the FP8
forward (quantisation included; roofline against twice the measured bf16
peak, the nominal e4m3/bf16 ratio).  Those lines carry no e2e or CPU leg.

``--impl reference`` times the float64 CPU oracle on the host cores instead
(there is no other implementation of this path to run), on a bounded sample
of the same workload per step.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from exact_attention_attn_gb300.workloads import (BENCH_WORKLOAD, WORKLOADS, make_workload_inputs,  # noqa: E402
                                                  sample_rows, to_f64)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def reduce_max(x: float, ws: int, device=None) -> float:
    """Max of a host scalar over ranks (timing only, not the data path)."""
    if ws <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


# --------------------------------------------------------------------------
# clocks during the timed region

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                smax.append(float(row[2]))
            except ValueError:
                continue
            for n, val in zip(names, row[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# ncu traffic recorded in profiles/ (null when the kernel source changed since)

# The sources a kernel's code and launch depend on: its own translation unit
# plus the shared headers, the tensor-map builder and the launch planner.
_COMMON_SOURCES = ("attn_internal.h", "attn_mask.cuh", "sm100_ptx.cuh", "tma_host.cu", "attn_api.cu")
KERNEL_SOURCES = {
    "attn_tc2_kernel": ("attn_tc2.cu",) + _COMMON_SOURCES,
    "attn_tc_kernel": ("attn_tc.cu",) + _COMMON_SOURCES,
    "attn_tcx_kernel": ("attn_tcx.cu",) + _COMMON_SOURCES,
    "attn_bwd_dkdv_kernel": ("attn_bwd.cu",) + _COMMON_SOURCES,
    "attn_bwd_dq_kernel": ("attn_bwd.cu",) + _COMMON_SOURCES,
    "attn_fp8_kernel": ("attn_fp8.cu",) + _COMMON_SOURCES,
}


def _code_only(src: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed, so
    that an edit of comments or layout alone leaves the hash unchanged.
    String and character literals are kept whole."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str) -> str:
    """First 16 hex digits of sha256 over the code (comments and layout
    removed) of the named kernel's source files."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_attn_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """Parse profiles/ncu_traffic.md rows: | workload | kernel | source hash | bytes per launch |.
    A row counts only while its kernel's sources still hash to its value."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None, None
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) < 4 or cells[0] != workload:
            continue
        base = cells[1].split("<")[0]
        if base not in KERNEL_SOURCES or cells[2] != kernel_source_hash(base):
            continue
        try:
            return float(cells[3]), cells[1]
        except ValueError:
            pass
    return None, None


# --------------------------------------------------------------------------
# CPU oracle timing

def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else None
    except Exception:
        return None


def oracle_rows(w):
    """Query rows the CPU oracle runs per head: the workload's seeded sample
    (256 rows per head on the large workloads, the rows its parity checks
    use), else every row."""
    return sample_rows(w.Nq, w.sample_rows, w.seed) if w.sample_rows else None


def path_host_inputs(path: str, w):
    """Seeded host tensors a path adds to q, k and v: the additive mask
    ([Nq, Nkv] bf16, a view of a row store padded to a multiple of 8
    columns) of the masked path and the upstream gradient dO of the
    backward.  Both legs of the bench (kernels and oracle) use these."""
    extra = {}
    if path == "mask":
        g = torch.Generator().manual_seed(w.seed + 7)
        pad = (w.Nkv + 7) // 8 * 8
        extra["mask"] = (torch.randn((w.Nq, pad), generator=g) * 2.0).to(torch.bfloat16)[:, :w.Nkv]
    if path == "bwd":
        g = torch.Generator().manual_seed(w.seed + 1000)
        extra["dout"] = torch.randn((w.B, w.Hq, w.Nq, w.D), generator=g).to(torch.bfloat16)
    return extra


def time_oracle(w, q, k, v, budget_s: float, max_heads: int | None = None, path: str = "fwd",
                extra: dict | None = None):
    """Run the oracle of `path` head by head over the workload until
    budget_s seconds have passed (at least one head).  Returns (TFLOPS,
    heads, seconds, rows per head).

    fwd, mask, fp8: the forward of one (b, hq) head on its sampled rows
    where the workload samples (fp8 first rotates and quantises that head's
    Q, K and V as the FP8 path does); the FLOPs credited are the workload's
    FLOPs per head times the share of rows that ran (a per-row linear
    extrapolation when rows are sampled).  bwd: the whole backward of one
    head (every row: dK and dV need them all), credited 2.5 x the forward's
    FLOPs per head."""
    import oracle
    B, Hq = w.B, w.Hq
    heads = [(b, h) for b in range(B) for h in range(Hq)]
    if max_heads:
        heads = heads[:max_heads]
    rows = None if path == "bwd" else oracle_rows(w)
    nrows = w.Nq if rows is None else len(rows)
    per_head_flops = (2.5 if path == "bwd" else 1.0) * w.flops() / (B * Hq) * nrows / w.Nq
    mask = None if path != "mask" else to_f64(extra["mask"])
    done = 0
    t0 = time.perf_counter()
    group = w.Hq // w.Hkv
    for b, h in heads:
        kvh = h // group
        if path == "fp8":
            (qd, kd, vd), _ = oracle.fp8.fp8_inputs(to_f64(q[b:b + 1, h:h + 1]),
                                                    to_f64(k[b:b + 1, kvh:kvh + 1]),
                                                    to_f64(v[b:b + 1, kvh:kvh + 1]))
            oracle.attention_head(qd[0, 0], kd[0, 0], vd[0, 0], w.scale, w.causal, rows)
        elif path == "bwd":
            oracle.attention_backward_head(to_f64(q[b, h]), to_f64(k[b, kvh]), to_f64(v[b, kvh]),
                                           to_f64(extra["dout"][b, h]), w.scale, w.causal)
        else:
            oracle.attention_head(to_f64(q[b, h]), to_f64(k[b, kvh]), to_f64(v[b, kvh]), w.scale, w.causal,
                                  rows, mask)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return per_head_flops * done / dt / 1e12, done, dt, nrows


def oracle_sample_text(w, heads, dt, nrows, threads, path="fwd"):
    if path != "fwd":
        what = {"mask": "the masked forward", "fp8": "FWHT rotation + e4m3 quantisation of Q, K, V, then the forward",
                "bwd": "the whole backward (dQ, dK, dV; FLOPs credited 2.5 x the forward's)"}[path]
        rows = f"{nrows} seeded rows" if nrows < w.Nq else f"all {w.Nq} rows"
        return (f"{what} on {rows} of each of {heads} (b,hq) heads (of {w.B * w.Hq}) of {w.name}; "
                f"float64 numpy on {threads} host thread(s), {dt:.1f} s")
    what = (f"{nrows} seeded rows of each of {heads} (b,hq) heads (of {w.B * w.Hq}) of {w.name}; TFLOPS credit "
            f"each head with its FLOPs x {nrows}/{w.Nq} (per-row linear extrapolation)" if nrows < w.Nq else
            f"{heads} of {w.B * w.Hq} (b,hq) heads of {w.name}, all {w.Nq} rows each")
    return f"{what}; float64 numpy on {threads} host thread(s), {dt:.1f} s"


def single_thread_oracle(w, budget_s: float):
    """The oracle on one host thread, in a child process whose BLAS pools are
    capped at one thread before numpy loads.  Returns the cpu_baseline-style
    dict, or None if the child fails."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-only", "--workload", w.name,
           "--cpu-seconds", str(budget_s)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s * 4 + 120)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except (subprocess.TimeoutExpired, ValueError, IndexError):
        return None


def oracle_only(args, w):
    q, k, v = make_workload_inputs(w)
    tf, heads, dt, nrows = time_oracle(w, q, k, v, budget_s=args.cpu_seconds)
    threads = blas_threads() or int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0) or cpu_cores()
    print(json.dumps({"value": tf, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                      "sample": oracle_sample_text(w, heads, dt, nrows, threads)}), flush=True)
    return 0


def bench_config(w, ws: int) -> dict:
    """The workload as both arms report it."""
    return dict(w.describe(), l2="flushed between steps (512 MiB write, outside the events)",
                parallelism=f"replicas x{ws}" if ws > 1 else "1 GPU")


# --------------------------------------------------------------------------

def run_reference(args, w):
    ws, rank, _ = dist_info()
    if ws > 1 and rank != 0:
        return 0
    q, k, v = make_workload_inputs(w)
    extra = path_host_inputs(args.path, w)
    # about 100 s of oracle work for the whole run (5 s a step at 20 steps),
    # at least half a second and one head a step
    per_step_budget = min(5.0, max(0.5, 100.0 / max(args.steps, 1)))
    for _ in range(args.warmup):
        time_oracle(w, q, k, v, budget_s=0.0, max_heads=1, path=args.path, extra=extra)
    vals, heads_total, secs, nrows = [], 0, 0.0, w.Nq
    for _ in range(args.steps):
        tf, heads, dt, nrows = time_oracle(w, q, k, v, budget_s=per_step_budget, path=args.path, extra=extra)
        vals.append(tf)
        heads_total += heads
        secs += dt
    value = statistics.mean(vals)
    cores = blas_threads() or cpu_cores()
    sample = (oracle_sample_text(w, heads_total, secs, nrows, cores, args.path) +
              f"; {args.steps} steps, each stopping after {per_step_budget:.1f} s")
    flops_per_head = (2.5 if args.path == "bwd" else 1.0) * w.flops() / (w.B * w.Hq)
    line = {
        "impl": "reference", "metric": PATHS[args.path][0] or METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": 0 if ws <= 1 else ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(bench_config(w, ws), **({"path": args.path} if args.path != "fwd" else {})),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "flops_per_head": flops_per_head,
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = "attn fwd TFLOPS (bf16, device-timed, 1 GPU) and % of GB300 dense BF16 peak"


PATHS = {
    # path: (metric, dtype, what a step runs)
    "fwd": (None, "bf16", "attn_fwd: one forward"),
    "mask": ("attn fwd with an additive mask TFLOPS (bf16, device-timed, 1 GPU)", "bf16",
             "attn_fwd_masked with one [Nq, Nkv] bf16 mask shared by every batch and head"),
    "bwd": ("attn bwd TFLOPS (bf16, device-timed, 1 GPU; FLOPs = 2.5 x the forward's)", "bf16",
            "attn_bwd: Delta/LSE prep, dK/dV kernel, dQ kernel"),
    "fp8": ("attn fwd FP8 TFLOPS (e4m3 operands, device-timed, 1 GPU)", "e4m3",
            "attn_fp8_quantize of bf16 q, k, v then attn_fwd_fp8"),
}


def make_step(path, w, dev, dq, dk, dv, out, lse, stream, extra):
    """The callable one step runs, its FLOPs, its algorithmic HBM bytes, and
    for the end-to-end leg the (host, device) input pairs a user copies in
    and the device results a user reads back."""
    from exact_attention_attn_gb300 import attn_bwd, attn_fp8_quantize, attn_fwd, attn_fwd_fp8
    ins, outs = [], [out, lse]
    if path == "fwd":
        step = lambda: attn_fwd(dq, dk, dv, scale=w.scale, causal=w.causal, out=out, lse=lse,  # noqa: E731
                                stream=stream)
        return step, w.flops(), w.hbm_bytes(), ins, outs
    if path == "mask":
        host_store = extra["mask"].as_strided((w.Nq, (w.Nkv + 7) // 8 * 8), extra["mask"].stride())
        store = host_store.to(dev)
        mask = store[:, :w.Nkv]
        ins = [(host_store, store)]
        step = lambda: attn_fwd(dq, dk, dv, scale=w.scale, causal=w.causal, out=out, lse=lse,  # noqa: E731
                                stream=stream, mask=mask)
        return step, w.flops(), w.hbm_bytes() + w.Nq * w.Nkv * 2, ins, outs
    if path == "bwd":
        attn_fwd(dq, dk, dv, scale=w.scale, causal=w.causal, out=out, lse=lse, stream=stream)
        dout = extra["dout"].to(dev)
        gq, gk, gv = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
        qo = w.B * w.Hq * w.Nq * w.D * 2
        kv = w.B * w.Hkv * w.Nkv * w.D * 2
        byts = 3 * qo + 2 * kv + w.B * w.Hq * w.Nq * 4 + qo + 2 * kv   # q, o, dO, k, v, lse in; dq, dk, dv out
        ins = [(out.cpu(), out), (lse.cpu(), lse), (extra["dout"], dout)]
        step = lambda: attn_bwd(dq, dk, dv, out, lse, dout, scale=w.scale, causal=w.causal,  # noqa: E731
                                stream=stream, dq=gq, dk=gk, dv=gv)
        return step, 2.5 * w.flops(), byts, ins, [gq, gk, gv]
    if path == "fp8":
        step = lambda: attn_fwd_fp8(attn_fp8_quantize(dq, dk, dv, stream=stream),  # noqa: E731
                                    scale=w.scale, causal=w.causal, out=out, lse=lse, stream=stream)
        return step, w.flops(), w.hbm_bytes(), ins, outs
    raise ValueError(path)


def e2e_path(step, flops, ins, outs, q, k, v, dq, dk, dv, stream, n, ws, dev):
    """A path's metric end to end through the Python API: every step copies
    its inputs from pinned host memory to the device, runs the path, and
    copies its results back to pinned host memory, timed on the host."""
    pairs = [(t.pin_memory(), d) for t, d in [(q, dq), (k, dk), (v, dv)] + ins]
    backs = [(torch.empty(d.shape, dtype=d.dtype, pin_memory=True), d) for d in outs]

    def once():
        with torch.cuda.stream(stream):
            for h, d in pairs:
                d.copy_(h, non_blocking=True)
            step()
            for h, d in backs:
                h.copy_(d, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        once()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(n):
        once()
    dt = reduce_max((time.perf_counter() - t0) / n, ws, dev)
    return {"value": flops * max(ws, 1) / dt / 1e12, "unit": "TFLOPS",
            "h2d_bytes_per_step": int(sum(h.numel() * h.element_size() for h, _ in pairs)),
            "d2h_bytes_per_step": int(sum(h.numel() * h.element_size() for h, _ in backs)),
            "ms_per_step": dt * 1e3, "steps": n, "api": "pinned host -> device copies, the path's Python calls, "
            "device -> pinned host copies, one stream"}


def run_ours(args, w):
    from exact_attention_attn_gb300 import attn_fwd, attn_fwd_host, attn_fwd_status, load_library

    ws, rank, local = dist_info()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    load_library()
    peaks, peak_src = load_peaks()

    q, k, v = make_workload_inputs(w)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty((w.B, w.Hq, w.Nq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    extra = path_host_inputs(args.path, w)
    step, flops, alg_bytes, e2e_ins, e2e_outs = make_step(args.path, w, dev, dq, dk, dv, out, lse, stream, extra)
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize(dev)
    st = attn_fwd_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    time.sleep(0.25)
    barrier(ws)
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)                      # L2 flush, outside the events
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    st = attn_fwd_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")

    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = statistics.mean(step_ms)
    ms = reduce_max(ms_local, ws, dev)
    value = flops * max(ws, 1) / (ms * 1e-3) / 1e12

    # roofline of the dominant (here: the only) kernel of a step: the tensor
    # pipe where the workload's FLOPs per algorithmic byte exceed the
    # machine's ridge (peak FLOP/s / HBM B/s), else HBM
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_label = f"{peak_src} bf16 dense burst"
    if args.path == "fp8":  # the measured bf16 peak times the nominal fp8 / bf16 ratio (4.5 / 2.25)
        peak *= 2.0
        peak_label = f"{peak_src} bf16 dense burst x 2 (nominal e4m3 / bf16 ratio)"
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = flops / (ms_local * 1e-3) / 1e12
    achieved_gbs = alg_bytes / (ms_local * 1e-3) / 1e9
    traffic, traffic_kernel = recorded_traffic(w.name) if args.path == "fwd" else (None, None)
    common = {"traffic": traffic, "algorithmic_flops_per_launch": flops, "algorithmic_hbm_bytes_per_launch": alg_bytes,
              "kernel": traffic_kernel}
    if args.path != "fwd":
        common["scope"] = "the whole step (" + PATHS[args.path][2] + ")"
    if flops / alg_bytes > peak * 1e3 / hbm_peak:
        roofline = dict({"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_source": peak_label,
                         "achieved_hbm_gbs": achieved_gbs}, **common)
    else:
        roofline = dict({"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved_gbs / hbm_peak, "peak_source": f"{peak_src} HBM copy",
                         "achieved_tflops": achieved, "us_per_launch": ms_local * 1e3}, **common)

    # end to end through the public API with host buffers (the forward path)
    e2e = None
    if not args.no_e2e and args.path == "fwd":
        pq, pk, pv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        po = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        pl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        for _ in range(2):
            attn_fwd_host(pq, pk, pv, scale=w.scale, causal=w.causal, device=dev, out=po, lse=pl)
        n_e2e = max(3, min(args.steps, 20))
        barrier(ws)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            attn_fwd_host(pq, pk, pv, scale=w.scale, causal=w.causal, device=dev, out=po, lse=pl)
        dt = (time.perf_counter() - t0) / n_e2e
        dt = reduce_max(dt, ws, dev)
        e2e = {"value": flops * max(ws, 1) / dt / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": int(q.numel() * 2 + k.numel() * 2 + v.numel() * 2),
               "d2h_bytes_per_step": int(out.numel() * 2 + lse.numel() * 4), "ms_per_step": dt * 1e3,
               "steps": n_e2e}
    elif not args.no_e2e:
        e2e = e2e_path(step, flops, e2e_ins, e2e_outs, q, k, v, dq, dk, dv, stream, max(3, min(args.steps, 20)),
                       ws, dev)

    cpu = None
    if rank == 0 and ws <= 1 and not args.no_cpu_baseline:
        tf, heads, dt, nrows = time_oracle(w, q, k, v, budget_s=args.cpu_seconds, path=args.path, extra=extra)
        threads = blas_threads() or cpu_cores()
        cpu = {"value": tf, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
               "sample": oracle_sample_text(w, heads, dt, nrows, threads, args.path)}
        if w.sample_rows == 0 and args.path == "fwd":  # the two small workloads: also on one host thread
            cpu["single_thread"] = single_thread_oracle(w, args.cpu_seconds)

    if rank == 0:
        metric, dtype, _ = PATHS[args.path]
        line = {
            "metric": metric or METRIC, "value": value, "unit": "TFLOPS", "n_gpus": max(ws, 1), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": dict(bench_config(w, ws), **({"path": args.path} if args.path != "fwd" else {})),
            "pct_of_peak": 100.0 * value / max(ws, 1) / peak,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * kernels_per_call(w, args.path),
            "clocks": clocks, "timed_wall_s": t_wall,
            "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms), "max": max(step_ms)},
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def kernels_per_call(w, path: str = "fwd") -> int:
    """Kernels of ours one step launches."""
    if path == "bwd":
        return 3          # prep, dK/dV, dQ
    if path == "fp8":
        return 6          # Q rows, K rows, V maxima, V codes, V scales, attention
    from exact_attention_attn_gb300.binding import attn_fwd_plan
    return attn_fwd_plan(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.causal)["launches"]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=BENCH_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--path", default="fwd", choices=list(PATHS),
                    help="what a step runs: the forward (default), the masked forward, the backward, the FP8 forward")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-only", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    w = WORKLOADS[args.workload]
    if args.oracle_only:  # the single-thread CPU leg's child process
        return oracle_only(args, w)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
