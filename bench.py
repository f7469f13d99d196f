#!/usr/bin/env python
"""Benchmark of the absorbed-form MLA split-KV decode on GB300.

One step = one ``mla_decode`` call (decode kernel + split-K combine) over one batch of the
chosen workload, with every input resident in HBM.  Prints ONE JSON line (rank 0):
KV-cache GB/s (the value), microseconds per call, TFLOP/s, the roofline fraction of the
path against the measured HBM / bf16 peaks, an end-to-end figure through the C ABI with
host buffers, the float64 CPU oracle timed on a bounded sample, and the SM clocks seen.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--window W] [--sinks] [--op decode|kv_append|absorb] [--append-tokens T]

``--window`` / ``--sinks`` time the sliding-window / attention-sink variant of the same
call.  ``--op kv_append`` times the KV-cache append with quantise-on-write instead (the
step before the decode): T new tokens (default B*q_len, one per query of the step) written
into the workload's cache in its format; its own JSON line, HBM roofline.  ``--op absorb``
times the Q absorption and V up-projection around the decode for the step's tokens.

For N > 1 it is launched by torch.distributed.run, one rank per GPU; every rank decodes
its own copy of the workload (independent replicas, weak scaling) and the slowest rank's
time is used.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/call, KV-cache GB/s and % of roofline on 1 GB300"
DEFAULT_WORKLOAD = "paged_bf16_uniform"
BYTES_PER_TOKEN = {"bf16": 1152, "fp8": 576, "nvfp4": 324}
L2_FLUSH_BYTES = 512 << 20  # > 4x the 129 MB L2


def algorithmic_work(inp, window: int = 0) -> tuple[float, float, float]:
    """(bytes, flops, kv_bytes) one decode call must move / compute at minimum: the cache
    rows of every attended position once (the union of a request's query windows), the
    queries, outputs, LSEs, the block-table entries read and seq_lens; FLOPs of QK^T (576)
    and PV (512) per attended position and query."""
    import numpy as np
    w = inp["workload"]
    sl = np.clip(inp["seq_lens"].astype(np.int64), 0, None)

    def span(L, i):  # [lo, hi) attended by query i
        hi = max(0, int(L) - w.q_len + i + 1)
        return (hi - window if window > 0 and hi > window else 0), hi

    T = sum(span(L, w.q_len - 1)[1] - span(L, 0)[0] if span(L, w.q_len - 1)[1] > 0 else 0 for L in sl)
    kv = T * BYTES_PER_TOKEN[w.kv_dtype]
    io = w.B * w.q_len * w.H * (576 * 2 + 512 * 2 + 4)
    table = 0
    for L in sl:
        lo, hi = span(L, 0)[0], span(L, w.q_len - 1)[1]
        table += (-(-hi // w.page_size) - lo // w.page_size) * 4 if hi > lo else 0
    table += 4 * w.B
    vis = sum(span(L, i)[1] - span(L, i)[0] for L in sl for i in range(w.q_len))
    flops = 2.0 * w.H * (576 + 512) * vis
    return float(kv + io + table), flops, float(kv)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def _code_tokens(text: str) -> str:
    """C++ source without comments and blank lines (string literals in these files hold no
    comment markers), so that an edit to comments alone keeps the identity of the code."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


# The decode kernel's translation unit: the kernel and every header it includes.
DECODE_SOURCES = ("mla_common.cuh", "mla_decode_tc.cu", "mla_device.cuh", "mla_ptx.cuh", "mla_tmap.cuh")


def kernel_source_sha() -> str:
    """Identity of the decode kernel's compiled code: a hash of its sources' code (comments
    excluded), which keys the ncu traffic recorded for it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_split_gb300", "csrc")
    for fn in DECODE_SOURCES:
        h.update(fn.encode())
        h.update(_code_tokens(open(os.path.join(csrc, fn)).read()).encode())
    h.update(_code_tokens(open(os.path.join(ROOT, "include", "mla_decode.h")).read()).encode())
    return h.hexdigest()[:16]


def traffic_for(workload: str):
    """ncu DRAM bytes per decode launch for this workload, if recorded for the current
    kernel sources (profiles/traffic.json); None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("source_sha") != kernel_source_sha():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=lambda: [self.lines.append(l) for l in self.proc.stdout], daemon=True)
        self.thread.start()
        # the first sample arrives a few hundred ms after the query starts: wait for it, so
        # that the sampler is live when the timed region begins
        t_end = time.time() + 3.0
        while not self.lines and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        # a timed region shorter than the 50 ms interval may hold no sample: take the next
        # one too, so that the record brackets the region
        n0, t_end = len(self.lines), time.time() + 1.0
        while len(self.lines) == n0 and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.005)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=sorted(reasons), samples=len(sm))


def cpu_oracle_sample(inp, seconds: float, start_b: int = 0, window: int = 0, sinks=None):
    """The float64 oracle, as it stands, on whole requests of the workload until `seconds`
    of CPU time have passed.  Returns (kv_bytes, elapsed, requests, rows)."""
    import oracle
    w = inp["workload"]
    kv_b, n_req, rows = 0.0, 0, 0
    t0 = time.perf_counter()
    b = start_b
    while True:
        bb = b % w.B
        oracle.mla_decode_ref(inp["q_nope"], inp["q_pe"], inp["cache"], inp["block_table"], inp["seq_lens"],
                              w.sm_scale, kv_dtype=w.kv_dtype, kv_scale=inp["kv_scale"], page_size=w.page_size,
                              rows=[(bb, i) for i in range(w.q_len)], window=window,
                              sinks=None if sinks is None else sinks.astype("float64"))
        L = max(0, int(inp["seq_lens"][bb]))
        kv_b += (min(L, window + w.q_len - 1) if window > 0 else L) * BYTES_PER_TOKEN[w.kv_dtype]
        n_req += 1
        rows += w.q_len
        b += 1
        el = time.perf_counter() - t0
        if el >= seconds or n_req >= 4 * w.B:
            return kv_b, el, n_req, rows


def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def workload_config(w, l2_note: str, window: int = 0, sinks: bool = False):
    cfg = {"workload": w.name, "B": w.B, "q_len": w.q_len, "H": w.H, "page_size": w.page_size,
           "kv_dtype": w.kv_dtype, "sm_scale": "1/sqrt(192)", "num_splits": w.num_splits or "schedule",
           "l2": l2_note}
    if window:
        cfg["window"] = window
    if sinks:
        cfg["sinks"] = "per head, uniform in [0, 12], every 8th head -inf, head 1 at 32 (seeded)"
    if w.seq_len is not None:
        cfg["seq_len"] = w.seq_len
    if w.ragged is not None:
        cfg["seq_lens"] = f"uniform integers in [{w.ragged[0]}, {w.ragged[1]}], seed {w.seed}"
    return cfg


def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over all ranks (the slowest rank's times), or the
    values themselves with one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job throughput: every rank processes its own copy of the workload (weak
    scaling), so the job moves world x the per-rank units in the slowest rank's time."""
    return world * units_per_rank / seconds


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def run_reference(args):
    """The float64 CPU oracle, timed on this host's cores, on bounded samples of the same
    workload: one request per step."""
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return
    from mla_latent_kv_split_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w)
    if args.op != "decode":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the decode only"}), flush=True)
        return
    sinks = W.draw_sinks(w.H, seed=0) if args.sinks else None
    for s in range(args.warmup):
        cpu_oracle_sample(inp, 0.0, start_b=s, window=args.window, sinks=sinks)
    t_steps, kv_total, rows_total = [], 0.0, 0
    for s in range(args.steps):
        kv_b, el, n_req, rows = cpu_oracle_sample(inp, 0.0, start_b=args.warmup + s, window=args.window, sinks=sinks)
        t_steps.append(el)
        kv_total += kv_b
        rows_total += rows
    total = sum(t_steps)
    value = kv_total / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, "n/a (CPU)", args.window, args.sinks),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
                         "sample": f"one whole request (all {w.q_len} queries, {w.H} heads) per step, "
                                   f"{args.steps} steps, {rows_total} (b,i) rows"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _roofline(nbytes: float, flops: float, t_s: float, peaks: dict) -> dict:
    t_mem = nbytes / (peaks["hbm"] * 1e9)
    t_mma = flops / (peaks["bf16"] * 1e12)
    if t_mem >= t_mma:
        roof = {"bound": "hbm", "achieved": nbytes / t_s / 1e9, "peak": peaks["hbm"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / t_s / 1e12, "peak": peaks["bf16"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = peaks["source"]
    roof["roofline_us"] = 1e6 * max(t_mem, t_mma)
    return roof


class DecodeCase:
    """One workload resident on the device, with a bound ``call()`` of ``mla_decode``."""

    def __init__(self, w, inp, dev, window: int = 0, h_sinks=None):
        import numpy as np
        import torch
        from mla_latent_kv_split_gb300 import binding as mb

        self.w, self.inp, self.dev, self.window = w, inp, dev, window

        def to_dev(a, bf16=False):
            t = torch.from_numpy(a.view(np.int16) if bf16 else a)
            return (t.view(torch.bfloat16) if bf16 else t).to(dev)

        self.q_nope = to_dev(inp["q_nope"], True)
        self.q_pe = to_dev(inp["q_pe"], True)
        self.cache = to_dev(inp["cache"], inp["cache"].dtype == np.uint16)
        self.table = to_dev(inp["block_table"])
        self.seq_lens = to_dev(inp["seq_lens"])
        self.ws = mb.alloc_workspace(w.B, w.q_len, w.H, w.num_splits, dev)
        self.out = torch.empty((w.B, w.q_len, w.H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.q_len, w.H), dtype=torch.float32, device=dev)
        self.sinks = None if h_sinks is None else torch.from_numpy(h_sinks).to(dev)
        self.stream = torch.cuda.current_stream(dev)

    def call(self, q_nope=None, q_pe=None, table=None, seq_lens=None, out=None, lse=None):
        from mla_latent_kv_split_gb300 import binding as mb
        w = self.w
        mb.mla_decode(self.q_nope if q_nope is None else q_nope, self.q_pe if q_pe is None else q_pe, self.cache,
                      self.table if table is None else table, self.seq_lens if seq_lens is None else seq_lens,
                      w.sm_scale, w.kv_dtype, self.inp["kv_scale"], w.num_splits, page_size=w.page_size,
                      num_pages=self.inp["num_pages"], workspace=self.ws, out=self.out if out is None else out,
                      lse=self.lse if lse is None else lse, stream=self.stream, window=self.window, sinks=self.sinks)


def make_l2_flush(dev):
    import torch
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_head = flush[: flush.numel() // 2]

    def l2_flush():
        # Write 512 MB (evicts every line of the call's inputs and outputs), then read the
        # first 256 MB back so that the lines left in L2 are clean: the timed call then does
        # not pay for writing back the flush buffer's dirty lines.
        flush.zero_()
        flush_head.sum()
    return l2_flush


def time_calls(case, l2_flush, steps: int, warmup: int, barrier=None, prewarm=None):
    """Warm-up calls, then `steps` calls each timed with CUDA events on the launching stream,
    L2 flushed before each.  `prewarm` (untimed, after the flush) is a call on other, small
    inputs that brings the kernels' instructions back into L2 while leaving the timed call's
    data cold.  Returns (times in ms, device status of the last call)."""
    import torch
    from mla_latent_kv_split_gb300 import binding as mb
    t_warm = time.perf_counter()
    k = 0
    while k < max(3, warmup) or time.perf_counter() - t_warm < 0.3:
        l2_flush()
        case.call()
        torch.cuda.synchronize()
        k += 1
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if barrier:
        barrier()
    torch.cuda.synchronize()
    for s in range(steps):
        l2_flush()
        if prewarm is not None:
            prewarm()
        evs[s][0].record(case.stream)
        case.call()
        evs[s][1].record(case.stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    # the status word of the last timed call; a call that hit a bounded wait shows as a
    # time outlier (the waits give up after seconds)
    status = mb.mla_decode_read_status(case.ws)
    times_ms = [a.elapsed_time(b) for a, b in evs]
    if status or max(times_ms) > 20 * statistics.median(times_ms):
        print(f"bench.py: {case.w.name}: device status {status:#x}, slowest call {max(times_ms):.3f} ms",
              file=sys.stderr)
    return times_ms, status


def pipelined_steps_ms(cases, h_in, d_in, d_res, offs, srcs, inp, w, out_bytes, warmup: int, steps: int, ref_res):
    """Consecutive end-to-end steps as a serving loop runs them: two sets of device input
    and result buffers; step k's inputs are copied in on one stream, its call (on
    cases[k % 2]: two copies of the same cache, as consecutive layers have two caches) runs
    on the call's stream, its results are copied back on a third; a buffer set is reused
    only once the call (inputs) or the copy back (results) of step k - 2 is done with it.
    Returns the mean time per step of `steps` steps after `warmup` untimed ones (one pair
    of CUDA events around all of them).  The copied-back results are checked afterwards."""
    import torch
    dev = d_in.device
    d_ins = [d_in, torch.empty_like(d_in)]
    d_ress = [d_res, torch.empty_like(d_res)]
    h_ress = [torch.empty(d_res.numel(), dtype=torch.uint8).pin_memory() for _ in range(2)]

    def views(j):
        sl = lambda i: d_ins[j][int(offs[i]):int(offs[i]) + srcs[i].size]
        r = d_ress[j]
        return (sl(0).view(torch.bfloat16).view(inp["q_nope"].shape), sl(1).view(torch.bfloat16).view(inp["q_pe"].shape),
                sl(2).view(torch.int32).view(inp["block_table"].shape), sl(3).view(torch.int32).view(inp["seq_lens"].shape),
                r[:out_bytes].view(torch.bfloat16).view(w.B, w.q_len, w.H, 512),
                r[(out_bytes + 255) // 256 * 256:].view(torch.float32).view(w.B, w.q_len, w.H))

    bufs = [views(0), views(1)]
    comp = cases[0].stream
    assert all(c.stream == comp for c in cases)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        in_free, res_free = [None, None], [None, None]
        for k in range(n):
            j = k & 1
            if in_free[j] is not None:
                s_in.wait_event(in_free[j])
            with torch.cuda.stream(s_in):
                d_ins[j].copy_(h_in, non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(s_in)
            comp.wait_event(e_in)
            if res_free[j] is not None:
                comp.wait_event(res_free[j])
            cases[j].call(*bufs[j])
            e_call = torch.cuda.Event()
            e_call.record(comp)
            in_free[j] = e_call
            s_out.wait_event(e_call)
            with torch.cuda.stream(s_out):
                h_ress[j].copy_(d_ress[j], non_blocking=True)
            e_out = torch.cuda.Event()
            e_out.record(s_out)
            res_free[j] = e_out

    torch.cuda.synchronize()
    run(warmup)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    run(steps)
    b.record(s_out)
    torch.cuda.synchronize()
    # every step had the same inputs: both buffer sets hold the serial run's results
    lse_at = (out_bytes + 255) // 256 * 256
    for h in h_ress[: min(2, steps)]:
        assert torch.equal(h[:out_bytes], ref_res[:out_bytes]) and torch.equal(h[lse_at:], ref_res[lse_at:])
    return a.elapsed_time(b) / steps


def cpu_baseline_entry(inp, seconds: float, window: int = 0, sinks=None) -> dict:
    w = inp["workload"]
    cpu_kv, cpu_el, cpu_req, cpu_rows = cpu_oracle_sample(inp, seconds, window=window, sinks=sinks)
    return {"value": cpu_kv / cpu_el / 1e9, "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"{cpu_req} whole requests ({cpu_rows} (b,i) rows x {w.H} heads) of the same "
                      f"workload, {cpu_el:.1f} s, float64 NumPy"}


def measure_config(name: str, dev, l2_flush, steps: int, warmup: int, cpu_seconds: float, index: int) -> dict:
    """All of one workload's figures, measured in this run: µs per call (mean, median,
    max), KV GB/s, TFLOP/s, the roofline fraction, ncu DRAM traffic when recorded for these
    kernel sources, the SM clocks seen while timing, and the oracle on a bounded sample."""
    import torch
    from mla_latent_kv_split_gb300 import workloads as W
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    nbytes, flops, kv_bytes = algorithmic_work(inp)
    case = DecodeCase(w, inp, dev)
    sampler = ClockSampler(index)
    sampler.start()
    times_ms, status = time_calls(case, l2_flush, steps, warmup)
    clocks = sampler.stop()
    # the same calls with the kernels' instructions resident (a 1-request call of the same
    # shape class on its own inputs after each flush, which takes the same decode kernel:
    # at most 1024 positions, the workload's own length if shorter): as in a decode loop,
    # where the kernels run every layer; the timed call's data stays cold
    warm_len = min(w.seq_len, 1024) if w.seq_len else 1024
    tw = w.scaled(B=1, seq_lens_override=(warm_len,))
    tiny = DecodeCase(tw, W.make_inputs(tw), dev)
    warm_ms, _ = time_calls(case, l2_flush, steps, 3, prewarm=tiny.call)
    del case, tiny
    torch.cuda.empty_cache()
    t_s = sum(times_ms) / len(times_ms) * 1e-3
    roof = _roofline(nbytes, flops, t_s, load_peaks())
    roof["traffic"] = traffic_for(name)
    return {
        "config": workload_config(w, "flushed between steps"),
        "us_per_call": 1e6 * t_s, "us_per_call_median": 1e3 * statistics.median(times_ms),
        "us_per_call_max": 1e3 * max(times_ms), "steps": len(times_ms),
        "us_per_call_code_warm": 1e3 * statistics.mean(warm_ms),
        "kv_gbs": kv_bytes / t_s / 1e9, "tflops": flops / t_s / 1e12,
        "algorithmic_bytes": nbytes, "algorithmic_flops": flops, "device_status": status,
        "roofline": roof, "clocks": clocks, "gpu_launches": 2 * len(times_ms),
        "cpu_baseline": cpu_baseline_entry(inp, cpu_seconds),
    }


def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_setup(args.gpus)
    from mla_latent_kv_split_gb300 import binding as mb
    from mla_latent_kv_split_gb300 import build
    from mla_latent_kv_split_gb300 import workloads as W

    if rank == 0:
        build.build()
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        barrier = dist.barrier
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w)
    if args.op == "kv_append":
        return run_append(args, w, inp, world, rank, dev)
    if args.op == "absorb":
        return run_absorb(args, w, world, rank, dev)
    nbytes, flops, kv_bytes = algorithmic_work(inp, args.window)
    h_sinks = W.draw_sinks(w.H, seed=0) if args.sinks else None
    case = DecodeCase(w, inp, dev, args.window, h_sinks)
    l2_flush = make_l2_flush(dev)
    stream = case.stream
    smi_index = local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0

    sampler = ClockSampler(smi_index)
    sampler.start()
    times_ms, status = time_calls(case, l2_flush, args.steps, args.warmup, barrier)
    clocks = sampler.stop()
    t_mean = sum(times_ms) / len(times_ms)

    # end to end through the C ABI with host buffers: the step's inputs staged in one pinned
    # buffer (256-byte aligned segments) and copied in with one copy; out and lse written into
    # one device buffer and copied back with one copy (each copy has a fixed cost)
    seg = lambda n: (n + 255) // 256 * 256
    srcs = [inp["q_nope"].view(np.uint8).reshape(-1), inp["q_pe"].view(np.uint8).reshape(-1),
            inp["block_table"].view(np.uint8).reshape(-1), inp["seq_lens"].view(np.uint8).reshape(-1)]
    offs = np.cumsum([0] + [seg(a.size) for a in srcs])
    h_in = torch.empty(int(offs[-1]), dtype=torch.uint8).pin_memory()
    for a, o in zip(srcs, offs[:-1]):
        h_in[int(o):int(o) + a.size].copy_(torch.from_numpy(a))
    d_in = torch.empty_like(h_in, device=dev)
    sl = lambda i: d_in[int(offs[i]):int(offs[i]) + srcs[i].size]
    d_qn = sl(0).view(torch.bfloat16).view(inp["q_nope"].shape)
    d_qp = sl(1).view(torch.bfloat16).view(inp["q_pe"].shape)
    d_bt = sl(2).view(torch.int32).view(inp["block_table"].shape)
    d_sl = sl(3).view(torch.int32).view(inp["seq_lens"].shape)
    out_bytes, lse_bytes = w.B * w.q_len * w.H * 512 * 2, w.B * w.q_len * w.H * 4
    d_res = torch.empty(seg(out_bytes) + lse_bytes, dtype=torch.uint8, device=dev)
    d_out = d_res[:out_bytes].view(torch.bfloat16).view(w.B, w.q_len, w.H, 512)
    d_lse = d_res[seg(out_bytes):].view(torch.float32).view(w.B, w.q_len, w.H)
    h_res = torch.empty_like(d_res, device="cpu").pin_memory()
    h2d, d2h = h_in.numel(), h_res.numel()
    # (1) one step at a time: L2 flushed, the inputs copied in, the call, the results copied
    # back, all on the call's stream, synchronised after each step
    serial_ms = []
    for s in range(args.warmup + args.steps):
        l2_flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        d_in.copy_(h_in, non_blocking=True)
        case.call(d_qn, d_qp, d_bt, d_sl, d_out, d_lse)
        h_res.copy_(d_res, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if s >= args.warmup:
            serial_ms.append(a.elapsed_time(b))
    # the copied-back results are the call's (a check, outside the timed region)
    ref_res = d_res.cpu()
    assert torch.equal(h_res[:out_bytes].view(torch.int16), d_out.view(torch.int16).cpu().reshape(-1))
    serial_mean = sum(serial_ms) / len(serial_ms)
    # the pipelined loop alternates two copies of the cache (as consecutive layers would), so
    # that no cache row is found in L2 from the step before
    case_b = DecodeCase(w, inp, dev, args.window, h_sinks)
    e2e_mean = pipelined_steps_ms([case, case_b], h_in, d_in, d_res, offs, srcs, inp, w, out_bytes, args.warmup,
                                  args.steps, ref_res)
    del case_b

    t_mean, e2e_mean = max_over_ranks([t_mean, e2e_mean], dev)
    if rank != 0:
        dist.destroy_process_group()
        return

    peaks = load_peaks()
    t_s = t_mean * 1e-3
    roof = _roofline(nbytes, flops, t_s, peaks)
    roof["traffic"] = traffic_for(w.name) if not (args.window or args.sinks) else None
    roof["kernel"] = "mla_decode call (decode kernel + split-K combine)"
    del case
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": job_rate(kv_bytes, t_s, world) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_mean, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, "flushed between steps (512 MB write, then 256 MB read so no dirty lines remain)",
                                  args.window, args.sinks),
        "us_per_call": 1e3 * t_mean, "us_per_call_median": 1e3 * statistics.median(times_ms),
        "us_per_call_max": 1e3 * max(times_ms),
        "kv_gbs": kv_bytes / t_s / 1e9, "tflops": flops / t_s / 1e12,
        "algorithmic_bytes": nbytes, "algorithmic_flops": flops, "device_status": status,
        "roofline": roof,
        "cpu_baseline": cpu_baseline_entry(inp, args.cpu_seconds, args.window, h_sinks),
        "e2e": {"value": job_rate(kv_bytes, e2e_mean * 1e-3, world) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_mean,
                "serial": {"value": job_rate(kv_bytes, serial_mean * 1e-3, world) / 1e9, "ms_per_step": serial_mean},
                "note": "every step copies q_nope, q_pe, block_table, seq_lens in from one pinned host buffer "
                        "(one copy) and out, lse back from one device buffer (one copy); the KV cache is "
                        "resident device state.  value: consecutive steps as a serving loop runs them, "
                        "double-buffered, the next step's inputs copied in on one stream and the previous "
                        "step's results copied back on another while the current call runs; total time of "
                        "the timed steps / steps; no L2 flush: consecutive steps read two copies of the cache "
                        "in turn (as consecutive layers do; 2 x the cache, more than L2 holds), the kernels' "
                        "instructions stay resident.  serial: each step alone, L2 flushed before it, copies "
                        "and call on one stream"},
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,
    }
    if args.configs == "all" and world == 1 and not (args.window or args.sinks):
        # every workload of the path, each timed in this same run (the headline one again,
        # so that each entry comes from one uniform procedure)
        line["configs"] = {name: measure_config(name, dev, l2_flush, args.steps, args.warmup,
                                                min(args.cpu_seconds, 3.0), smi_index)
                           for name in W.WORKLOADS}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def append_cpu_baseline(x, cache_np, w, inp, seconds):
    """The append oracle, as it stands, on the batch's tokens 64 at a time for a bounded time,
    each chunk written into one page of a cache of the same format (the oracle returns a
    copy of the cache it is given, so the sample's cache is kept to one page); GB/s of the
    same algorithmic bytes per token."""
    import numpy as np
    from oracle import kv_append_ref
    bits = x.view(torch_int16()).cpu().numpy().view(np.uint16)
    page = np.zeros_like(cache_np[:1])
    n, T = 0, bits.shape[0]
    t0 = time.perf_counter()
    while n < T and (n == 0 or time.perf_counter() - t0 < seconds):
        k = min(T - n, w.page_size)
        kv_append_ref.kv_append_ref(page, bits[n:n + k, :512], bits[n:n + k, 512:], np.arange(k), w.kv_dtype,
                                    w.page_size, inp["kv_scale"])
        n += k
    el = time.perf_counter() - t0
    per_tok = 1152 + BYTES_PER_TOKEN[w.kv_dtype] + 8
    return {"value": n * per_tok / el / 1e9, "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"{n} tokens of the same batch, {el:.2f} s, NumPy"}


def absorb_cpu_baseline(q_raw, w_ukT, o_lat, w_uv, nbytes, seconds):
    """The projection oracle (float64) on both projections of the same tensors, once."""
    import numpy as np
    from oracle import absorb_ref
    b = lambda t: t.contiguous().view(torch_int16()).cpu().numpy().view(np.uint16)
    xq, wq, xo, wo = b(q_raw[:, :, :128]), b(w_ukT), b(o_lat), b(w_uv)
    t0 = time.perf_counter()
    absorb_ref.batched_gemv_ref(xq, wq)
    absorb_ref.batched_gemv_ref(xo, wo)
    el = time.perf_counter() - t0
    return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"both projections of the same step once, {el:.2f} s, float64 NumPy"}


def torch_int16():
    import torch
    return torch.int16


def run_append(args, w, inp, world, rank, dev):
    """The KV-cache append with quantise-on-write: T new tokens (bf16 [T, 576]) written to
    distinct locations of the workload's cache, in its format.  Algorithmic bytes per token:
    1152 read + the stored bytes (1152 / 576 / 324) + 8 for the location."""
    import numpy as np
    import torch
    from mla_latent_kv_split_gb300 import binding as mb

    T = args.append_tokens or w.B * w.q_len
    cache_np = inp["cache"]
    num_pages, ps = inp["num_pages"], w.page_size
    if T > num_pages * ps:
        raise SystemExit(f"--append-tokens {T} exceeds the cache's {num_pages * ps} locations")
    g = torch.Generator().manual_seed(5)
    x = (torch.randn((T, 576), generator=g) * 2).to(torch.bfloat16).to(dev)
    slots = torch.randperm(num_pages * ps, generator=g)[:T].to(torch.int64).to(dev)
    cache = torch.from_numpy(cache_np.view(np.int16) if cache_np.dtype == np.uint16 else cache_np).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_head = flush[: flush.numel() // 2]
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        mb.mla_kv_append(x[:, :512], x[:, 512:], slots, cache, page_size=ps, kv_dtype=w.kv_dtype,
                         kv_scale=inp["kv_scale"], num_pages=num_pages, device_status=status, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        flush_head.sum()
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for s in range(args.steps):
        flush.zero_()
        flush_head.sum()
        evs[s][0].record(stream)
        call()
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    times_ms = [a.elapsed_time(b) for a, b in evs]
    t_mean = max_over_ranks([sum(times_ms) / len(times_ms)], dev)[0]
    if rank != 0:
        return
    nbytes = T * (1152 + BYTES_PER_TOKEN[w.kv_dtype] + 8)
    peaks = load_peaks()
    achieved = nbytes / (t_mean * 1e-3) / 1e9
    line = {
        "metric": "KV-cache append with quantise-on-write, GB/s of algorithmic bytes",
        "value": job_rate(nbytes, t_mean * 1e-3, world) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_mean,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
        "config": {"workload": w.name, "op": "kv_append", "tokens": T, "kv_dtype": w.kv_dtype, "page_size": ps,
                   "l2": "flushed between steps"},
        "us_per_call": 1e3 * t_mean, "us_per_call_median": 1e3 * statistics.median(times_ms),
        "us_per_call_max": 1e3 * max(times_ms),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm"], "traffic": None, "peak_source": peaks["source"],
                     "kernel": "mla_kv_append_kernel"},
        "device_status": int(status.item()), "clocks": clocks, "gpu_launches": args.steps,
        "cpu_baseline": append_cpu_baseline(x, cache_np, w, inp, args.cpu_seconds),
    }
    print(json.dumps(line), flush=True)


def run_absorb(args, w, world, rank, dev):
    """The two per-head projections around the decode for the step's T = B*q_len tokens:
    Q absorption (q_nope [T, H, 128] read out of [T, H, 192] raw query rows, W_UK^T
    [H, 512, 128]) and V up-projection (o_lat [T, H, 512], W_UV [H, 128, 512]).  One step =
    both launches.  Algorithmic bytes: both weights once plus every activation read and
    written once."""
    import torch
    from mla_latent_kv_split_gb300 import binding as mb

    T, H = w.B * w.q_len, w.H
    g = torch.Generator().manual_seed(3)
    bf = lambda shape, sc=1.0: (torch.randn(shape, generator=g) * sc).to(torch.bfloat16).to(dev)
    q_raw = bf((T, H, 192))
    w_ukT = bf((H, 512, 128), 128 ** -0.5)
    o_lat = bf((T, H, 512), 0.2)
    w_uv = bf((H, 128, 512), 512 ** -0.5)
    q_lat = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    o = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_head = flush[: flush.numel() // 2]
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        mb.mla_batched_gemv(q_raw[:, :, :128], w_ukT, out=q_lat, device_status=status, stream=stream)
        mb.mla_batched_gemv(o_lat, w_uv, out=o, device_status=status, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        flush_head.sum()
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for s in range(args.steps):
        flush.zero_()
        flush_head.sum()
        evs[s][0].record(stream)
        call()
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    times_ms = [a.elapsed_time(b) for a, b in evs]
    t_mean = max_over_ranks([sum(times_ms) / len(times_ms)], dev)[0]
    if rank != 0:
        return
    nbytes = 2 * H * 512 * 128 * 2 + 2 * T * H * (128 + 512) * 2
    flops = 2 * 2.0 * T * H * 512 * 128
    peaks = load_peaks()
    achieved = nbytes / (t_mean * 1e-3) / 1e9
    line = {
        "metric": "MLA Q absorption + V up-projection (per-head batched GEMV), GB/s of algorithmic bytes",
        "value": job_rate(nbytes, t_mean * 1e-3, world) / 1e9, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_mean, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "op": "absorb", "tokens": T, "H": H, "nope": 128, "latent": 512, "v": 128,
                   "l2": "flushed between steps"},
        "us_per_call": 1e3 * t_mean, "us_per_call_median": 1e3 * statistics.median(times_ms),
        "us_per_call_max": 1e3 * max(times_ms), "tflops": flops / (t_mean * 1e-3) / 1e12,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm"], "traffic": None, "peak_source": peaks["source"],
                     "kernel": "mla_batched_gemv_kernel x2"},
        "device_status": int(status.item()), "clocks": clocks, "gpu_launches": 2 * args.steps,
        "cpu_baseline": absorb_cpu_baseline(q_raw, w_ukT, o_lat, w_uv, nbytes, args.cpu_seconds),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--window", type=int, default=0, help="sliding window (0: none)")
    ap.add_argument("--sinks", action="store_true", help="per-head attention sinks")
    ap.add_argument("--op", default="decode", choices=["decode", "kv_append", "absorb"])
    ap.add_argument("--append-tokens", type=int, default=0, help="kv_append: tokens per call (default B*q_len)")
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="decode: also time every workload in this run (one entry per workload under 'configs')")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
