#!/usr/bin/env python
"""Benchmark of one paged decode step (libpagedattn.pa_decode) on GB300.

A bench step is one pa_decode call over the whole batch of the named workload (inputs
resident in HBM; default: the ragged serving mix, the largest configuration), with L2
flushed before every step, outside the timed interval: a 256 MiB write evicts every line,
then a 256 MiB read replaces the write's dirty lines with clean ones, so the timed kernel
neither finds its inputs in L2 nor pays for the flush's own write-back. Prints one JSON line
(rank 0): KV-cache read GB/s, microseconds per call, the roofline of the decode kernel
against the measured HBM copy bandwidth, SM clocks sampled during the timed region, an
end-to-end figure through the C ABI with every step's inputs copied from pinned host memory
and its output copied back, and the CPU oracle timed on the host cores. The other full-size
decode workloads follow as complete blocks of their own (steps, roofline, clocks, e2e), then
the multi-token kernel's lines.

``--impl reference`` times the CPU oracle itself (there is no runnable reference library
for this method) on the same workload and metric.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV-read GB/s (% of HBM peak) and μs per call"
DEFAULT_WORKLOAD = "ragged"
PREFILL_WORKLOADS = ("prefill_gqa4", "prefill_chunked", "prefill_mha", "prefill_gqa6_hd256")
# the library's other kernels, each timed alone on a full-size workload by --kernel-case
KERNEL_CASES = ("append", "split_combine", "prefill_hd256")
# the other full-size decode workloads, each measured into a block of its own
OTHER_WORKLOADS = ("gqa4_mid", "mha", "long_gqa6")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
L2_FLUSH_NOTE = ("flushed before every step, outside the timed interval: 256 MiB write, then a "
                 "256 MiB read so the write's dirty lines are written back before the interval")


class L2Flush:
    """Evicts L2 (129 MB on GB300) between timed steps. The write alone would leave L2 full
    of dirty lines whose write-back then lands inside the next timed kernel; the read after
    it turns them into clean lines of a buffer no kernel under test touches."""

    def __init__(self, torch):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.sum()
KERNEL_SOURCES = ["device_common.cuh", "decode_kernel.cuh", "decode_launch.cuh", "internal.h",
                  "api.cpp", "launch.cu"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-others", action="store_true",
                    help="skip the blocks of the other decode workloads and the prefill lines")
    ap.add_argument("--layout", choices=["token_major", "head_major"], default="token_major",
                    help="K/V cache layout of the timed workload: [page][slot][kv_head][hd] (the "
                         "pages') or [page][kv_head][slot][hd]")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the multi-token kernel on its workloads (one JSON line)")
    ap.add_argument("--kernel-case", choices=KERNEL_CASES,
                    help="time one other library kernel alone on a full-size workload (one JSON "
                         "line): the K/V append on ragged, the fixed split's partial and combine "
                         "kernels on long_gqa6, or the head_dim-256 multi-token kernel")
    ap.add_argument("--splits", type=int, default=64,
                    help="splits per sequence of the split_combine case")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work for the oracle baseline sample")
    ap.add_argument("--math", default="auto")
    ap.add_argument("--schedule", default="auto")
    ap.add_argument("--combine", default="auto")
    ap.add_argument("--workers", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--warps", type=int, default=0)
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_of(text: str) -> str:
    """C/C++/CUDA source without comments, whitespace runs collapsed to one space (string
    literals kept), so that a comment edit leaves a recorded capture valid while a code
    change invalidates it."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c.isspace():
            if out and out[-1] != " ":
                out.append(" ")
            i += 1
        else:
            out.append(c)
            i += 1
    return "".join(out).strip()


def kernel_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_63_gb300", "csrc", name)) as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on the current
    kernel sources (profiles/traffic.json maps workload -> {kernel_hash, dram_bytes})."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_hash") != kernel_hash():
        return None
    return float(rec["dram_bytes_per_launch"])


def algorithmic_bytes(w) -> dict:
    ctx = w.context_lengths.astype(np.int64).clip(min=0)
    kv = int(ctx.sum()) * w.kv_heads * w.head_dim * 2 * 2
    q = w.batch * w.query_heads * w.head_dim * 2
    out = w.batch * w.query_heads * w.head_dim * 4
    bt = int((-(-ctx // w.page_size)).sum()) * 4 + w.batch * 4
    return dict(kv=kv, total=kv + q + out + bt, h2d=q + w.block_tables.nbytes + ctx.size * 4,
                d2h=out)


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, busy_from: float = 0.0) -> dict:
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 8:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v == "Active"})
        load = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(sm)}


def to_device(w, torch):
    return dict(q=torch.from_numpy(w.query).cuda(), k=torch.from_numpy(w.key_cache).cuda(),
                v=torch.from_numpy(w.value_cache).cuda(), bt=torch.from_numpy(w.block_tables).cuda(),
                ctx=torch.from_numpy(w.context_lengths).cuda(),
                out=torch.empty((w.batch, w.query_heads, w.head_dim), dtype=torch.float32,
                                device="cuda"))


def time_decode(w, d, opts, steps, warmup, torch, lib, sampler_dev=None):
    """Per-step CUDA-event times (ms) of pa_decode_ex, L2 flushed before each step."""
    prob = lib.problem_of(w)
    n = lib.pa_workspace_size(prob, opts)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
    lib.pa_workspace_init(ws, n)
    flush = L2Flush(torch)
    stream = torch.cuda.current_stream()

    def step():
        lib.pa_decode_ex(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"], w.scale, d["out"], opts,
                         ws if n else None, n, stream.cuda_stream)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    world, _, _ = dist_env()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(sampler_dev) if sampler_dev is not None else None
    if sampler:
        sampler.__enter__()
    t0 = time.perf_counter()
    for i in range(steps):
        flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    if sampler:
        sampler.__exit__(None, None, None)
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    clocks = sampler.summary() if sampler else None
    return ms, wall, clocks


def time_e2e(w, d, opts, steps, warmup, torch, lib):
    """End-to-end throughput through the C ABI with the per-step inputs in pinned host memory:
    every step copies its query, block table and context lengths host-to-device, decodes, and
    copies its output back. The copies run on two copy streams and the decode on the compute
    stream, with two device input/output buffers, so step i's copies overlap the decode of
    steps i - 1 and i + 1, as a serving loop would run them. Returns (ms per step over the
    whole pipelined run, ms of one step run alone: upload, decode, download)."""
    prob = lib.problem_of(w)
    n = lib.pa_workspace_size(prob, opts)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
    lib.pa_workspace_init(ws, n)
    parts = [w.query.view(np.uint8).reshape(-1), w.block_tables.view(np.uint8).reshape(-1),
             w.context_lengths.view(np.uint8).reshape(-1)]
    offs, total = [], 0
    for p in parts:
        offs.append(total)
        total += (p.size + 255) // 256 * 256
    packed = torch.empty(total, dtype=torch.uint8).pin_memory()
    for p, o in zip(parts, offs):
        packed[o:o + p.size] = torch.from_numpy(p)
    bufs = []
    for _ in range(2):
        dev = torch.empty(total, dtype=torch.uint8, device="cuda")
        bufs.append(dict(dev=dev, q=dev[offs[0]:offs[0] + parts[0].size],
                         bt=dev[offs[1]:offs[1] + parts[1].size],
                         ctx=dev[offs[2]:offs[2] + parts[2].size],
                         out=torch.empty_like(d["out"]),
                         host_out=torch.empty(d["out"].shape, dtype=torch.float32).pin_memory(),
                         uploaded=torch.cuda.Event(), decoded=torch.cuda.Event(),
                         downloaded=torch.cuda.Event()))
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def run(count):
        for b in bufs:  # both buffers free at the start
            b["decoded"].record(comp)
            b["downloaded"].record(comp)
        for i in range(count):
            b = bufs[i % 2]
            with torch.cuda.stream(up):
                up.wait_event(b["decoded"])  # the decode two steps back has read this buffer
                b["dev"].copy_(packed, non_blocking=True)
                b["uploaded"].record(up)
            comp.wait_event(b["uploaded"])
            comp.wait_event(b["downloaded"])  # its output buffer has been read back
            lib.pa_decode_ex(prob, b["q"], d["k"], d["v"], b["bt"], b["ctx"], w.scale, b["out"],
                             opts, ws if n else None, n, comp.cuda_stream)
            b["decoded"].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(b["decoded"])
                b["host_out"].copy_(b["out"], non_blocking=True)
                b["downloaded"].record(down)
        comp.wait_event(bufs[(count - 1) % 2]["downloaded"])
        if count > 1:
            comp.wait_event(bufs[count % 2]["downloaded"])

    run(max(warmup, 2))
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    run(steps)
    t1.record(comp)
    torch.cuda.synchronize()
    pipelined = t0.elapsed_time(t1) / steps
    serial = []
    for _ in range(5):
        torch.cuda.synchronize()
        t0.record(comp)
        run(1)
        t1.record(comp)
        torch.cuda.synchronize()
        serial.append(t0.elapsed_time(t1))
    return pipelined, statistics.median(serial)


def measured_tensor_peak():
    """Dense fp16/bf16 tensor peak (TFLOP/s): the measured bf16 GEMM burst figure (fp16 and
    bf16 share one dense rate on these tensor cores)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def time_prefill(p, steps, warmup, torch, lib):
    """Mean CUDA-event time (ms) of one pa_prefill call, L2 flushed before each call."""
    w = p.cache
    d = [torch.from_numpy(x).cuda() for x in (p.query, p.query_start, w.key_cache, w.value_cache,
                                               w.block_tables, w.context_lengths)]
    out = torch.empty((p.total, w.query_heads, w.head_dim), dtype=torch.float32, device="cuda")
    flush = L2Flush(torch)
    prob = lib.problem_of(w)
    stream = torch.cuda.current_stream()

    def step():
        lib.pa_prefill(prob, d[0], d[1], p.total, p.max_query_len(), d[2], d[3], d[4], d[5],
                       w.scale, out, None, stream.cuda_stream)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    return sum(ms) / len(ms)


def prefill_lines(torch, lib, steps):
    """The multi-token (prefill) kernel on its workloads, against the dense tensor peak."""
    from paged_kv_cache_63_gb300.workloads import make_prefill

    peak, kind = measured_tensor_peak()
    res = {}
    for name in PREFILL_WORKLOADS:
        p = make_prefill(name)
        ms = time_prefill(p, steps, 5, torch, lib)
        assert lib.pa_get_device_error() == 0
        flops = 4.0 * p.causal_pairs() * p.cache.query_heads * p.cache.head_dim
        tf = flops / (ms * 1e-3) / 1e12
        res[name] = {"us_per_call": round(ms * 1e3, 1), "tflops": round(tf, 1),
                     "causal_flops": flops,
                     "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak,
                                  "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                                  "peak_source": f"{kind} (bf16 GEMM burst; fp16 same rate)",
                                  "kernel": ("pa::prefill2_kernel" if p.cache.head_dim <= 128
                                             else "pa::prefill_kernel")}}
        torch.cuda.empty_cache()
    return res


def reduce_over_ranks(torch, device, maxima, sums):
    """Whole-job figures for weak scaling: the slowest rank's times (max over ranks) and the
    bytes all ranks moved (sum). With one process the values pass through."""
    t_max = torch.tensor([float(x) for x in maxima], dtype=torch.float64, device=device)
    t_sum = torch.tensor([float(x) for x in sums], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized() and \
            torch.distributed.get_world_size() > 1:
        torch.distributed.all_reduce(t_max, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(t_sum, op=torch.distributed.ReduceOp.SUM)
    return t_max.tolist(), t_sum.tolist()


def cpu_baseline(w, seconds: float) -> dict:
    """The fp64 oracle on the host cores over a bounded sample of the same workload: all
    query heads of a subset of sequences (calibrated to about `seconds` of work)."""
    import oracle

    oracle.build()
    g = w.query_heads
    order = np.argsort(w.context_lengths)[::-1]
    b0 = int(order[len(order) // 2])  # a median-length sequence to calibrate on
    t0 = time.perf_counter()
    oracle.decode(w, rows=np.arange(b0 * g, (b0 + 1) * g))
    t_one = max(time.perf_counter() - t0, 1e-4)
    n_seq = int(max(1, min(w.batch, seconds / t_one)))
    rng = np.random.default_rng(7)
    seqs = np.sort(rng.choice(w.batch, size=n_seq, replace=False))
    rows = np.concatenate([np.arange(b * g, (b + 1) * g) for b in seqs])
    cores = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.decode(w, rows=rows)
    dt = time.perf_counter() - t0
    kv = int(w.context_lengths[seqs].astype(np.int64).sum()) * w.kv_heads * w.head_dim * 4
    # the same oracle on one core, over the calibration sequence alone (then all cores again)
    t0 = time.perf_counter()
    oracle.decode(w, rows=np.arange(b0 * g, (b0 + 1) * g), threads=1)
    dt1 = max(time.perf_counter() - t0, 1e-6)
    oracle.decode(w, rows=np.arange(b0 * g, b0 * g + 1), threads=cores)
    kv1 = int(w.context_lengths[b0]) * w.kv_heads * w.head_dim * 4
    return {"value": kv / dt / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n_seq} of {w.batch} sequences (all {g} query heads each), "
                      f"{kv / 1e6:.1f} MB of K/V, {dt:.2f} s",
            "single_core": {"value": kv1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": f"sequence {b0} ({int(w.context_lengths[b0])} tokens, "
                                      f"all {g} query heads), {dt1:.2f} s"}}


def config_of(w, plan, extra=None):
    c = {"workload": w.name, "batch": w.batch, "query_heads": w.query_heads,
         "kv_heads": w.kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
         "max_pages_per_sequence": w.max_pages_per_sequence,
         "context_tokens": int(w.context_lengths.sum()),
         "l2": L2_FLUSH_NOTE,
         "schedule": ["auto", "single", "balanced"][plan["schedule"]],
         "math": ["auto", "simt", "mma"][plan["math"]],
         "workers": plan["workers"], "stages": plan["stages"],
         "warps_per_cta": plan["warps_per_cta"], "parallelism": "replicas"}
    if extra:
        c.update(extra)
    return c


def run_prefill_only(args):
    import torch

    from paged_kv_cache_63_gb300 import lib

    torch.cuda.set_device(0)
    lib.load()
    print(json.dumps({"prefill": prefill_lines(torch, lib, args.steps),
                      "steps": args.steps, "l2": L2_FLUSH_NOTE}), flush=True)


def time_calls(fns, steps, warmup, torch):
    """Mean CUDA-event time (ms) of each of `fns` (callables that launch on the current
    stream), called in order every step, L2 flushed before each step."""
    flush = L2Flush(torch)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        for f in fns:
            f()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
          for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        for k, f in enumerate(fns):
            f()
            ev[i][k + 1].record(stream)
    torch.cuda.synchronize()
    return [sum(e[k].elapsed_time(e[k + 1]) for e in ev) / steps for k in range(len(fns))]


def run_kernel_case(args):
    """One of the library's other kernels on a full-size workload, timed alone: the command
    its ncu capture runs. Prints one JSON line with microseconds per call and the kernel's
    roofline (bytes or FLOPs of the call / its CUDA-event time)."""
    import torch

    from paged_kv_cache_63_gb300 import lib
    from paged_kv_cache_63_gb300.workloads import make_prefill, make_workload

    torch.cuda.set_device(0)
    lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    hbm, hbm_kind = measured_peak()
    line = {"kernel_case": args.kernel_case, "steps": args.steps, "warmup": args.warmup,
            "l2": L2_FLUSH_NOTE}
    if args.kernel_case == "append":
        # one new K/V row per (sequence, K/V head) of ragged, written at the last cached
        # index (context - 1), whose page every table already holds
        w = make_workload("ragged")
        prob = lib.problem_of(w)
        rng = np.random.default_rng(11)
        shape = (w.batch, w.kv_heads, w.head_dim)
        nk = torch.from_numpy(rng.standard_normal(shape).astype(np.float16)).cuda()
        nv = torch.from_numpy(rng.standard_normal(shape).astype(np.float16)).cuda()
        k, v = torch.from_numpy(w.key_cache).cuda(), torch.from_numpy(w.value_cache).cuda()
        bt = torch.from_numpy(w.block_tables).cuda()
        ctx = torch.from_numpy(w.context_lengths - 1).cuda()
        (ms,) = time_calls([lambda: lib.pa_append_kv(prob, nk, nv, bt, ctx, k, v, stream)],
                           args.steps, args.warmup, torch)
        nbytes = 2 * 2 * nk.numel() * 2 + w.batch * 4 * 2  # rows read and written, ctx, bt
        line.update(workload="ragged", kernel="pa::append_kv_kernel", us_per_call=round(ms * 1e3, 2),
                    roofline={"bound": "hbm", "achieved": round(nbytes / (ms * 1e-3) / 1e9, 2),
                              "peak": hbm, "unit": "GB/s",
                              "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                              "peak_source": f"{hbm_kind} (HBM copy)",
                              "algorithmic_bytes_per_launch": nbytes})
    elif args.kernel_case == "split_combine":
        # the pages' fixed split: every sequence of long_gqa6 cut into `splits` ranges
        w = make_workload("long_gqa6")
        prob = lib.problem_of(w)
        d = to_device(w, torch)
        n = args.splits
        pm = torch.empty((w.batch, n, w.query_heads), dtype=torch.float32, device="cuda")
        ps = torch.empty_like(pm)
        po = torch.empty((w.batch, n, w.query_heads, w.head_dim), dtype=torch.float32,
                         device="cuda")
        ms_p, ms_c = time_calls(
            [lambda: lib.pa_split_kv_partial(prob, d["q"], d["k"], d["v"], d["bt"], d["ctx"],
                                             w.scale, n, pm, ps, po, stream=stream),
             lambda: lib.pa_split_kv_combine(prob, n, pm, ps, po, d["out"], stream)],
            args.steps, args.warmup, torch)
        part = (pm.numel() + ps.numel() + po.numel()) * 4
        comb = part + d["out"].numel() * 4
        kv = algorithmic_bytes(w)["total"] + part
        line.update(workload="long_gqa6", splits=n,
                    partial={"kernel": "pa::decode_kernel (fixed split)",
                             "us_per_call": round(ms_p * 1e3, 2),
                             "achieved": round(kv / (ms_p * 1e-3) / 1e9, 2), "unit": "GB/s",
                             "frac": round(kv / (ms_p * 1e-3) / 1e9 / hbm, 4)},
                    kernel="pa::combine_split_kernel", us_per_call=round(ms_c * 1e3, 2),
                    roofline={"bound": "hbm", "achieved": round(comb / (ms_c * 1e-3) / 1e9, 2),
                              "peak": hbm, "unit": "GB/s",
                              "frac": round(comb / (ms_c * 1e-3) / 1e9 / hbm, 4),
                              "peak_source": f"{hbm_kind} (HBM copy)",
                              "algorithmic_bytes_per_launch": comb})
    else:
        p = make_prefill("prefill_gqa6_hd256")
        ms = time_prefill(p, args.steps, args.warmup, torch, lib)
        peak, kind = measured_tensor_peak()
        flops = 4.0 * p.causal_pairs() * p.cache.query_heads * p.cache.head_dim
        tf = flops / (ms * 1e-3) / 1e12
        line.update(workload="prefill_gqa6_hd256", kernel="pa::prefill_kernel<256>",
                    us_per_call=round(ms * 1e3, 1),
                    roofline={"bound": "tensor", "achieved": round(tf, 1), "peak": peak,
                              "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                              "peak_source": f"{kind} (bf16 GEMM burst; fp16 same rate)",
                              "causal_flops": flops})
    assert lib.pa_get_device_error() == 0
    print(json.dumps(line), flush=True)


def measure(w, layout, opts, steps, warmup, e2e_steps, torch, lib, sm_count, sampler_dev):
    """One workload's complete block: device-timed steps (L2 flushed between them) with the
    clocks sampled during them, the roofline of that interval, and the pipelined end-to-end
    figure. Returns (block, ms per step, e2e ms per step, algorithmic bytes)."""
    plan = lib.pa_plan(lib.problem_of(w), opts, sm_count)
    d = to_device(w, torch)
    nbytes = algorithmic_bytes(w)
    ms, wall, clocks = time_decode(w, d, opts, steps, warmup, torch, lib, sampler_dev=sampler_dev)
    assert lib.pa_get_device_error() == 0
    e2e_ms, serial_ms = time_e2e(w, d, opts, e2e_steps, warmup, torch, lib)
    assert lib.pa_get_device_error() == 0
    del d
    torch.cuda.empty_cache()
    ms_step = sum(ms) / len(ms)
    peak, peak_kind = measured_peak()
    achieved = nbytes["total"] / (ms_step * 1e-3) / 1e9
    kv_gbs = nbytes["kv"] / (ms_step * 1e-3) / 1e9
    launches_per_call = 2 if (plan["schedule"] == 2 and plan["combine"] == 2) else 1
    # the recorded captures are of the token-major layout
    traffic = recorded_traffic(w.name) if layout == "token_major" else None
    block = {
        "workload": w.name,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_call": round(ms_step * 1e3, 2),
        "us_per_call_median": round(statistics.median(ms) * 1e3, 2),
        "value": round(kv_gbs, 2),
        "unit": "GB/s",
        "pct_of_hbm_peak": round(100 * kv_gbs / peak, 2),
        "config": config_of(w, plan, {"kv_bytes": nbytes["kv"], "cache_layout": layout}),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (HBM copy)", "traffic": traffic,
                     "algorithmic_bytes_per_launch": nbytes["total"],
                     "kernel": "pa::decode_kernel",
                     "launches_per_call": launches_per_call,
                     "interval": ("CUDA events on the launching stream around each pa_decode_ex "
                                  "call: the decode kernel"
                                  + (" and its dependent combine kernel" if launches_per_call == 2
                                     else ", the only launch"))},
        "clocks": clocks,
        "e2e": {"value": round(nbytes["kv"] / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_ms * 1e3, 2), "steps": e2e_steps,
                "serial_us_per_step": round(serial_ms * 1e3, 2),
                "h2d_bytes_per_step": nbytes["h2d"], "d2h_bytes_per_step": nbytes["d2h"],
                "note": "every step copies its q, block table and context lengths from pinned "
                        "host memory (one copy) and its output back, through pa_decode_ex; "
                        "copies on two copy streams with two device buffers overlap the "
                        "neighbouring steps' decodes; serial_us_per_step is one step alone; the "
                        "K/V cache is resident state (inputs larger than L2, no flush)"},
        "gpu_launches": steps * launches_per_call,
        "wall_s_timed_region": round(wall, 3),
    }
    return block, ms_step, e2e_ms, nbytes


def run_ours(args):
    import torch

    from paged_kv_cache_63_gb300 import lib
    from paged_kv_cache_63_gb300.workloads import make_workload

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    lib.load()
    opts = lib.options(schedule=args.schedule, math=args.math, combine=args.combine,
                       workers=args.workers, stages=args.stages, warps_per_cta=args.warps)
    sm_count = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    dev_index = torch.cuda.current_device()
    phys = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    smi_index = int(phys[dev_index]) if phys and phys[0].strip().isdigit() else dev_index

    def workload(name, seed=None):
        w = make_workload(name, seed=seed)
        if args.layout == "head_major":
            from paged_kv_cache_63_gb300.workloads import to_head_major

            w = to_head_major(w)
        return w

    seed = None if rank == 0 else 1000 + rank  # each rank decodes its own batch
    w = workload(args.workload, seed)
    e2e_steps = max(10, args.steps // 4)
    block, ms_step, e2e_step, nbytes = measure(
        w, args.layout, opts, args.steps, args.warmup, e2e_steps, torch, lib, sm_count,
        smi_index if rank == 0 else None)
    (ms_step, e2e_step), (kv_all, total_all) = reduce_over_ranks(
        torch, "cuda", [ms_step, e2e_step], [nbytes["kv"], nbytes["total"]])
    if rank != 0:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
        return
    line = {
        "metric": METRIC,
        "value": round(kv_all / (ms_step * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_call": block["us_per_call"],
        "pct_of_hbm_peak": block["pct_of_hbm_peak"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "accumulate": "f32",
        "data": "synthetic (seeded numpy draws of the workload's shapes and length mix)",
        "config": block["config"],
        "roofline": block["roofline"],
        "clocks": block["clocks"],
        "e2e": dict(block["e2e"], value=round(kv_all / (e2e_step * 1e-3) / 1e9, 2)),
        "gpu_launches": block["gpu_launches"],
        "wall_s_timed_region": block["wall_s_timed_region"],
    }
    if not args.no_others:
        others = {}
        for name in OTHER_WORKLOADS:
            if name == w.name:
                continue
            wo = workload(name)
            steps_o = max(args.steps, 200)
            others[name], _, _, _ = measure(wo, args.layout, opts, steps_o, max(args.warmup, 3),
                                            max(10, steps_o // 4), torch, lib, sm_count, smi_index)
            del wo
        line["other_workloads"] = others
        line["prefill"] = prefill_lines(torch, lib, 20)
    line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm: each step decodes a bounded sample of the
    workload (all heads of a few sequences) on the host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_63_gb300.workloads import make_workload

    oracle.build()
    w = make_workload(args.workload)
    g = w.query_heads
    budget = 120.0 / max(1, args.steps + args.warmup)  # seconds of CPU work per step
    b0 = int(np.argsort(w.context_lengths)[len(w.context_lengths) // 2])
    t0 = time.perf_counter()
    oracle.decode(w, rows=np.arange(b0 * g, (b0 + 1) * g))
    t_seq = max(time.perf_counter() - t0, 1e-4)
    if budget >= t_seq:
        rows = np.arange(b0 * g, (b0 + 1) * g)
        kv = int(w.context_lengths[b0]) * w.kv_heads * w.head_dim * 4
        desc = f"all {g} heads of sequence {b0}"
    else:
        heads = max(1, int(g * budget / t_seq))
        kvh = w.kv_heads
        heads = max(1, heads // (g // kvh)) * (g // kvh)  # whole GQA groups
        heads = min(heads, g)
        rows = np.arange(b0 * g, b0 * g + heads)
        kv = int(w.context_lengths[b0]) * (heads // (g // kvh)) * w.head_dim * 4
        desc = f"{heads} of {g} heads of sequence {b0}"
    for _ in range(args.warmup):
        oracle.decode(w, rows=rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.decode(w, rows=rows)
        times.append(time.perf_counter() - t0)
    step = sum(times) / len(times)
    value = kv / step / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "query_heads": w.query_heads,
                       "kv_heads": w.kv_heads, "head_dim": w.head_dim,
                       "page_size": w.page_size,
                       "max_pages_per_sequence": w.max_pages_per_sequence,
                       "context_tokens": int(w.context_lengths.sum()),
                       "parallelism": "replicas", "sample_per_step": desc},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"each step: {desc}"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill_only:
        run_prefill_only(args)
    elif args.kernel_case:
        run_kernel_case(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
