"""Benchmark of Prof-K exact top-k on GB300.

One step = one exact top-k call (sample, threshold, filter, check, refine) on
a 2^30-element float32 standard-normal vector with k = 1024, eps = 1e-3, the
input already resident in HBM.  The input (4 GiB) is far larger than L2
(129 MB), so no flush is needed between steps.

Prints ONE JSON line (rank 0).  Keys beyond the base contract:
  roofline      filter kernel: algorithmic bytes 4n per launch / its mean
                device time (CUDA events the library records on the launch
                stream), against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle (full sort) on a bounded prefix of the input
  e2e           the same metric through the C-ABI with host buffers: each step
                copies x host->device from pinned memory, runs the call and
                copies the k results back (two device buffers: the next
                step's copy runs while this step selects)
  sweep         the other k and distributions at 2^30 (fewer steps each)
  synchronous   the same calls through profk_topk (one host round trip per call)

The timed steps go through the asynchronous form (profk_topk_async, all K calls
in flight, each completed by profk_wait): one step is still one whole exact
top-k call, check included.

--impl reference times the CPU oracle itself (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

N_DEFAULT = 1 << 30
K_DEFAULT = 1024
EPS = 1e-3
METRIC = "top-k Gelem/s and HBM GB/s vs peak, N=2^30 fp32, k∈{32,1024,2^19}"


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def filter_source_hash() -> str:
    """Hash of the source the filter kernel is compiled from: filter.cu,
    common.cuh, and the parts of kernels.h it uses (the PDL helpers, the launch
    helper and FilterArgs)."""
    csrc = ROOT / "streaming_selection_primitive_gb300" / "csrc"
    h = hashlib.sha256()
    for name in ("filter.cu", "common.cuh"):
        h.update((csrc / name).read_bytes())
    k = (csrc / "kernels.h").read_text()
    start = k.index("__device__ __forceinline__ void pdl_wait()")
    end = k.index("\n}\n", k.index("inline cudaError_t launch_kernel")) + 3
    h.update(k[start:end].encode())
    m = re.search(r"struct FilterArgs \{.*?\};", k, flags=re.S)
    h.update(m.group(0).encode())
    return h.hexdigest()[:16]


def traffic_from_profile(n: int):
    """DRAM bytes per filter launch from the committed ncu figures
    (profiles/filter_normal_2p28.json), scaled to n; None when absent or when
    the filter source changed since the capture."""
    p = ROOT / "profiles" / "filter_normal_2p28.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text())
    if d.get("filter_source_hash") != filter_source_hash():
        return None
    return float(d["dram_bytes_per_element"]) * n


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms while
    active; the summary keeps the samples taken inside the timed region
    (mark() at its start and end), or, for a region shorter than the sampling
    interval, the two samples nearest to it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.path = None
        self.marks = []

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark(self):
        self.marks.append(time.time())

    def __exit__(self, *exc):
        time.sleep(0.05)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        from datetime import datetime

        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), [nm for nm, v in zip(names, f[6:10])
                                                              if v.lower() == "active"]))
            except ValueError:
                continue
        os.unlink(self.path)
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (float("-inf"), float("inf"))
        inside = [r for r in rows if t0 <= r[0] <= t1]
        where = "inside the timed region"
        if not inside and rows:
            mid = 0.5 * (t0 + t1) if len(self.marks) >= 2 else rows[len(rows) // 2][0]
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
            where = "nearest to the timed region (shorter than the 20 ms sampling interval)"
        reasons = sorted({nm for r in inside for nm in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": reasons, "samples": len(inside), "samples_from": where}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(x_host, k, reps=3):
    """The oracle on the whole input, on the host cores: its threaded form
    (topk_chunked, one thread per core, four chunks per thread) gives the
    value; its single-thread O(n) form (topk_partition) is timed once beside it."""
    from oracle.topk import topk_chunked, topk_partition

    cores = host_cores()
    n = x_host.size
    multi = []
    for _ in range(reps):
        t0 = time.perf_counter()
        topk_chunked(x_host, k, cores, 4 * cores)
        multi.append(time.perf_counter() - t0)
    t0 = time.perf_counter()
    topk_partition(x_host, k)
    single = time.perf_counter() - t0
    t = statistics.median(multi)
    return {"value": round(n / t / 1e9, 4), "unit": "Gelem/s", "cores": cores, "kind": "oracle",
            "ms_per_call": round(1e3 * t, 1),
            "sample": f"the whole {n}-element input of the timed steps, copied to the host; "
                      f"oracle.topk.topk_chunked (numpy selection per chunk on {cores} threads, then the "
                      f"exact merge), median of {reps} calls, k={k}",
            "single_thread": {"value": round(n / single / 1e9, 4), "unit": "Gelem/s", "cores": 1,
                              "ms_per_call": round(1e3 * single, 1),
                              "sample": "oracle.topk.topk_partition (numpy, one thread), one call on the same input"}}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


INPUTS = {
    "normal": "float32 N(0,1)",
    "uniform": "float32 Uniform[0,1) (2^24 levels)",
    "pareto": "float32 Pareto alpha = 1.5, x_m = 1",
    "ulps_below_one": "float32: 99.9 % in the 256 values just below 1.0, else Uniform[0,1)",
    "levels16": "float32: 16 equally likely levels i / 16",
    "sorted_normal": "float32 N(0,1) sorted ascending",
    "sae": "float32 ReLU(X W + b) flattened: X 4096 x 512 N(0,1), W 512 x 12288 N(0, 1/512), b N(0, 0.01)",
}


def l2_note(n: int) -> str:
    mb = 4 * n / 1e6
    if mb > 129:
        return f"input {mb:.0f} MB > L2 129 MB: no flush between steps"
    return f"input {mb:.0f} MB fits L2 (129 MB) and is not flushed: a hot-cache figure"


def workload_name(gen: str, n: int, k: int) -> str:
    size = f"2^{n.bit_length() - 1}" if n & (n - 1) == 0 else str(n)
    return f"{gen}_{size}_k{k}"


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest of every rank's x (a job takes its slowest rank's time);
    a collective of the ranks' process group (nccl on the GPUs, gloo on CPU)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gelems(n: int, steps: int, ws: int, ms: float) -> float:
    """Whole-job throughput: every rank's steps x n elements (each rank selects
    from its own row: weak scaling) over the slowest rank's time."""
    return n * steps * ws / (ms / 1e3) / 1e9


L2_FLUSH_BYTES = 256 << 20  # written between timed calls whose input fits the 129 MB L2


def time_sync_calls(call, reps, stream, flush=None):
    """Per-call latency of synchronous calls: CUDA events on the launch stream
    around each call.  With `flush` (a device buffer larger than L2) the
    buffer is overwritten before each call, outside the events, so that the
    call starts from a cold L2.  Returns (mean ms, every call's stats)."""
    import torch

    times, sts = [], []
    for s in range(reps):
        if flush is not None:
            flush.fill_(s & 0x7F)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st = call(s)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
        sts += st if isinstance(st, list) else [st]
    return statistics.mean(times), sts


def time_async_calls(submit, reps, stream):
    """Calls in flight together (the asynchronous form, the timed steps'
    form), each completed by profk_wait: (ms per call, every call's stats)."""
    import torch

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pend = [submit(s) for s in range(reps)]
    sts = []
    for p in pend:
        st = p.wait()[2]
        sts += st if isinstance(st, list) else [st]
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps, sts


def config_entry(n_elems, ms, sts, peak, **extra):
    """One configuration's figures: ms per call, Gelem/s, the input bytes per
    second as a fraction of 8 TB/s and of the measured copy peak, retries
    (attempts beyond the first, over every call and row), workspace, paths."""
    gbs = 4 * n_elems / (ms / 1e3) / 1e9
    return {"ms": round(ms, 4), "gelem_s": round(n_elems / ms / 1e6, 2), "hbm_gbs": round(gbs, 1),
            "hbm_frac_of_8TBs": round(gbs / 8000, 3), "hbm_frac_of_measured": round(gbs / peak, 3),
            "retries": int(sum(max(st["attempts"] - 1, 0) for st in sts)),
            "aux_bytes": int(max(st["aux_bytes"] for st in sts)),
            "paths": sorted({int(st["path"]) for st in sts}), **extra}


def binom_upper(n, p, q=0.99):
    """Smallest F with P(Binomial(n, p) <= F) >= q (log-space pmf recurrence)."""
    import math

    logp = n * math.log1p(-p)
    cdf, f = 0.0, 0
    while True:
        cdf += math.exp(logp)
        if cdf >= q or f >= n:
            return f
        logp += math.log((n - f) / (f + 1)) + math.log(p) - math.log1p(-p)
        f += 1


def baseline_configs(pk, dev, stream, rank, peak):
    """Every configuration of the project's specification beyond the headline
    2^30 row (those are in `sweep`), each with its own figures."""
    import torch

    import workloads

    out = {}

    def buf(k, rows=1):
        shape = (k,) if rows == 1 else (rows, k)
        return (torch.empty(shape, dtype=torch.float32, device=dev), torch.empty(shape, dtype=torch.int64, device=dev))

    # 1. 2^22 uniform, k = 32: the 16 MB input fits L2, so the per-call figure
    # flushes L2 before every call; the calls in flight are a hot-cache figure.
    x = workloads.uniform(1 << 22, 1 + rank, dev)
    o = buf(32)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for w in range(3):
        pk.topk(x, 32, EPS, 69_000 + w, out=o)
    ms, sts = time_sync_calls(lambda s: pk.topk(x, 32, EPS, 70_000 + s, out=o)[2], 30, stream, flush)
    out["uniform_2^22_k32_l2_flushed"] = config_entry(x.numel(), ms, sts, peak,
                                                      form="profk_topk, L2 flushed before each call")
    ms, sts = time_async_calls(lambda s: pk.topk_async(x, 32, EPS, 71_000 + s, out=o), 30, stream)
    out["uniform_2^22_k32_hot"] = config_entry(x.numel(), ms, sts, peak, form="30 async calls in flight, hot L2")
    del x, flush

    # 2. 2^26 normal, k in {32, 1024, 32768}; the retry rate over 10^4 seeds at 2^20, k = 64.
    x = workloads.normal(1 << 26, 1 + rank, dev)
    for kk in (32, 1024, 32768):
        o = buf(kk)
        for w in range(2):
            pk.topk(x, kk, EPS, 72_000 + w, out=o)
        ms, sts = time_async_calls(lambda s: pk.topk_async(x, kk, EPS, 73_000 + s, out=o), 20, stream)
        out[f"normal_2^26_k{kk}"] = config_entry(x.numel(), ms, sts, peak, form="20 async calls in flight")
    del x
    x = workloads.normal(1 << 20, 1 + rank, dev)
    o = buf(64)
    seeds, fails, t0 = 10_000, 0, time.perf_counter()
    for b0 in range(0, seeds, 250):
        pend = [pk.topk_async(x, 64, EPS, 100_000 + b0 + s, out=o) for s in range(250)]
        fails += sum(p.wait()[2]["attempts"] > 1 for p in pend)
    out["retry_rate_normal_2^20_k64"] = {
        "calls": seeds, "first_attempt_failures": int(fails), "rate": fails / seeds, "eps": EPS,
        "binomial_99_upper_at_eps": binom_upper(seeds, EPS), "seconds": round(time.perf_counter() - t0, 2),
        "seeds": "algorithm seeds 100000 .. 109999 on one input"}
    del x

    # 4. The 2^28 tie-stress variants, k = 4096.
    for gen in ("ulps_below_one", "levels16", "sorted_normal"):
        x = workloads.GENERATORS[gen](1 << 28, 4 + rank, dev)
        o = buf(4096)
        for w in range(2):
            pk.topk(x, 4096, EPS, 74_000 + w, out=o)
        ms, sts = time_async_calls(lambda s: pk.topk_async(x, 4096, EPS, 75_000 + s, out=o), 10, stream)
        out[f"{gen}_2^28_k4096"] = config_entry(x.numel(), ms, sts, peak, form="10 async calls in flight")
        del x
        torch.cuda.empty_cache()

    # 5. The SAE-shaped selection and 64 batched rows of 2^24.
    x = workloads.sae_preacts(5 + rank, dev)
    o = buf(131_072)
    for w in range(2):
        pk.topk(x, 131_072, EPS, 76_000 + w, out=o)
    ms, sts = time_async_calls(lambda s: pk.topk_async(x, 131_072, EPS, 77_000 + s, out=o), 10, stream)
    out["sae_50331648_k131072"] = config_entry(x.numel(), ms, sts, peak, form="10 async calls in flight")
    del x
    x = workloads.normal_rows(64, 1 << 24, 6 + rank, dev)
    o = buf(32, rows=64)
    for w in range(2):
        pk.topk_batched(x, 32, EPS, 78_000 + w, out=o)
    ms, sts = time_async_calls(lambda s: pk.topk_batched_async(x, 32, EPS, 79_000 + s, out=o), 10, stream)
    out["batched_64x2^24_k32"] = config_entry(x.numel(), ms, sts, peak, form="10 async calls in flight")
    del x
    torch.cuda.empty_cache()
    return out


REF_SAMPLE_ELEMS = 1 << 26


def run_reference(args):
    """The reference arm: the CPU oracle itself, as it stands, on the host
    cores.  Each step selects the top k of a 2^26-element sample of the same
    workload (standard normal, from the CPU generator) with the oracle's
    threaded form on every core; the config says so."""
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    import workloads
    from oracle.topk import topk_chunked

    n_sample = min(REF_SAMPLE_ELEMS, args.n)
    cores = host_cores()
    x = workloads.normal(n_sample, 1, "cpu").numpy()
    for _ in range(args.warmup):
        topk_chunked(x, args.k, cores, 4 * cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        topk_chunked(x, args.k, cores, 4 * cores)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n_sample * args.steps / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Gelem/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name("normal", args.n, args.k), "n": n_sample, "k": args.k, "eps": EPS,
                   "sample_of": f"each step selects from {n_sample} elements of the {args.n}-element workload's "
                                f"distribution (the oracle would take about {args.n // n_sample} times as long "
                                f"per call on the whole input)"},
        "cpu_baseline": {"value": value, "unit": "Gelem/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: oracle.topk.topk_chunked (numpy selection per chunk on {cores} "
                                   f"threads, then the exact merge) on a {n_sample}-element standard-normal "
                                   f"sample, k={args.k}"},
        "e2e": {"value": value, "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="profk", choices=["profk", "reference"])
    ap.add_argument("--n", type=int, default=N_DEFAULT)
    ap.add_argument("--k", type=int, default=K_DEFAULT)
    ap.add_argument("--gen", default="normal",
                    help="input generator of the timed steps (workloads.GENERATORS; default normal)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-protocol", action="store_true",
                    help="skip the per-call latency over several input tensors")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch

    import streaming_selection_primitive_gb300 as pk
    import workloads

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    pk.lib()
    pk.reset_options()
    n, k = args.n, args.k
    if args.gen == "sae":  # fixed shape: 4096 x 12288 activations, flattened
        x = workloads.sae_preacts(1 + rank, dev)
        n = x.numel()
    elif args.gen in workloads.GENERATORS:
        x = workloads.GENERATORS[args.gen](n, 1 + rank, dev)
    else:
        raise SystemExit(f"--gen: sae or one of {sorted(workloads.GENERATORS)}")
    stream = torch.cuda.current_stream()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    out = (torch.empty(k, dtype=torch.float32, device=dev), torch.empty(k, dtype=torch.int64, device=dev))
    for w in range(args.warmup):
        pk.topk(x, k, EPS, 10_000 + w, out=out)
        pk.topk_async(x, k, EPS, 20_000 + w, out=out).wait()
    barrier()
    filter_ms, attempts, launches, paths, Rs = [], [], 0, [], []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(dev.index)
    # The job: K calls on the resident input through the asynchronous form
    # (profk_topk_async), all in flight, each completed with profk_wait.
    with ClockSampler(gpu_id) as clk:
        barrier()
        clk.mark()
        ev0.record(stream)
        pending = [pk.topk_async(x, k, EPS, 1000 + s, out=out) for s in range(args.steps)]
        for p in pending:
            _, _, st = p.wait()
            attempts.append(st["attempts"])
            launches += st["launches"]
            paths.append(st["path"])
            Rs.append(st["R_first"])
        ev1.record(stream)
        barrier()
        clk.mark()
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    clocks = clk.summary()
    ms_step = total_ms / args.steps
    value = job_gelems(n, args.steps, ws, total_ms)
    peak, peak_kind = measured_peaks()
    traffic = traffic_from_profile(n) if args.gen == "normal" else None  # the capture is of the normal input
    aux = pk.topk(x, k, EPS, 7, out=out)[2]["aux_bytes"]
    # The same calls through the synchronous form (profk_topk: each call
    # returns after its check, so the host round trip sits between calls).
    barrier()
    ev0.record(stream)
    for s in range(args.steps):
        pk.topk(x, k, EPS, 30_000 + s, out=out)
    ev1.record(stream)
    barrier()
    sync_ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    synchronous = {"api": "profk_topk", "value": round(job_gelems(n, args.steps, ws, sync_ms), 3),
                   "unit": "Gelem/s", "ms_per_step": round(sync_ms / args.steps, 4),
                   "hbm_frac_of_8TBs": round(4 * n / (sync_ms / args.steps / 1e3) / 8e12, 4)}
    # Stage breakdown and the filter's own launch time, from CUDA events the
    # library records around each stage on the call's stream (PROFK_OPT_TIMING),
    # in separate calls after the timed loop so the events cost it nothing.
    pk.set_option(pk.OPT_TIMING, 1)
    stage_acc = {}
    for s in range(max(10, args.steps)):
        _, _, st = pk.topk(x, k, EPS, 60_000 + s, out=out)
        filter_ms.append(st["filter_ms"])
        for name, ms in pk.last_stage_ms().items():
            stage_acc.setdefault(name, []).append(ms)
    pk.set_option(pk.OPT_TIMING, 0)
    stages = {name: round(statistics.mean(v), 4) for name, v in stage_acc.items()}
    f_ms = statistics.mean(filter_ms)
    achieved = 4.0 * n / (f_ms / 1e3) / 1e9

    # End to end through the C-ABI with host buffers: every step copies its
    # input host -> device (pinned) and its result device -> host.  Two device
    # buffers and a copy stream let the copy of step s + 1 run while step s
    # selects; the copies still cross the link every step, so the job is bound
    # by the host link rather than by the call.
    xh = torch.empty(n, dtype=torch.float32, pin_memory=True)
    xh.copy_(x)
    xds = [torch.empty_like(x), torch.empty_like(x)]
    vh = torch.empty(k, dtype=torch.float32, pin_memory=True)
    ih = torch.empty(k, dtype=torch.int64, pin_memory=True)
    cstream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_run(steps, seed0):
        with torch.cuda.stream(cstream):
            cstream.wait_stream(stream)
            xds[0].copy_(xh, non_blocking=True)
            copied[0].record(cstream)
        for s in range(steps):
            b = s % 2
            if s + 1 < steps:  # the other buffer's previous call has returned (synchronous API)
                with torch.cuda.stream(cstream):
                    cstream.wait_stream(stream)
                    xds[1 - b].copy_(xh, non_blocking=True)
                    copied[1 - b].record(cstream)
            stream.wait_event(copied[b])
            pk.topk(xds[b], k, EPS, seed0 + s, out=out)
            vh.copy_(out[0], non_blocking=True)
            ih.copy_(out[1], non_blocking=True)

    e2e_run(2, 20_000)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.e2e_steps, 30_000)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    e2e_value = job_gelems(n, args.e2e_steps, ws, e2e_ms)
    del xh, xds

    # Per-call latency as the pages measure it: several input tensors (data
    # seeds), each with 20 synchronous calls of their own algorithm seeds,
    # every call bracketed by CUDA events on the launch stream.
    protocol = None
    if not args.no_protocol:
        per_call = []
        inputs = 5
        for d in range(inputs):
            if d == 0:
                xs = x
            elif args.gen == "sae":
                xs = workloads.sae_preacts(101 + d + 10 * rank, dev)
            else:
                xs = workloads.GENERATORS[args.gen](n, 101 + d + 10 * rank, dev)
            pk.topk(xs, k, EPS, 60_000 + d, out=out)  # warm for this tensor
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
            for s, (a0, a1) in enumerate(evs):
                a0.record(stream)
                pk.topk(xs, k, EPS, 61_000 + 100 * d + s, out=out)
                a1.record(stream)
            torch.cuda.synchronize()
            per_call += [a0.elapsed_time(a1) for a0, a1 in evs]
            if d > 0:
                del xs
        per_call.sort()
        q = lambda f: per_call[min(len(per_call) - 1, int(f * len(per_call)))]
        protocol = {"api": "profk_topk", "inputs": inputs, "calls_each": 20, "mean_ms": round(statistics.mean(per_call), 4),
                    "p50_ms": round(q(0.50), 4), "p99_ms": round(q(0.99), 4), "max_ms": round(per_call[-1], 4)}

    sweep = {}
    if not args.no_sweep:
        for gen in ("uniform", "normal", "pareto"):
            xs = x if gen == "normal" else workloads.GENERATORS[gen](n, 1 + rank, dev)
            for kk in (32, 1024, 1 << 19):
                o2 = (torch.empty(kk, dtype=torch.float32, device=dev), torch.empty(kk, dtype=torch.int64, device=dev))
                for w in range(2):
                    pk.topk(xs, kk, EPS, 40_000 + w, out=o2)
                torch.cuda.synchronize()
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 5
                a0.record(stream)
                for p in [pk.topk_async(xs, kk, EPS, 50_000 + s, out=o2) for s in range(reps)]:
                    p.wait()
                a1.record(stream)
                torch.cuda.synchronize()
                ms = a0.elapsed_time(a1) / reps
                sweep[f"{gen}_k{kk}"] = {"ms": round(ms, 4), "gelem_s": round(n / ms / 1e6, 2),
                                         "hbm_frac_of_8TBs": round(4 * n / (ms / 1e3) / 8e12, 3)}
            if gen != "normal":
                del xs
                torch.cuda.empty_cache()
        # The corrected paper's own sample-size rule (Proposition 7 with the
        # GB300 cost ratio) on the same normal input, beside the default rule.
        pk.set_option(pk.OPT_PARAM_MODE, pk.PARAMS_CORRECTED)
        try:
            for kk in (32, 1024, 1 << 19):
                o2 = (torch.empty(kk, dtype=torch.float32, device=dev), torch.empty(kk, dtype=torch.int64, device=dev))
                for w in range(2):
                    pk.topk(x, kk, EPS, 40_000 + w, out=o2)
                torch.cuda.synchronize()
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 5
                a0.record(stream)
                for p in [pk.topk_async(x, kk, EPS, 50_000 + s, out=o2) for s in range(reps)]:
                    p.wait()
                a1.record(stream)
                torch.cuda.synchronize()
                ms = a0.elapsed_time(a1) / reps
                sweep[f"normal_k{kk}_corrected_rule"] = {
                    "S": pk.params(n, kk, EPS, pk.PARAMS_CORRECTED)[0], "ms": round(ms, 4),
                    "gelem_s": round(n / ms / 1e6, 2), "hbm_frac_of_8TBs": round(4 * n / (ms / 1e3) / 8e12, 3)}
        finally:
            pk.set_option(pk.OPT_PARAM_MODE, pk.PARAMS_DEFAULT)
        # The corrected paper's Table 4 sizes (single rows beyond 2^31, standard
        # normal): latency and auxiliary memory of synchronous calls.  Rows above
        # 2^32 elements are split into segments and merged.
        table4 = {}
        for big_n, kks in ((1 << 31, (1 << 10, 1 << 14, 1 << 18, 1 << 22)), (3_000_000_000, (1 << 10, 1 << 18)),
                           (4_300_000_000, (1 << 10, 1 << 18, 1 << 22))):
            xb = workloads.normal(big_n, 31 + rank, dev)
            for kk in kks:
                o2 = (torch.empty(kk, dtype=torch.float32, device=dev), torch.empty(kk, dtype=torch.int64, device=dev))
                for w in range(2):
                    pk.topk(xb, kk, EPS, 40_000 + w, out=o2)
                torch.cuda.synchronize()
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 5
                a0.record(stream)
                for s in range(reps):
                    _, _, st = pk.topk(xb, kk, EPS, 50_000 + s, out=o2)
                a1.record(stream)
                torch.cuda.synchronize()
                ms = a0.elapsed_time(a1) / reps
                table4[f"n{big_n}_k{kk}"] = {"ms": round(ms, 4), "gelem_s": round(big_n / ms / 1e6, 2),
                                             "hbm_frac_of_8TBs": round(4 * big_n / (ms / 1e3) / 8e12, 3),
                                             "aux_mb": round(st["aux_bytes"] / 1e6, 2), "path": st["path"]}
            del xb
            torch.cuda.empty_cache()
        sweep["table4"] = table4

    configs = None
    if not args.no_sweep and args.gen == "normal" and n == N_DEFAULT:
        configs = baseline_configs(pk, dev, stream, rank, peak)

    cpu = None
    if rank == 0 and ws >= 1 and not args.no_cpu and args.gpus == 1:
        cpu = cpu_baseline(x.cpu().numpy(), k)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "Gelem/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_name(args.gen, n, k), "n": n, "k": k, "eps": EPS,
                       "input": INPUTS.get(args.gen, args.gen),
                       "l2": l2_note(n), "parallelism": f"replicas x{ws}",
                       "api": f"profk_topk_async, {args.steps} calls in flight, each completed by profk_wait"},
            "hbm_gbs_end_to_end": round(4 * n / (ms_step / 1e3) / 1e9, 1),
            "hbm_frac_of_8TBs": round(4 * n / (ms_step / 1e3) / 8e12, 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_kind,
                         "kernel": "k_filter", "bytes_per_launch": 4 * n, "mean_launch_ms": round(f_ms, 4)},
            "e2e": {"value": round(e2e_value, 3), "unit": "Gelem/s", "h2d_bytes_per_step": 4 * n,
                    "d2h_bytes_per_step": 12 * k, "ms_per_step": round(e2e_ms / args.e2e_steps, 3)},
            "stages_ms": stages,
            "synchronous": synchronous,
            "gpu_launches": launches,
            "retries": int(sum(a - 1 for a in attempts if a > 0)),
            "aux_bytes": aux,
            "R_first_mean": round(float(np.mean(Rs)), 1),
            "clocks": clocks,
            "cpu_baseline": cpu,
            "protocol": protocol,
            "sweep": sweep,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
