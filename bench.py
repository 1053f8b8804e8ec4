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
    """DRAM bytes per filter launch from the committed ncu summary, scaled to n;
    None when absent or when the filter source changed since the capture."""
    p = ROOT / "profiles" / "filter_normal_2p28.md"
    if not p.exists():
        return None
    text = p.read_text()
    m_hash = re.search(r"filter_source_hash:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_element:\s*([0-9.]+)", text)
    if not m_hash or not m_b or m_hash.group(1) != filter_source_hash():
        return None
    return float(m_b.group(1)) * n


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


def cpu_baseline(x_host_prefix, k, budget_s=12.0):
    """The oracle (full sort) on a bounded prefix of the same input."""
    from oracle.topk import topk_sort

    elems, t0, reps = 0, time.perf_counter(), 0
    while True:
        topk_sort(x_host_prefix, k)
        reps += 1
        elems += x_host_prefix.size
        if time.perf_counter() - t0 >= budget_s or reps >= 50:
            break
    dt = time.perf_counter() - t0
    return {"value": elems / dt / 1e9, "unit": "Gelem/s", "cores": 1, "kind": "oracle",
            "sample": f"oracle.topk_sort (numpy lexsort, one thread) on the first {x_host_prefix.size} elements "
                      f"of the same normal input, k={k}, {reps} calls in {dt:.1f} s"}


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


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch

    import workloads
    from oracle.topk import topk_sort

    n_sample = 1 << 22
    x = workloads.normal(n_sample, 1, "cpu").numpy()
    for _ in range(args.warmup):
        topk_sort(x, args.k)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        topk_sort(x, args.k)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n_sample * args.steps / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Gelem/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name("normal", args.n, args.k), "n": args.n, "k": args.k, "eps": EPS,
                   "sample_elems": n_sample},
        "cpu_baseline": {"value": value, "unit": "Gelem/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: oracle.topk_sort (full sort, one thread) on a {n_sample}-element "
                                   f"prefix-sized sample of the normal workload, k={args.k}"},
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

    cpu = None
    if rank == 0 and ws >= 1 and not args.no_cpu and args.gpus == 1:
        cpu = cpu_baseline(x[: 1 << 24].cpu().numpy(), k)

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
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
