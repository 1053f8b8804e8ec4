"""Calibrates the sample-size rule's cost ratio r(k) on the current GPU.

The corrected paper chooses the sample size S by minimising a cost model of the
stages that depend on it (Appendix B, Proposition 7; Appendix E.1 "Sample
Size"):

    C(S) = c + (g + b) S + d(k) M(S),

where g + b is the per-element cost of drawing and ranking the sample, d(k) the
per-element cost of selecting the top k from the M buffer slots, and c a fixed
cost per configuration.  Its single hardware constant is the ratio
r(k) = (g + b) / d(k), which the paper fits once per GPU as
1/r(k) = a log2(k) + b0 for k above a cut-off (r = infinity below it).

This script repeats that calibration with this library: for every (n, k) of a
grid it forces S over powers of two (PROFK_OPT_FORCE_S; t and M then follow the
fast rule of Algorithm 1 at that S), times whole exact calls (sampling, filter,
check and refinement) with CUDA events on standard-normal inputs, fits the
model by least squares (one intercept per configuration, one sampling cost,
one buffer cost per k) and prints the fitted costs and the line for 1/r(k) as
one JSON object.  The sample-size rule PROFK_PARAMS_CORRECTED uses the constants
found this way on a GB300.

    python -m streaming_selection_primitive_gb300.calibrate --out calib.json
"""
from __future__ import annotations

import argparse
import json
import math
import sys

import numpy as np


def _sweep(pk, torch, ns, ks, Ss, calls, inputs, s_min_fit):
    dev = torch.device("cuda")
    rows = []
    for n in ns:
        for inp in range(inputs):
            g = torch.Generator(device=dev)
            g.manual_seed(1000 + inp)
            x = torch.randn(n, device=dev, generator=g)
            for k in ks:
                if 64 * k > n:
                    continue
                out = (torch.empty(k, dtype=torch.float32, device=dev), torch.empty(k, dtype=torch.int64, device=dev))
                for S in Ss:
                    if 32 * S > n:  # the paper's sweep caps S at n/32
                        continue
                    pk.set_option(pk.OPT_FORCE_S, S)
                    try:
                        for w in range(3):
                            pk.topk(x, k, 1e-3, 7 + w, out=out)
                        torch.cuda.synchronize()
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record()
                        Ms = []
                        for c in range(calls):
                            _, _, st = pk.topk(x, k, 1e-3, 100 + c, out=out)
                            Ms.append(st["M"])
                        e1.record()
                        torch.cuda.synchronize()
                        ms = e0.elapsed_time(e1) / calls
                        pk.set_option(pk.OPT_TIMING, 1)
                        stage = {}
                        for c in range(5):
                            pk.topk(x, k, 1e-3, 500 + c, out=out)
                            for name, v in pk.last_stage_ms().items():
                                stage.setdefault(name, []).append(v)
                        pk.set_option(pk.OPT_TIMING, 0)
                    finally:
                        pk.set_option(pk.OPT_FORCE_S, 0)
                        pk.set_option(pk.OPT_TIMING, 0)
                    rows.append({"n": n, "k": k, "S": S, "input": inp, "M": int(Ms[0]), "ms": ms,
                                 "stages_ms": {a: float(np.mean(b)) for a, b in stage.items()}})
            del x
            torch.cuda.empty_cache()
    return rows


def fit(rows, s_min_fit=1 << 14, k_cut=1 << 7):
    """Least-squares fit of C = c_(n,k) + gb S + d_k M over the rows with S >= s_min_fit;
    then 1/r(k) = d_k / gb and its line in log2 k over k > k_cut.  Times in ns."""
    pts = [r for r in rows if r["S"] >= s_min_fit]
    cfgs = sorted({(r["n"], r["k"]) for r in pts})
    ks = sorted({r["k"] for r in pts})
    nc, nk = len(cfgs), len(ks)
    A = np.zeros((len(pts), nc + 1 + nk))
    y = np.zeros(len(pts))
    for i, r in enumerate(pts):
        A[i, cfgs.index((r["n"], r["k"]))] = 1.0
        A[i, nc] = r["S"]
        A[i, nc + 1 + ks.index(r["k"])] = r["M"]
        y[i] = r["ms"] * 1e6  # ns
    coef, *_ = np.linalg.lstsq(A, y, rcond=None)
    pred = A @ coef
    rel = float(np.mean(np.abs(pred - y) / y))
    r2 = float(1.0 - np.sum((pred - y) ** 2) / np.sum((y - y.mean()) ** 2))
    gb = float(coef[nc])
    d = {k: float(coef[nc + 1 + j]) for j, k in enumerate(ks)}
    inv_r = {k: d[k] / gb for k in ks} if gb > 0 else {}
    big = [k for k in ks if k > k_cut and k in inv_r]
    line = None
    if len(big) >= 2:
        xs = np.array([math.log2(k) for k in big])
        ys = np.array([inv_r[k] for k in big])
        a, b0 = np.polyfit(xs, ys, 1)
        line = {"slope": float(a), "intercept": float(b0), "k_cut": k_cut}
    # Latency-optimal S per configuration, for comparison with any rule.
    best = {}
    for r in rows:
        key = f"{r['n']}:{r['k']}"
        cur = best.get(key)
        ms = np.mean([q["ms"] for q in rows if q["n"] == r["n"] and q["k"] == r["k"] and q["S"] == r["S"]])
        if cur is None or ms < cur[1]:
            best[key] = (r["S"], float(ms))
    return {"sampling_ns_per_elem": gb, "buffer_ns_per_elem": {str(k): v for k, v in d.items()},
            "inv_r": {str(k): v for k, v in inv_r.items()}, "inv_r_line": line, "mean_rel_err": rel, "r2": r2,
            "points": len(pts), "best_S": {k: {"S": v[0], "ms": round(v[1], 4)} for k, v in best.items()}}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--n", type=int, nargs="+", default=[1 << 22, 1 << 24, 1 << 26, 1 << 28, 1 << 30])
    ap.add_argument("--k", type=int, nargs="+", default=[1 << 5, 1 << 8, 1 << 11, 1 << 14, 1 << 17, 1 << 19])
    ap.add_argument("--S", type=int, nargs="+", default=[1 << e for e in range(12, 19)])
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--inputs", type=int, default=2)
    ap.add_argument("--out", default=None)
    args = ap.parse_args(argv)

    import torch

    import streaming_selection_primitive_gb300 as pk

    if not torch.cuda.is_available():
        print("calibrate: no CUDA device", file=sys.stderr)
        return 2
    rows = _sweep(pk, torch, args.n, args.k, args.S, args.calls, args.inputs, 1 << 14)
    res = {"device": torch.cuda.get_device_name(), "fit": fit(rows), "rows": rows}
    text = json.dumps(res)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text)
    print(json.dumps(res["fit"]))
    return 0


if __name__ == "__main__":
    sys.exit(main())
