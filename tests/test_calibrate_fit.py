"""The sample-size calibration's least-squares fit (no GPU).

The fit of C = c_(n,k) + (g + b) S + d(k) M (the corrected paper's Appendix
E.1 model) must recover planted costs from synthetic latencies, and the line
1/r(k) = a log2 k + b0 over k > 2^7 must follow them."""
import math

import numpy as np

from oracle import params as P
from streaming_selection_primitive_gb300.calibrate import fit


def synthetic_rows(gb, inv_r, noise, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for n in (1 << 24, 1 << 26, 1 << 28):
        for k in (1 << 5, 1 << 8, 1 << 11, 1 << 14, 1 << 17):
            if 64 * k > n:
                continue
            c = 20_000.0 + 1000.0 * math.log2(n)  # per-configuration intercept, ns
            for S in (1 << e for e in range(12, 19)):
                if 32 * S > n:
                    continue
                _, M = P.params_fast(n, k, S, 1e-3)
                d = gb * inv_r(k)
                ns = (c + gb * S + d * M) * (1 + noise * rng.standard_normal())
                rows.append({"n": n, "k": k, "S": S, "input": 0, "M": M, "ms": ns / 1e6, "stages_ms": {}})
    return rows


def test_fit_recovers_planted_costs():
    inv_r = lambda k: 0.59 * math.log2(k) - 4.3 if k > 2 ** 11 else 0.0  # the paper's form, zero below
    rows = synthetic_rows(0.36, inv_r, noise=0.0)
    f = fit(rows)
    assert abs(f["sampling_ns_per_elem"] - 0.36) < 1e-6
    for k in (1 << 14, 1 << 17):
        assert abs(f["inv_r"][str(k)] - inv_r(k)) < 1e-6
    assert f["r2"] > 0.999999 and f["mean_rel_err"] < 1e-9


def test_fit_with_noise_and_best_sample():
    inv_r = lambda k: 0.5
    rows = synthetic_rows(0.1, inv_r, noise=0.01, seed=3)
    f = fit(rows)
    assert abs(f["sampling_ns_per_elem"] - 0.1) / 0.1 < 0.2
    line = f["inv_r_line"]
    assert line is not None and abs(line["slope"]) < 0.2 and abs(line["intercept"] - 0.5) < 1.0
    # the latency-optimal S reported for every configuration is one of the swept ones
    for key, b in f["best_S"].items():
        assert b["S"] in [1 << e for e in range(12, 19)]
