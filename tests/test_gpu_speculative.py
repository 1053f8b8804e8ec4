"""Redraws enqueued on the device (PROFK_OPT_SPECULATIVE), against the oracle.

The run-time check (corrected paper, Section 3 stage 4; Appendix D "Cost of
the Run-Time Check") redraws a row whose count R misses k <= R <= M.  With the
option at D, a call enqueues attempts 1 .. D right after attempt 0, before the
host reads any count; each attempt's refinement records whether its row is
settled (passed, tie exit, NaN or error), and the kernels of the later
attempts leave a settled row alone.  Every call here must give the oracle
procedure's result and statistics (it redraws one attempt at a time, as the
pages describe), the same as the call with the option off, and a row that
passes within the D + 1 attempts must complete with no kernel launched after
the report: every such call launches the same number of kernels.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from oracle import profk as PK
from routing import oracle_profk

pytestmark = pytest.mark.gpu

STAT_KEYS = ("S", "t", "M", "R_first", "R_gt_first", "tau_first", "R_final", "R_gt_final", "tau_final",
             "attempts", "path")


def check_oracle(st, v, i, h, k, eps, seed, what, **kw):
    ov, oi, ost = oracle_profk(h, k, eps, seed, **kw)
    assert_same(v, i, ov, oi, what)
    assert (st["attempts"], st["path"], st["R_first"], st["R_gt_first"], st["R_final"], st["R_gt_final"]) == \
        (ost.attempts, ost.path, ost.R_first, ost.R_gt_first, ost.R_final, ost.R_gt_final), (what, st, ost)
    assert st["tau_first"] == ost.taus[0] and st["tau_final"] == ost.taus[-1], (what, st, ost.taus)
    return ost


# eps = 0.5 makes the first check fail often: the candidate-list sampler
# (t = 4), the sampler's grid passes with the reset kernel (t = 12), and the
# buffer sort as the refinement (k > 8192).
@pytest.mark.parametrize("n,k", [((1 << 22) + 4, 300), ((1 << 20) + 4, 300), ((1 << 22) + 4, 9000)])
def test_device_redraws_match_oracle(pk, cuda_device, n, k):
    x = workloads.normal(n, 23, cuda_device)
    h = x.cpu().numpy()
    seeds = range(16)
    off = [pk.topk(x, k, 0.5, s) for s in seeds]
    pk.set_option(pk.OPT_SPECULATIVE, 5)
    launches = set()
    redrawn = 0
    for s, ref in zip(seeds, off):
        for form in ("async", "sync"):
            if form == "async":
                v, i, st = pk.topk_async(x, k, 0.5, s).wait()
            else:
                v, i, st = pk.topk(x, k, 0.5, s)
            ost = check_oracle(st, v, i, h, k, 0.5, s, f"{form} n={n} k={k} seed={s}")
            assert torch.equal(v, ref[0]) and torch.equal(i, ref[1])
            assert all(st[key] == ref[2][key] for key in STAT_KEYS), (s, st, ref[2])
            if ost.path == PK.PATH_FILTER:
                launches.add(st["launches"])
        redrawn += ost.attempts > 1 and ost.path == PK.PATH_FILTER
    assert redrawn > 0, "no seed needed a redraw"
    # Redrawn rows finished on the device: no launch after the report.
    assert len(launches) == 1, launches


def test_device_redraws_in_flight(pk, cuda_device):
    # Calls in flight back to back, several of them redrawn on the device.
    x = workloads.normal((1 << 22) + 4, 5, cuda_device)
    h = x.cpu().numpy()
    pk.set_option(pk.OPT_SPECULATIVE, 5)
    pend = [pk.topk_async(x, 300, 0.5, s) for s in range(12)]
    attempts = []
    for s, p in enumerate(pend):
        v, i, st = p.wait()
        check_oracle(st, v, i, h, 300, 0.5, s, f"in flight seed={s}")
        attempts.append(st["attempts"])
    assert max(attempts) > 1


@pytest.mark.parametrize("off", [0, 1])
def test_tie_rows_kept_for_the_tie_exit(pk, cuda_device, off):
    # 16 levels: attempt 0 settles the row for the tie exit; the later
    # attempts must leave its state (tau, counts, the filter's bookkeeping)
    # to the tie step.  Offset 1: the selection-based tie step.
    n = 1 << 22
    base = workloads.levels16(n + 8, 3, cuda_device)
    x = base[off:off + n]
    h = x.cpu().numpy()
    pk.set_option(pk.OPT_SPECULATIVE, 3)
    for k in (100, 9000):
        for form in ("async", "sync"):
            v, i, st = pk.topk_async(x, k, 1e-3, 7).wait() if form == "async" else pk.topk(x, k, 1e-3, 7)
            ost = check_oracle(st, v, i, h, k, 1e-3, 7, f"tie {form} k={k} offset {off}")
            assert ost.path == PK.PATH_TIE


def test_batched_rows_settle_independently(pk, cuda_device):
    # Rows that pass at once, rows redrawn on the device and tie rows, in one
    # call: each row equals the oracle's at eps / rows.
    rows, n, k, eps = 4, 1 << 21, 200, 0.99
    x = torch.empty((rows, n), dtype=torch.float32, device=cuda_device)
    x[0] = workloads.normal(n, 1, cuda_device)
    x[1] = workloads.levels16(n, 2, cuda_device)
    x[2] = workloads.normal(n, 3, cuda_device)
    x[3] = workloads.normal(n, 4, cuda_device)
    h = x.cpu().numpy()
    pk.set_option(pk.OPT_SPECULATIVE, 5)
    seen = set()
    for seed in range(10):
        for form in ("async", "sync"):
            if form == "async":
                vals, idx, sts = pk.topk_batched_async(x, k, eps, seed).wait()
            else:
                vals, idx, sts = pk.topk_batched(x, k, eps, seed)
            for r in range(rows):
                ost = check_oracle(sts[r], vals[r], idx[r], np.ascontiguousarray(h[r]), k, eps / rows, seed,
                                   f"{form} row {r} seed {seed}", row=r, rows=rows)
                seen.add((ost.path, ost.attempts > 1))
    assert (PK.PATH_TIE, False) in seen and (PK.PATH_FILTER, True) in seen, seen


def test_capped_by_max_attempts(pk, cuda_device):
    # Two attempts at most: one speculative attempt, then the exact fallback
    # for the rows that failed both.
    x = workloads.normal((1 << 22) + 4, 23, cuda_device)
    h = x.cpu().numpy()
    pk.set_option(pk.OPT_SPECULATIVE, 5)
    pk.set_option(pk.OPT_MAX_ATTEMPTS, 2)
    paths = set()
    for s in range(16):
        v, i, st = pk.topk_async(x, 300, 0.5, s).wait()
        ost = check_oracle(st, v, i, h, 300, 0.5, s, f"capped seed={s}", max_attempts=2)
        paths.add(ost.path)
    assert PK.PATH_FALLBACK in paths and PK.PATH_FILTER in paths


def test_nan_settles_the_row(pk, cuda_device):
    x = workloads.normal(1 << 22, 3, cuda_device)
    x[777] = float("nan")
    pk.set_option(pk.OPT_SPECULATIVE, 3)
    for call in (lambda: pk.topk(x, 64, 1e-3, 1), lambda: pk.topk_async(x, 64, 1e-3, 1).wait()):
        with pytest.raises(pk.ProfkError) as e:
            call()
        assert e.value.code == -3

