"""Seeded random shapes through the whole call, against the oracle.

Each case draws a shape (rows, row length, row stride and start offset, k,
eps, input distribution, seed) from a fixed generator, so the cases are the
same on every run.  Together they reach every form of every step (the grid,
lists and step-by-step samplers; the filter's aligned and unaligned
instantiations and its tie bookkeeping; the refinement's shortcuts, its grid
and one-CTA forms and the buffer sort; the tie exit, the exact routes, the
redraws).  Every row's result must equal the oracle procedure's: values as
bits, indices and order, and the path, attempts and first counts.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from oracle.topk import topk_sort
from routing import oracle_profk

pytestmark = pytest.mark.gpu

GENS = ("uniform", "normal", "pareto", "ulps_below_one", "levels16", "sorted_normal")
CASES = 40
BUDGET = 1 << 24  # elements per case, rows x n, so that the oracle stays quick


def draw(case):
    rng = np.random.default_rng(90_000 + case)
    rows = int(rng.choice([1, 1, 1, 1, 2, 3, 5, 9, 17, 40, 130]))
    n_max = max(16, BUDGET // rows)
    lo = 1 << 18 if rng.random() < 0.75 and n_max > (1 << 18) else 16  # mostly rows long enough to sample
    n = int(min(n_max, np.exp(rng.uniform(np.log(lo), np.log(n_max)))))
    off = int(rng.integers(0, 4)) if rng.random() < 0.3 else 0
    ld = n + (int(rng.integers(0, 5)) if rows > 1 else 0)
    k_max = min(n, 30_000)
    k = int(min(k_max, max(1, np.exp(rng.uniform(0, np.log(k_max))))))
    eps = float(rng.choice([1e-3, 1e-3, 1e-2, 0.2]))
    gen = str(rng.choice(GENS))
    seed = int(rng.integers(0, 2**31))
    return rows, n, off, ld, k, eps, gen, seed


@pytest.mark.parametrize("case", range(CASES))
def test_random_shape(pk, cuda_device, case):
    rows, n, off, ld, k, eps, gen, seed = draw(case)
    base = workloads.GENERATORS[gen](rows * ld + off + 4, case, cuda_device)
    what = f"case {case}: rows={rows} n={n} ld={ld} off={off} k={k} eps={eps} {gen}"
    if rows == 1:
        x = base[off:off + n]
        v, i, st = pk.topk(x, k, eps, seed)
        ov, oi, ost = oracle_profk(x.cpu().numpy(), k, eps, seed)
        assert_same(v, i, ov, oi, what)
        assert (st["path"], st["attempts"], st["R_first"]) == (ost.path, ost.attempts, ost.R_first), (what, st)
        return
    x = base[off:off + rows * ld].view(rows, ld)[:, :n]
    v, i, sts = pk.topk_batched(x, k, eps, seed)
    h = x.cpu().numpy()
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, eps / rows, seed, row=r, rows=rows)
        assert_same(v[r], i[r], ov, oi, f"{what} row {r}")
        assert (sts[r]["path"], sts[r]["attempts"], sts[r]["R_first"]) == (ost.path, ost.attempts, ost.R_first), \
            (what, r, sts[r])


OPTION_CASES = 30


def draw_options(case):
    rng = np.random.default_rng(95_000 + case)
    rows = int(rng.choice([1, 1, 2, 5, 24]))
    n_max = max(16, (1 << 23) // rows)
    lo = 1 << 17 if rng.random() < 0.8 and n_max > (1 << 17) else 16
    n = int(min(n_max, np.exp(rng.uniform(np.log(lo), np.log(n_max)))))
    ld = n + (int(rng.integers(0, 3)) if rows > 1 else 0)
    k = int(min(n, max(1, np.exp(rng.uniform(0, np.log(min(n, 20_000)))))))
    eps = float(rng.choice([1e-3, 0.05, 0.3]))
    gen = str(rng.choice(GENS))
    seed = int(rng.integers(0, 2**31))
    opts = {"sampler": int(rng.choice([0, 1, 2, 3])), "spec": int(rng.choice([0, 0, 2, 5])),
            "tie_exit": bool(rng.random() < 0.8), "max_attempts": int(rng.choice([1, 2, 6, 6])),
            "api": str(rng.choice(["sync", "async"]))}
    return rows, n, ld, k, eps, gen, seed, opts


@pytest.mark.parametrize("case", range(OPTION_CASES))
def test_random_options(pk, cuda_device, case):
    """Seeded shapes under seeded options: the sampler form forced, redraws
    enqueued on the device, the tie exit off, few attempts before the exact
    fallback, the asynchronous form.  None of them changes a row's result,
    path or attempts from the oracle procedure's."""
    rows, n, ld, k, eps, gen, seed, o = draw_options(case)
    pk.set_option(pk.OPT_SAMPLER, o["sampler"])
    pk.set_option(pk.OPT_SPECULATIVE, o["spec"])
    pk.set_option(pk.OPT_TIE_EXIT, int(o["tie_exit"]))
    pk.set_option(pk.OPT_MAX_ATTEMPTS, o["max_attempts"])
    base = workloads.GENERATORS[gen](rows * ld + 4, 500 + case, cuda_device)
    what = f"case {case}: rows={rows} n={n} ld={ld} k={k} eps={eps} {gen} {o}"
    kw = {"tie_exit": o["tie_exit"], "max_attempts": o["max_attempts"]}
    if rows == 1:
        x = base[:n]
        if o["api"] == "sync":
            v, i, st = pk.topk(x, k, eps, seed)
        else:
            v, i, st = pk.topk_async(x, k, eps, seed).wait()
        ov, oi, ost = oracle_profk(x.cpu().numpy(), k, eps, seed, **kw)
        assert_same(v, i, ov, oi, what)
        assert (st["path"], st["attempts"]) == (ost.path, ost.attempts), (what, st)
        return
    x = base[:rows * ld].view(rows, ld)[:, :n]
    if o["api"] == "sync":
        v, i, sts = pk.topk_batched(x, k, eps, seed)
    else:
        v, i, sts = pk.topk_batched_async(x, k, eps, seed).wait()
    h = x.cpu().numpy()
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, eps / rows, seed, row=r, rows=rows, **kw)
        assert_same(v[r], i[r], ov, oi, f"{what} row {r}")
        assert (sts[r]["path"], sts[r]["attempts"]) == (ost.path, ost.attempts), (what, r, sts[r])


SEGMENT_CASES = 16


def draw_segmented(case):
    rng = np.random.default_rng(97_000 + case)
    rows = int(rng.choice([1, 1, 2, 3]))
    n = int(rng.integers((1 << 16) + 1, 1 << 21))
    seg = max(1 << 16, 4 * int(rng.integers(1 << 14, max((1 << 14) + 1, n // 8))))  # a multiple of 4, >= 2^16
    off = int(rng.integers(0, 4)) if rng.random() < 0.4 else 0
    ld = n + (int(rng.integers(0, 5)) if rows > 1 else 0)
    k = int(min(n, max(1, np.exp(rng.uniform(0, np.log(min(n, 50_000)))))))
    gen = str(rng.choice(GENS))
    seed = int(rng.integers(0, 2**31))
    return rows, n, off, ld, seg, k, gen, seed


@pytest.mark.parametrize("case", range(SEGMENT_CASES))
def test_random_segmented(pk, cuda_device, case):
    """Seeded rows split into segments (the split point lowered to a random
    multiple of 4), starting anywhere, with any row stride: each row's
    merged result must be its exact top k (values as bits, indices, order)."""
    rows, n, off, ld, seg, k, gen, seed = draw_segmented(case)
    pk.set_option(pk.OPT_MAX_SEGMENT, seg)
    base = workloads.GENERATORS[gen](rows * ld + off + 4, 700 + case, cuda_device)
    what = f"case {case}: rows={rows} n={n} off={off} ld={ld} segment={seg} k={k} {gen}"
    if rows == 1:
        x = base[off:off + n]
        v, i, _ = pk.topk(x, k, 1e-3, seed)
        assert_same(v, i, *topk_sort(x.cpu().numpy(), k), what)
        return
    x = base[off:off + rows * ld].view(rows, ld)[:, :n]
    v, i, _ = pk.topk_batched(x, k, 1e-3, seed)
    h = x.cpu().numpy()
    for r in range(rows):
        assert_same(v[r], i[r], *topk_sort(np.ascontiguousarray(h[r]), k), f"{what} row {r}")
