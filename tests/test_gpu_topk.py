"""The whole Prof-K call (profk_topk / profk_topk_batched) against the oracle.

Besides the output (bit-exact values, indices and order), the per-attempt
statistics must equal the oracle procedure's: the same draw stream gives the
same sample, the same threshold and the same exact counts."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from oracle import params as PP
from oracle import profk as PK
from routing import oracle_profk, uses_filter
from oracle.topk import topk_sort

pytestmark = pytest.mark.gpu


def check_call(pk, x, k, eps, seed, force=None, tie_exit=True, max_attempts=6):
    if force:
        pk.set_option(pk.OPT_FORCE_S, force.get("S", 0))
        pk.set_option(pk.OPT_FORCE_T, force.get("t", 0))
        pk.set_option(pk.OPT_FORCE_M, force.get("M", 0))
    pk.set_option(pk.OPT_TIE_EXIT, int(tie_exit))
    pk.set_option(pk.OPT_MAX_ATTEMPTS, max_attempts)
    vals, idx, st = pk.topk(x, k, eps, seed)
    h = x.cpu().numpy()
    ov, oi, ost = oracle_profk(h, k, eps, seed, force=force, tie_exit=tie_exit, max_attempts=max_attempts)
    assert_same(vals, idx, ov, oi, f"n={h.size} k={k} seed={seed} force={force}")
    assert (st["S"], st["t"], st["M"]) == (ost.S, ost.t, ost.M)
    assert st["path"] == ost.path, (st, ost)
    assert st["attempts"] == ost.attempts
    assert st["R_first"] == ost.R_first and st["R_gt_first"] == ost.R_gt_first
    assert st["R_final"] == ost.R_final and st["R_gt_final"] == ost.R_gt_final
    if ost.taus:
        assert st["tau_first"] == ost.taus[0]
    return st


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_uniform_2p22_k32(pk, cuda_device, seed):
    x = workloads.uniform(1 << 22, seed, cuda_device)
    for s in range(4):
        st = check_call(pk, x, 32, 1e-3, 1000 + s)
        assert st["path"] == pk.PATH_FILTER


@pytest.mark.parametrize("gen,n,k", [("normal", 1 << 20, 64), ("pareto", 3_000_017, 100), ("levels16", 1 << 21, 16),
                                     ("ulps_below_one", 1 << 22, 64), ("sorted_normal", 1 << 22, 1000),
                                     ("uniform", (1 << 23) + 5, 1)])
def test_distributions(pk, cuda_device, gen, n, k):
    x = workloads.GENERATORS[gen](n, n % 1000, cuda_device)
    for s in range(3):
        check_call(pk, x, k, 1e-3, 7 + s)


@pytest.mark.parametrize("force,tie_exit,attempts", [
    ({"S": 4096, "t": 4096, "M": 100}, True, 6),   # tau = sample min: overflow every attempt -> fallback
    ({"S": 4096, "t": 1, "M": 40}, True, 6),       # tau = sample max: recall failure, redraws
    ({"S": 4096, "t": 3, "M": 5000}, True, 6),
    ({"S": 2048, "t": 2, "M": 64}, True, 2),
    ({"S": 4096, "t": 5, "M": 3000}, False, 6),
    ({"S": 4096, "t": 5, "M": 3000}, True, 0),     # straight to the exact fallback
])
def test_forced_paths(pk, cuda_device, force, tie_exit, attempts):
    x = workloads.normal((1 << 20) + 3, 4, cuda_device)
    for s in range(3):
        check_call(pk, x, 32, 1e-3, 50 + s, force=force, tie_exit=tie_exit, max_attempts=attempts)


@pytest.mark.parametrize("tie_exit", [True, False])
def test_tie_path(pk, cuda_device, tie_exit):
    # 40 distinct values above a level holding most of the input: tau lands on the
    # level, R >> M while R_gt < k.
    n, k = (1 << 20) + 11, 100
    x = torch.full((n,), 0.5, device=cuda_device)
    top = torch.randperm(n, device=cuda_device)[:40]
    x[top] = torch.rand(40, device=cuda_device) + 1.0
    x[torch.randperm(n, device=cuda_device)[:1000]] = 0.25
    st = check_call(pk, x, k, 1e-3, 5, force={"S": 4096}, tie_exit=tie_exit)
    assert st["path"] == (pk.PATH_TIE if tie_exit else pk.PATH_FALLBACK)


def test_exact_route_small_inputs(pk, cuda_device):
    for n, k in [(1, 1), (10, 3), (1000, 1000), (1 << 16, 64), (200_000, 5000)]:
        x = workloads.normal(n, n, cuda_device)
        vals, idx, st = pk.topk(x, k, 1e-3, 1)
        assert st["path"] == pk.PATH_EXACT and st["attempts"] == 0
        assert_same(vals, idx, *topk_sort(x.cpu().numpy(), k), f"exact route n={n} k={k}")


@pytest.mark.parametrize("n,k", [((1 << 22) + 8, 1 << 17), (1 << 22, 1 << 20), (1 << 21, (1 << 21) - 3),
                                 (1_000_003, 400_000)])
def test_dense_k(pk, cuda_device, n, k):
    """k a large share of the row: the filter path while its parameters can
    meet the budget (here k/n = 1/32, 1/4 and 0.4), the exact path when k
    nearly equals n; every statistic as the oracle procedure predicts."""
    x = workloads.normal(n, 17, cuda_device)
    st = check_call(pk, x, k, 1e-3, 8)
    S, t, M = PP.params(n, k, 1e-3)
    assert st["path"] == (pk.PATH_FILTER if uses_filter(n, k, S, t, M) else pk.PATH_EXACT)


def test_nan_rejected(pk, cuda_device):
    x = workloads.normal(1 << 20, 3, cuda_device)
    x[12345] = float("nan")
    with pytest.raises(pk.ProfkError) as e:
        pk.topk(x, 64, 1e-3, 1)
    assert e.value.code == -3
    y = workloads.normal(1000, 3, cuda_device)
    y[3] = float("nan")
    with pytest.raises(pk.ProfkError) as e:
        pk.topk(y, 10, 1e-3, 1)
    assert e.value.code == -3


def test_special_values(pk, cuda_device):
    n = 1 << 20
    x = workloads.normal(n, 8, cuda_device)
    x[:1000] = 0.0
    x[1000:2000] = -0.0
    x[5] = float("inf")
    x[77] = float("inf")
    x[9] = float("-inf")
    for k in (1, 2, 3, 64):
        check_call(pk, x, k, 1e-3, 3)
    y = torch.zeros(n, device=cuda_device)
    y[::2] = -0.0
    check_call(pk, y, 64, 1e-3, 3, force={"S": 4096})


def test_reproducible(pk, cuda_device):
    x = workloads.normal(1 << 22, 1, cuda_device)
    a = pk.topk(x, 1000, 1e-3, 42)
    b = pk.topk(x, 1000, 1e-3, 42)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and a[2]["R_first"] == b[2]["R_first"]


def test_nondefault_stream(pk, cuda_device):
    x = workloads.normal(1 << 21, 2, cuda_device)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        vals, idx, st = pk.topk(x, 500, 1e-3, 9)
    s.synchronize()
    assert_same(vals, idx, *topk_sort(x.cpu().numpy(), 500), "side stream")


@pytest.mark.parametrize("rows,n,ld,k", [(4, 1 << 20, 1 << 20, 16), (3, 1_000_003, 1_000_008, 100),
                                         (16, 1 << 18, 1 << 18, 1), (2, 5000, 5000, 5000),
                                         (3, 1 << 22, 1 << 22, 10_000),
                                         # several chunks of more than 1024 draws per row
                                         (24, 1 << 20, 1 << 20, 64), (40, 1 << 19, (1 << 19) + 4, 5),
                                         # exact routing, one CTA per row (several rows per CTA for 700)
                                         (64, 1 << 16, (1 << 16) + 4, 1000), (700, 20_000, 20_004, 64)])
def test_batched(pk, cuda_device, rows, n, ld, k):
    base = workloads.normal_rows(rows, ld, rows + n, cuda_device)
    x = base[:, :n]
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 11)
    h = x.cpu().numpy()
    eps_row = 1e-3 / rows
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, eps_row, 11, row=r, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"batched row {r}")
        assert sts[r]["path"] == ost.path and sts[r]["R_first"] == ost.R_first
        assert sts[r]["R_gt_first"] == ost.R_gt_first
        if ost.taus:
            assert sts[r]["tau_first"] == ost.taus[0]


SAMPLER_FORMS = ("grid", "steps", "lists")


def sampler_option(pk, form):
    return {"grid": pk.SAMPLER_GRID, "steps": pk.SAMPLER_STEPS, "lists": pk.SAMPLER_LISTS}[form]


@pytest.mark.parametrize("form", SAMPLER_FORMS)
@pytest.mark.parametrize("rows,n,k", [(5, 1 << 20, 64), (12, (1 << 18) + 3, 700), (3, 3 * (1 << 20) + 8, 20_000),
                                      (2, 1 << 24, 32)])
def test_batched_sampler_forms(pk, cuda_device, form, rows, n, k):
    """Every form of the sampling kernels (the persistent grid kernel, the
    step-by-step kernels, the lists kernel where t <= 8) gives every row the
    oracle's sample: the same tau and counts.  The third shape draws about
    137,000 times per row."""
    pk.set_option(pk.OPT_SAMPLER, sampler_option(pk, form))
    ld = (n + 3) // 4 * 4  # row stride a multiple of 4 elements
    x = workloads.normal_rows(rows, ld, 3 * rows + k, cuda_device)[:, :n]
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 21)
    h = x.cpu().numpy()
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, 1e-3 / rows, 21, row=r, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"{form} row {r}")
        assert (sts[r]["path"], sts[r]["R_first"], sts[r]["R_gt_first"]) == (ost.path, ost.R_first, ost.R_gt_first)
        assert sts[r]["tau_first"] == ost.taus[0]


def test_batched_rows_retry_alone(pk, cuda_device):
    # Forced parameters that make roughly half the rows fail their first attempt.
    rows, n, k = 8, 1 << 18, 40
    x = workloads.normal_rows(rows, n, 99, cuda_device)
    force = {"S": 2048, "t": 1, "M": 2000}
    for o, v in ((pk.OPT_FORCE_S, 2048), (pk.OPT_FORCE_T, 1), (pk.OPT_FORCE_M, 2000)):
        pk.set_option(o, v)
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 5)
    h = x.cpu().numpy()
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, 1e-3 / rows, 5, row=r, force=force, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"row {r}")
        assert (sts[r]["attempts"], sts[r]["path"], sts[r]["R_first"]) == (ost.attempts, ost.path, ost.R_first)


@pytest.mark.parametrize("gen,n,k", [("normal", 1 << 24, 8193), ("normal", 1 << 24, 1 << 18),
                                     ("uniform", (1 << 24) + 3, 20_000), ("pareto", 1 << 24, 100_000),
                                     ("sorted_normal", 1 << 23, 1 << 16), ("levels16", 1 << 23, 50_000)])
def test_large_k(pk, cuda_device, gen, n, k):
    """k beyond one CTA's sort: the filter buffer is radix-sorted (levels16
    takes the tie path, whose k selected keys are radix-sorted)."""
    x = workloads.GENERATORS[gen](n, 17, cuda_device)
    for s in range(2):
        check_call(pk, x, k, 1e-3, 90 + s)


@pytest.mark.parametrize("gen,n,k,force", [
    # tau's top buckets hold nearly every sample key (all three passes run)
    ("ulps_below_one", 1 << 22, 4096, {"S": 131072, "t": 300}),
    ("levels16", 1 << 22, 4096, {"S": 131072, "t": 300}),  # one level's copies: 1/16 of the sample
    ("uniform", (1 << 22) + 3, 4096, {"S": 131072, "t": 300}),
    ("normal", 1 << 22, 4096, {"S": 262144, "t": 9}),  # t just above the candidate lists' range
    ("normal", 5000, 100, {"S": 1500, "t": 40}),  # a sample of a few chunks, the last one short
])
def test_sampler_passes_for_larger_t(pk, cuda_device, gen, n, k, force):
    """For t > 8 the sampler selects tau by radix passes over the sample
    keys; it finds the oracle's tau, and the oracle's counts and result
    follow, for tau buckets of every size."""
    x = workloads.GENERATORS[gen](n, 23, cuda_device)
    for s in range(2):
        check_call(pk, x, k, 1e-3, 40 + s, force=force)


def test_large_k_fallback(pk, cuda_device):
    x = workloads.normal(1 << 22, 5, cuda_device)
    st = check_call(pk, x, 20_000, 1e-3, 3, force={"S": 32768, "t": 1}, max_attempts=2)
    assert st["path"] == pk.PATH_FALLBACK


@pytest.mark.parametrize("form", ("auto",) + SAMPLER_FORMS)
def test_batched_wide_sampler_rows_retry_alone(pk, cuda_device, form):
    # 32 rows share the SMs, so each row's CTAs hold thousands of draws; about
    # half the rows overflow each attempt and redraw alone (a row list).
    rows, n, k = 32, 1 << 20, 1
    if form != "auto":
        pk.set_option(pk.OPT_SAMPLER, sampler_option(pk, form))
    x = workloads.normal_rows(rows, n, 41, cuda_device)
    force = {"S": 32768, "t": 1, "M": 22}
    for o, v in ((pk.OPT_FORCE_S, 32768), (pk.OPT_FORCE_T, 1), (pk.OPT_FORCE_M, 22)):
        pk.set_option(o, v)
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 8)
    h = x.cpu().numpy()
    retried = 0
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, 1e-3 / rows, 8, row=r, force=force, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"row {r}")
        assert (sts[r]["attempts"], sts[r]["path"], sts[r]["R_first"], sts[r]["tau_first"]) == \
            (ost.attempts, ost.path, ost.R_first, ost.taus[0])
        retried += sts[r]["attempts"] > 1
    assert retried > 0


def test_batched_fallback_rows(pk, cuda_device):
    # tau = the sample minimum overflows the buffer on every attempt: all rows
    # take the exact fallback (one CTA per row at this size), some rows tied.
    rows, n, k = 40, 1 << 17, 100
    x = workloads.normal_rows(rows, n, 63, cuda_device)
    x[3] = torch.round(x[3] * 4) / 4
    force = {"S": 4096, "t": 4096, "M": 100}
    for o, v in ((pk.OPT_FORCE_S, 4096), (pk.OPT_FORCE_T, 4096), (pk.OPT_FORCE_M, 100), (pk.OPT_MAX_ATTEMPTS, 2)):
        pk.set_option(o, v)
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 2)
    h = x.cpu().numpy()
    for r in range(rows):
        assert_same(vals[r], idx[r], *topk_sort(h[r], k), f"row {r}")
        assert sts[r]["path"] == pk.PATH_FALLBACK and sts[r]["attempts"] == 2


def test_batched_large_k_rows_retry_alone(pk, cuda_device):
    # About half the rows fail each attempt, so the radix sort runs on row lists.
    rows, n, k = 4, 1 << 20, 9000
    x = workloads.normal_rows(rows, n, 77, cuda_device)
    force = {"S": 8192, "t": 71, "M": 11000}
    for o, v in ((pk.OPT_FORCE_S, 8192), (pk.OPT_FORCE_T, 71), (pk.OPT_FORCE_M, 11000)):
        pk.set_option(o, v)
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 6)
    h = x.cpu().numpy()
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, 1e-3 / rows, 6, row=r, force=force, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"row {r}")
        assert (sts[r]["attempts"], sts[r]["path"], sts[r]["R_first"]) == (ost.attempts, ost.path, ost.R_first)


def test_caller_workspace(pk, cuda_device):
    x = workloads.normal((1 << 22) + 8, 12, cuda_device)
    k = 1000
    ref = pk.topk(x, k, 1e-3, 3)
    need = pk.workspace_size(1, x.numel(), k)
    buf = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    pk.set_workspace(buf)
    got = pk.topk(x, k, 1e-3, 3)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    assert got[2]["R_first"] == ref[2]["R_first"] and got[2]["path"] == ref[2]["path"]
    # Batched rows through the same buffer when it is big enough, else refused.
    xb = workloads.normal_rows(3, 1 << 20, 4, cuda_device)
    if pk.workspace_size(3, 1 << 20, 64) <= need:
        vb, ib, _ = pk.topk_batched(xb, 64, 1e-3, 2)
        for r in range(3):
            assert_same(vb[r], ib[r], *topk_sort(xb[r].cpu().numpy(), 64), f"row {r}")
    small = torch.empty(need // 2 & ~255, dtype=torch.uint8, device=cuda_device)
    pk.set_workspace(small)
    with pytest.raises(pk.ProfkError) as e:
        pk.topk(x, k, 1e-3, 3)
    assert e.value.code == -6
    pk.set_workspace(None)
    again = pk.topk(x, k, 1e-3, 3)
    assert torch.equal(again[1], ref[1])


@pytest.mark.parametrize("rows,n,k", [(1, 1 << 20, 100), (16, 393712, 5937), (3, 1 << 20, 40)])
def test_no_attempts_on_a_dirty_workspace(pk, cuda_device, rows, n, k):
    """With no attempt allowed every row goes straight to the exact fallback,
    before any attempt has set up its state: the call must not read whatever
    the workspace held (a caller's buffer filled with ones here)."""
    x = workloads.sorted_normal(rows * n, 324, cuda_device).view(rows, n)
    buf = torch.full((pk.workspace_size(rows, n, k, 0.5),), 0xFF, dtype=torch.uint8, device=cuda_device)
    pk.set_workspace(buf)
    pk.set_option(pk.OPT_MAX_ATTEMPTS, 0)
    try:
        vals, idx, sts = pk.topk_batched(x, k, 0.5, 2064010536)
    finally:
        pk.set_workspace(None)
    h = x.cpu().numpy()
    for r in range(rows):
        assert_same(vals[r], idx[r], *topk_sort(h[r], k), f"row {r}")
        assert (sts[r]["path"], sts[r]["attempts"]) == (pk.PATH_FALLBACK, 0), sts[r]


@pytest.mark.parametrize("rows,n,k", [(1024, 1 << 16, 16), (256, 1 << 20, 32), (512, (1 << 18) + 4, 100),
                                      (128, 1 << 21, 32), (160, (1 << 20) + 8, 2049)])
def test_batched_many_rows(pk, cuda_device, rows, n, k):
    """Many rows sharing the SMs: exact routing (one CTA per row) for rows
    whose sample would be 1/32 of the row or more, else the filter path with
    one sampler CTA per row."""
    x = workloads.normal_rows(rows, n, rows + k, cuda_device)
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 21)
    rng = np.random.default_rng(rows)
    for r in sorted(set(rng.integers(0, rows, 8).tolist()) | {0, rows - 1}):
        h = x[r].cpu().numpy()
        assert_same(vals[r], idx[r], *topk_sort(h, k), f"row {r}")
    paths = {s["path"] for s in sts}
    S, t, M = sts[0]["S"], sts[0]["t"], sts[0]["M"]
    assert paths == ({pk.PATH_FILTER} if uses_filter(n, k, S, t, M, rows) else {pk.PATH_EXACT})


def test_exact_parameter_mode(pk, cuda_device):
    """Theorem 4's exact t and M (PROFK_PARAMS_EXACT) through the whole call."""
    x = workloads.normal((1 << 22) + 12, 9, cuda_device)
    pk.set_option(pk.OPT_PARAM_MODE, pk.PARAMS_EXACT)
    h = x.cpu().numpy()
    for k in (32, 1000):
        vals, idx, st = pk.topk(x, k, 1e-3, 4)
        ov, oi, ost = oracle_profk(h, k, 1e-3, 4, mode=2)
        assert_same(vals, idx, ov, oi, f"exact-parameter mode k={k}")
        assert (st["S"], st["t"], st["M"]) == (ost.S, ost.t, ost.M)
        assert st["R_first"] == ost.R_first and st["attempts"] == ost.attempts


@pytest.mark.parametrize("n,k", [((1 << 22) + 12, 32), ((1 << 22) + 12, 1000), (1 << 24, 4096)])
def test_corrected_parameter_mode(pk, cuda_device, n, k):
    """The corrected Algorithm 1 throughout (PROFK_PARAMS_CORRECTED: its own
    sample size, from Proposition 7 with the GB300 cost ratio)."""
    x = workloads.normal(n, 10, cuda_device)
    pk.set_option(pk.OPT_PARAM_MODE, pk.PARAMS_CORRECTED)
    h = x.cpu().numpy()
    vals, idx, st = pk.topk(x, k, 1e-3, 5)
    ov, oi, ost = oracle_profk(h, k, 1e-3, 5, mode=PP.MODE_CORRECTED)
    assert_same(vals, idx, ov, oi, f"corrected-parameter mode n={n} k={k}")
    assert (st["S"], st["t"], st["M"]) == (ost.S, ost.t, ost.M) == PP.params(n, k, 1e-3, PP.MODE_CORRECTED)
    assert st["R_first"] == ost.R_first and st["attempts"] == ost.attempts and st["path"] == ost.path


STAT_KEYS = ("S", "t", "M", "R_first", "R_gt_first", "tau_first", "R_final", "attempts", "path")


def test_async_matches_oracle_and_sync(pk, cuda_device):
    """Asynchronous calls in flight together: each equals the oracle procedure
    (result, path and counts) and the synchronous call's statistics."""
    x = workloads.normal((1 << 22) + 4, 21, cuda_device)
    h = x.cpu().numpy()
    calls = ((1, 32), (2, 1000), (3, 5000), (4, 20000))
    ref = [pk.topk(x, k, 1e-3, s) for s, k in calls]
    pend = [pk.topk_async(x, k, 1e-3, s) for s, k in calls]  # all in flight at once
    for p, r, (s, k) in zip(pend, ref, calls):
        v, i, st = p.wait()
        ov, oi, ost = oracle_profk(h, k, 1e-3, s)
        assert_same(v, i, ov, oi, f"async k={k} seed={s}")
        assert (st["S"], st["t"], st["M"], st["path"], st["attempts"]) == (ost.S, ost.t, ost.M, ost.path, ost.attempts)
        assert (st["R_first"], st["R_gt_first"], st["tau_first"]) == (ost.R_first, ost.R_gt_first, ost.taus[0])
        assert all(st[key] == r[2][key] for key in STAT_KEYS), (st, r[2])


def test_async_rerun_when_not_cleared(pk, cuda_device):
    # 16 levels: tau lands on a level, R > M, the check does not clear the
    # first attempt and the call runs again (tie exit).
    x = workloads.levels16(1 << 20, 3, cuda_device)
    h = x.cpu().numpy()
    for k in (100, 5000):
        v, i, st = pk.topk_async(x, k, 1e-3, 5).wait()
        ov, oi, ost = oracle_profk(h, k, 1e-3, 5)
        assert_same(v, i, ov, oi, f"async tie k={k}")
        assert st["path"] == ost.path and st["attempts"] == ost.attempts


def test_async_resumes_redraws(pk, cuda_device):
    # eps = 0.5: many first attempts fail the check; the asynchronous call
    # continues from its first attempt (redraw, then the filter again) and
    # must end exactly as the synchronous call: result and every statistic.
    x = workloads.normal((1 << 20) + 4, 23, cuda_device)
    h = x.cpu().numpy()
    redraws = 0
    for seed in range(12):
        ref = pk.topk(x, 300, 0.5, seed)
        v, i, st = pk.topk_async(x, 300, 0.5, seed).wait()
        ov, oi, ost = oracle_profk(h, 300, 0.5, seed)
        assert_same(v, i, ov, oi, f"resumed async seed={seed}")
        assert (st["attempts"], st["path"], st["R_final"]) == (ost.attempts, ost.path, ost.R_final)
        assert torch.equal(v, ref[0]) and torch.equal(i, ref[1])
        assert all(st[key] == ref[2][key] for key in STAT_KEYS + ("R_gt_final",)), (seed, st, ref[2])
        redraws += st["attempts"] > 1
    assert redraws > 0  # the resumed path was taken


def test_async_batched_mixed_rows(pk, cuda_device):
    # Rows that clear the check in the first attempt and tie rows that take
    # the tie exit after it, in one asynchronous call.
    n = 1 << 19
    x = torch.empty((4, n), dtype=torch.float32, device=cuda_device)
    x[0] = workloads.normal(n, 1, cuda_device)
    x[1] = workloads.levels16(n, 2, cuda_device)
    x[2] = workloads.normal(n, 3, cuda_device)
    x[3] = workloads.levels16(n, 4, cuda_device)
    ref = pk.topk_batched(x, 700, 1e-3, 9)
    v, i, sts = pk.topk_batched_async(x, 700, 1e-3, 9).wait()
    assert torch.equal(v, ref[0]) and torch.equal(i, ref[1])
    for a, b in zip(sts, ref[2]):
        assert all(a[key] == b[key] for key in STAT_KEYS), (a, b)
    assert {s["path"] for s in sts} == {pk.PATH_FILTER, pk.PATH_TIE}


def test_async_nan(pk, cuda_device):
    x = workloads.normal(1 << 20, 3, cuda_device)
    x[777] = float("nan")
    p = pk.topk_async(x, 64, 1e-3, 1)
    with pytest.raises(pk.ProfkError) as e:
        p.wait()
    assert e.value.code == -3


@pytest.mark.parametrize("rows,n,k", [(3, 1 << 20, 50), (80, 1 << 18, 20)])
def test_async_batched(pk, cuda_device, rows, n, k):
    x = workloads.normal_rows(rows, n, 8, cuda_device)
    ref = pk.topk_batched(x, k, 1e-3, 2)
    v, i, sts = pk.topk_batched_async(x, k, 1e-3, 2).wait()
    assert torch.equal(v, ref[0]) and torch.equal(i, ref[1])
    assert [s["R_first"] for s in sts] == [s["R_first"] for s in ref[2]]


@pytest.mark.parametrize("rows,zeros,k", [(1, 120, 40), (100, 120, 40), (100, 1500, 1000), (1, 3000, 2000)])
def test_signed_zeros_at_the_top(pk, cuda_device, rows, zeros, k):
    """Rows whose largest values are copies of +0.0 and -0.0 (equal as
    values; the candidate key keeps no sign, so the refinement reads each
    zero back from x): the output keeps every zero's own sign bit, in index
    order.  The cases take the refinement's forms: few candidates placed at
    once (one row; 100 rows), one CTA per row with its passes and its sorted
    list (100 rows, 1500 zeros), the grid passes (one row, 3000 zeros)."""
    n = 1 << 21
    base = -torch.abs(workloads.normal_rows(rows, n, 12, "cpu")) - 1e-3
    for r in range(rows):
        g = torch.Generator().manual_seed(1000 + r)
        pos = torch.randperm(n, generator=g)[:zeros]
        base[r, pos[:zeros // 2]] = 0.0
        base[r, pos[zeros // 2:]] = -0.0
    x = base.to(cuda_device)
    h = base.numpy()
    if rows == 1:
        vals, idx, st = pk.topk(x[0], k, 1e-3, 5)
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[0]), k, 1e-3, 5)
        assert_same(vals, idx, ov, oi, "one row")
        assert st["path"] == ost.path
        return
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 5)
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, 1e-3 / rows, 5, row=r, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"row {r}")
        assert sts[r]["path"] == ost.path


# (generator, rows, n, k, M): the grid form of the refinement on one row and
# on three, and its one-CTA-per-row form (80 rows); S and t forced so that R
# (about n t / S) is far above the few-candidates shortcut, M above R.
PREFIX_CASES = {"grid_row": ("normal", 1, 1 << 22, 1000, 100_000), "grid_rows": ("uniform", 3, 1 << 20, 500, 40_000),
                "solo_rows": ("normal", 80, 1 << 18, 64, 10_000)}


@pytest.mark.parametrize("keep", [1, 9, 20])
@pytest.mark.parametrize("case", list(PREFIX_CASES))
def test_refinement_prefix_check_restarts(pk, cuda_device, case, keep):
    """The grid refinement's first digit starts below the high bits that the
    filter records every candidate sharing with tau, and its first pass
    checks that.  Told to trust only the low keep - 1 bits of the record, it
    assumes a longer shared prefix than the candidates have (keep = 1: tau's
    whole value), must find a key outside it and start the passes again from
    the top bit; the result is the oracle's all the same."""
    gen, rows, n, k, M = PREFIX_CASES[case]
    force = {"S": 4096, "t": 64, "M": M}
    x = workloads.GENERATORS[gen](rows * n, 17, cuda_device).view(rows, n)
    pk.set_option(pk.OPT_FORCE_S, force["S"])
    pk.set_option(pk.OPT_FORCE_T, force["t"])
    pk.set_option(pk.OPT_FORCE_M, force["M"])
    pk.set_option(pk.OPT_PREFIX_TEST, keep)
    if rows == 1:
        v, i, st = pk.topk(x[0], k, 1e-3, 8)
        v, i, sts = v[None], i[None], [st]
    else:
        v, i, sts = pk.topk_batched(x, k, 1e-3, 8)
    h = x.cpu().numpy()
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, 1e-3 / rows, 8, row=r, rows=rows, force=force)
        assert_same(v[r], i[r], ov, oi, f"{case} keep={keep} row {r}")
        assert (sts[r]["path"], sts[r]["attempts"], sts[r]["R_first"]) == (ost.path, ost.attempts, ost.R_first)
        assert sts[r]["path"] == pk.PATH_FILTER and sts[r]["R_first"] > 2048
