"""The tie exit after the filter pass, in both of its forms, against the oracle.

When the filter finds R > M elements >= tau but only R_gt < k above tau, tau
is the k-th largest value and the top-k is every x > tau plus the lowest-index
copies of tau.  A row whose sample holds tau more than once (a heavily tied
top) is filtered with the tie step's bookkeeping: per-block counts of tau and
every x > tau that the full buffer drops.  Its tie exit then needs no second
pass over the row.  A row that takes the tie exit without that hint gets the
counting pass instead.  Which form a row takes is decided here from the
oracle's own sample (the copies of tau among the sampled values), so the
tests know that both forms ran; each result is compared with the oracle bit
for bit, with the path, attempts and counts."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_same
from oracle import philox as PX
from oracle import profk as PK
from routing import oracle_profk

pytestmark = pytest.mark.gpu


def tied_top(n, copies, above, seed, device):
    """Clipped normal values (at most 3.5), `copies` copies of 4.0 and `above`
    distinct values in (4.5, 5) at random positions."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(n, generator=g).clamp_(-3.5, 3.5)
    pos = torch.randperm(n, generator=g)
    x[pos[:copies]] = 4.0
    x[pos[copies:copies + above]] = 4.5 + 0.5 * (torch.arange(above, dtype=torch.float32) + 1) / (above + 1)
    return x.to(device)


def sample_copies_of_tau(h, S, t, seed, attempt, row=0):
    """Copies of the attempt's tau among its sampled values (the oracle's sample)."""
    sv = h[PX.sample_indices(h.size, S, seed, row, attempt)]
    tau = PK.threshold(sv, t)
    return int(np.count_nonzero(sv == tau))


def run(pk, x, k, seed, force=None, eps=1e-3, sampler=None):
    pk.reset_options()
    if sampler is not None:
        pk.set_option(pk.OPT_SAMPLER, sampler)
    if force:
        pk.set_option(pk.OPT_FORCE_S, force.get("S", 0))
        pk.set_option(pk.OPT_FORCE_T, force.get("t", 0))
        pk.set_option(pk.OPT_FORCE_M, force.get("M", 0))
    vals, idx, st = pk.topk(x, k, eps, seed)
    h = x.cpu().numpy()
    ov, oi, ost = oracle_profk(h, k, eps, seed, force=force)
    assert_same(vals, idx, ov, oi, f"k={k} seed={seed} force={force} stats={st}")
    assert (st["path"], st["attempts"], st["R_first"], st["R_gt_first"], st["R_final"], st["R_gt_final"]) == \
        (ost.path, ost.attempts, ost.R_first, ost.R_gt_first, ost.R_final, ost.R_gt_final)
    return st, ost, h


def test_both_tie_forms_from_one_input(pk, cuda_device):
    """A tiny forced sample (S = 256, t = 1) catches the 6000 copies of 4.0 once
    for some seeds (the counting pass) and twice or more for others (the
    bookkeeping); 30 x > tau, most of them dropped after the buffer (M = 400)
    has filled, the rest in the buffer."""
    n, k = 1 << 20, 200
    x = tied_top(n, 6000, 30, 11, cuda_device)
    force = {"S": 256, "t": 1, "M": 400}
    forms = set()
    for seed in range(24):
        st, ost, h = run(pk, x, k, seed, force)
        if st["path"] != pk.PATH_TIE:
            continue
        assert st["R_gt_final"] == 30
        forms.add(sample_copies_of_tau(h, 256, 1, seed, st["attempts"] - 1) >= 2)
    assert forms == {False, True}


@pytest.mark.parametrize("copies,above,k", [(20_000, 0, 3000), (20_000, 1, 3000), (20_000, 700, 3000),
                                            (20_000, 2000, 3000), (30_000, 5000, 8000)])
def test_tie_exit_with_bookkeeping(pk, cuda_device, copies, above, k):
    """The default parameters: the sample holds hundreds of copies of tau.
    The x > tau count spans 0, 1 and sorted prefixes of 1024, 2048 and 8192
    keys, with the copies of tau after them in index order."""
    n = (1 << 21) + 12
    x = tied_top(n, copies, above, copies + above, cuda_device)
    for seed in (1, 2):
        st, ost, h = run(pk, x, k, seed)
        assert st["path"] == pk.PATH_TIE and st["R_gt_final"] == above
        assert sample_copies_of_tau(h, st["S"], st["t"], seed, st["attempts"] - 1) >= 2


def test_tied_sample_on_the_filter_path(pk, cuda_device):
    """Integer values with about 21 copies each and a quarter of the row
    sampled: tau has several copies in the sample, so the row is filtered with
    the bookkeeping, yet R lands in [k, M] and the refinement finishes it."""
    n, k = 1 << 20, 500
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    x = torch.randint(0, 50_000, (n,), generator=g).to(torch.float32).to(cuda_device)
    hinted = 0
    for seed in range(4):
        st, ost, h = run(pk, x, k, seed, {"S": 1 << 18})
        assert st["path"] == pk.PATH_FILTER
        hinted += sample_copies_of_tau(h, st["S"], st["t"], seed, 0) >= 2
    assert hinted >= 3


def test_batched_rows_mix_the_forms(pk, cuda_device):
    """Rows with a tied top (bookkeeping), plain normal rows and an integer row
    in one batched call: each loop of the filter skips the other's rows."""
    rows, n, k = 6, 1 << 20, 300
    parts = []
    for r in range(rows):
        if r % 3 == 0:
            parts.append(tied_top(n, 9000, 40 + r, 100 + r, "cpu"))
        elif r % 3 == 1:
            g = torch.Generator(device="cpu")
            g.manual_seed(200 + r)
            parts.append(torch.randn(n, generator=g))
        else:
            g = torch.Generator(device="cpu")
            g.manual_seed(300 + r)
            parts.append(torch.randint(0, 4000, (n,), generator=g).to(torch.float32))
    x = torch.stack(parts).to(cuda_device)
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 9)
    h = x.cpu().numpy()
    paths = set()
    for r in range(rows):
        ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, 1e-3 / rows, 9, row=r, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"row {r}")
        assert (sts[r]["path"], sts[r]["attempts"], sts[r]["R_first"], sts[r]["R_gt_first"]) == \
            (ost.path, ost.attempts, ost.R_first, ost.R_gt_first)
        paths.add(sts[r]["path"])
    assert pk.PATH_TIE in paths and pk.PATH_FILTER in paths


def test_batched_rows_take_both_tie_forms_in_one_attempt(pk, cuda_device):
    """Twelve tied rows with a tiny forced sample: in the same attempt some rows
    hold tau once in their sample (the counting pass) and others more often
    (the bookkeeping), so both tie flows run in one call, one after the other
    on their own row lists."""
    rows, n, k = 12, 1 << 20, 200
    force = {"S": 256, "t": 1, "M": 400}
    x = torch.stack([tied_top(n, 6000, 30, 500 + r, "cpu") for r in range(rows)]).to(cuda_device)
    for o, v in ((pk.OPT_FORCE_S, 256), (pk.OPT_FORCE_T, 1), (pk.OPT_FORCE_M, 400)):
        pk.set_option(o, v)
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 17)
    h = x.cpu().numpy()
    forms_by_attempt = {}
    for r in range(rows):
        hr = np.ascontiguousarray(h[r])
        ov, oi, ost = oracle_profk(hr, k, 1e-3 / rows, 17, row=r, force=force, rows=rows)
        assert_same(vals[r], idx[r], ov, oi, f"row {r}")
        assert (sts[r]["path"], sts[r]["attempts"], sts[r]["R_final"], sts[r]["R_gt_final"]) == \
            (ost.path, ost.attempts, ost.R_final, ost.R_gt_final)
        if ost.path == PK.PATH_TIE:
            copies = sample_copies_of_tau(hr, 256, 1, 17, ost.attempts - 1, row=r)
            forms_by_attempt.setdefault(ost.attempts, set()).add(copies >= 2)
    assert any(f == {False, True} for f in forms_by_attempt.values()), forms_by_attempt


@pytest.mark.parametrize("force", [{"S": 256, "t": 1, "M": 400}, {"S": 4096, "t": 8, "M": 400},
                                   {"S": 20_000, "t": 5, "M": 400}])
def test_lists_sampler_routes_ties_like_the_grid_form(pk, cuda_device, force):
    """The lists form of the sampler (forced) gives every seed the oracle's
    result and the persistent form's statistics, kernel launches included.
    The launches tell whether the row went through the filter's bookkeeping
    (tau at least twice in the sample) or the counting pass, so both forms
    count the copies of tau alike, across 1, 16 and 79 chunks."""
    n, k = 1 << 20, 200
    x = tied_top(n, 6000, 30, 11, cuda_device)
    paths = set()
    for seed in range(12):
        st_grid, ost, h = run(pk, x, k, seed, force)
        st_lists, _, _ = run(pk, x, k, seed, force, sampler=pk.SAMPLER_LISTS)
        assert st_lists == st_grid, (seed, st_lists, st_grid)
        paths.add(st_lists["path"])
    assert pk.PATH_TIE in paths
