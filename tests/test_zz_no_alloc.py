"""profk_topk_noalloc, the entry point that allocates nothing.

Some callers cannot allocate on the call path: a latency-bounded serving loop
(an allocation can synchronize or stall the device), a plugin whose host owns
all device memory through its own allocator, a process whose pool already holds
nearly all of the GPU.  profk_topk_noalloc serves them from a fixed scratch
array reserved when the library loads.  These tests call it through the C-ABI,
twice in a row per problem (the second call finds the first call's leftovers in
the shared scratch), and require the oracle's result bit for bit, with the
oracle's path and counts, and the same output as profk_topk.  Problems of
different sizes follow one another, so that stale scratch contents from a
larger call meet a smaller one.

Kept in a file that pytest collects last, so that a failure here cannot stop a
run before the other tests; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from oracle import profk as PK
from oracle.topk import topk_partition
from routing import oracle_profk

pytestmark = pytest.mark.gpu


def check_twice(pk, x, k, seed, eps=1e-3, **oracle_kw):
    """Two no-alloc calls in a row against the oracle procedure and profk_topk."""
    h = x.cpu().numpy()
    ov, oi, ost = oracle_profk(h, k, eps, seed, **oracle_kw)
    ref_v, ref_i, _ = pk.topk(x, k, eps, seed)
    for call in range(2):
        v, i, st = pk.topk_noalloc(x, k, eps, seed)
        torch.cuda.synchronize()
        what = f"n={h.size} k={k} seed={seed} call {call}"
        assert_same(v, i, ov, oi, what)
        assert torch.equal(v.view(torch.int32), ref_v.view(torch.int32)) and torch.equal(i, ref_i), what
        assert (st["S"], st["t"], st["M"]) == (ost.S, ost.t, ost.M), what
        assert (st["path"], st["attempts"], st["R_first"], st["R_gt_first"]) == \
            (ost.path, ost.attempts, ost.R_first, ost.R_gt_first), (what, st, ost)
        if ost.taus:
            assert st["tau_first"] == ost.taus[0]
        assert st["aux_bytes"] == 0
    return st


@pytest.mark.parametrize("gen,n,k,path", [
    ("normal", 1 << 24, 1024, PK.PATH_FILTER),
    ("uniform", (1 << 22) + 3, 32, PK.PATH_FILTER),       # ragged tail
    ("levels16", 1 << 22, 100, PK.PATH_TIE),               # tau on the k-th value, R >> M
    ("normal", 1 << 16, 64, PK.PATH_EXACT),                # S > n/8: no sampling
    ("normal", 1 << 24, 1 << 14, PK.PATH_FILTER),          # k > 8192: sort without scratch
    ("normal", 1 << 17, 1 << 14, PK.PATH_EXACT),
])
def test_noalloc_matches_oracle_twice(pk, cuda_device, gen, n, k, path):
    x = workloads.GENERATORS[gen](n, 3, cuda_device)
    st = check_twice(pk, x, k, 17)
    assert st["path"] == path


def test_noalloc_forced_fallback_and_literal_retries(pk, cuda_device):
    # No attempts at all: the exact fallback at once.
    x = workloads.normal((1 << 20) + 4, 9, cuda_device)
    pk.set_option(pk.OPT_MAX_ATTEMPTS, 0)
    st = check_twice(pk, x, 500, 4, max_attempts=0)
    assert st["path"] == PK.PATH_FALLBACK and st["attempts"] == 0
    pk.set_option(pk.OPT_MAX_ATTEMPTS, 6)
    # Tie exit off: the 16-level input overflows every attempt, six redraws, then the fallback.
    y = workloads.levels16(1 << 21, 5, cuda_device)
    pk.set_option(pk.OPT_TIE_EXIT, 0)
    st = check_twice(pk, y, 300, 6, tie_exit=False)
    assert st["path"] == PK.PATH_FALLBACK and st["attempts"] == 6


def test_noalloc_after_a_larger_problem(pk, cuda_device):
    big = workloads.normal(1 << 24, 21, cuda_device)
    small = workloads.uniform((1 << 20) + 8, 22, cuda_device)
    check_twice(pk, big, 1 << 14, 1)
    check_twice(pk, small, 64, 2)
    check_twice(pk, big, 1000, 3)


def test_noalloc_full_size(pk, cuda_device):
    # The bench's input size: n = 2^30 at k = 1024 and 2^19 (the largest
    # headline k, whose problem still fits the 32 MiB scratch).
    x = workloads.normal(1 << 30, 3, cuda_device)
    rv, ri = topk_partition(x.cpu().numpy(), 1 << 19)
    for k in (1024, 1 << 19):
        for call in range(2):
            v, i, st = pk.topk_noalloc(x, k, 1e-3, 1000 + call)
            assert_same(v, i, rv[:k], ri[:k], f"2^30 k={k} call {call} stats={st}")
    del x
    torch.cuda.empty_cache()


def test_noalloc_rejects_problems_beyond_its_scratch(pk, cuda_device):
    n = 1 << 23  # k = n takes the exact path and needs 8 * 2^23 = 64 MiB of sort keys
    x = workloads.normal(n, 4, cuda_device)
    with pytest.raises(pk.ProfkError) as e:
        pk.topk_noalloc(x, n, 1e-3, 1)
    assert e.value.code == -6
    assert b"scratch" in pk.lib().profk_strerror(-6)
    # The scratch is still usable after the refusal.
    check_twice(pk, x, 77, 5)
