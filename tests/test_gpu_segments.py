"""Rows longer than a candidate key's index reaches: split into segments, merged.

A row of more than 2^32 elements is split into contiguous segments whose exact
top-k lists are merged by value and global index (the paper's Table 4 runs
single rows of up to 4.3e9 elements).  PROFK_OPT_MAX_SEGMENT lowers the split
point so that the same code runs on rows the full-sort oracle finishes in
seconds: several segments, a shorter last segment, ties and signed zeros that
straddle segment borders, k above a segment's length.  The full-size case is a
single row of 4.3e9 standard-normal elements against the oracle's O(N) form."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from oracle.topk import topk_partition, topk_rows, topk_sort

pytestmark = pytest.mark.gpu

SEG = 1 << 16


def host_available_bytes() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def straddling_ties(n, seed, device):
    """Eight levels plus signed zeros and infinities, so that equal values sit in
    every segment and the k boundary falls inside a run of equal values."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    lv = torch.randint(0, 8, (n,), generator=g, device=device).to(torch.float32) - 4.0
    lv[lv == 0] = -0.0
    lv[torch.randint(0, n, (64,), generator=g, device=device)] = float("inf")
    lv[torch.randint(0, n, (64,), generator=g, device=device)] = -float("inf")
    lv[torch.randint(0, n, (256,), generator=g, device=device)] = 0.0
    return lv


@pytest.mark.parametrize("n,k", [(4 * SEG, 100), (4 * SEG + 12, 1), (1_000_003, 1000), (5 * SEG + 1, 70_000),
                                 (3 * SEG + 8, 3 * SEG + 8), (SEG + 4, SEG + 1)])
@pytest.mark.parametrize("gen", ["normal", "levels16", "ties"])
def test_segmented_row_matches_oracle(pk, cuda_device, n, k, gen):
    pk.set_option(pk.OPT_MAX_SEGMENT, SEG)
    x = straddling_ties(n, 5, cuda_device) if gen == "ties" else workloads.GENERATORS[gen](n, 5, cuda_device)
    vals, idx, st = pk.topk(x, k, 1e-3, 11)
    ov, oi = topk_sort(x.cpu().numpy(), k)
    assert_same(vals, idx, ov, oi, f"segmented n={n} k={k} {gen} stats={st}")
    assert st["attempts"] >= 0 and st["launches"] >= 1


def test_segmented_batched_rows(pk, cuda_device):
    pk.set_option(pk.OPT_MAX_SEGMENT, SEG)
    rows, n, ld, k = 3, 300_001, 300_004, 500
    x = workloads.normal(rows * ld, 6, cuda_device).view(rows, ld)[:, :n]
    vals, idx, sts = pk.topk_batched(x, k, 1e-3, 3)
    ov, oi = topk_rows(x.cpu().numpy(), k)
    for r in range(rows):
        assert_same(vals[r], idx[r], ov[r], oi[r], f"segmented batched row {r}")
    assert len(sts) == rows


def test_segmented_async_and_caller_workspace(pk, cuda_device):
    pk.set_option(pk.OPT_MAX_SEGMENT, SEG)
    n, k = 700_001, 300
    x = workloads.levels16(n, 7, cuda_device)
    ov, oi = topk_sort(x.cpu().numpy(), k)
    v1, i1, s1 = pk.topk_async(x, k, 1e-3, 9).wait()
    assert_same(v1, i1, ov, oi, "segmented async")
    need = pk.workspace_size(1, n, k, 1e-3)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    pk.set_workspace(ws)
    v2, i2, s2 = pk.topk(x, k, 1e-3, 9)
    assert_same(v2, i2, ov, oi, "segmented in the caller's workspace")
    pk.set_workspace(torch.empty(need - 4096, dtype=torch.uint8, device=cuda_device))
    with pytest.raises(pk.ProfkError):
        pk.topk(x, k, 1e-3, 9)
    pk.set_workspace(None)


def test_segment_option_validated(pk):
    for bad in (-1, 4, (1 << 16) - 4, (1 << 16) + 2, (1 << 32) + 4):
        with pytest.raises(pk.ProfkError):
            pk.set_option(pk.OPT_MAX_SEGMENT, bad)
    pk.set_option(pk.OPT_MAX_SEGMENT, 1 << 20)
    assert pk.get_option(pk.OPT_MAX_SEGMENT) == 1 << 20


@pytest.mark.slow
def test_row_of_4_3e9(pk, cuda_device):
    """The paper's Table 4 size above 2^32 (4.3e9, standard normal, k = 2^10 and 2^18)
    through the default split point: two segments of 2.15e9."""
    n = 4_300_000_000
    if torch.cuda.get_device_properties(cuda_device).total_memory < 3 * 4 * n:
        pytest.skip("needs about 52 GB of device memory")
    if host_available_bytes() < 4 * 4 * n:
        pytest.skip("the oracle needs about 69 GB of free host memory")
    x = workloads.normal(n, 21, cuda_device)
    h = x.cpu().numpy()
    rv, ri = topk_partition(h, 1 << 18)
    del h
    for k in (1 << 10, 1 << 18):
        vals, idx, st = pk.topk(x, k, 1e-3, 5)
        assert_same(vals, idx, rv[:k], ri[:k], f"n=4.3e9 k={k} stats={st}")
        assert int(idx.max()) >= 1 << 32 or k < 1 << 12  # indices beyond 2^32 are reachable
        assert st["path"] == pk.PATH_FILTER
