"""Full-size workloads, in the launch configuration the benchmark times.

The oracle's O(N) form of the definition (``topk_partition``) computes the
reference; smaller k are prefixes of the sorted top-k_max, which holds by the
definition of the order."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from oracle.topk import topk_partition

pytestmark = pytest.mark.gpu

SEEDS = (1000, 1001)


def run_config(pk, x, ks, eps=1e-3, seeds=SEEDS):
    h = x.cpu().numpy()
    kmax = max(ks)
    rv, ri = topk_partition(h, kmax)
    for k in ks:
        for s in seeds:
            vals, idx, st = pk.topk(x, k, eps, s)
            assert_same(vals, idx, rv[:k], ri[:k], f"n={h.size} k={k} seed={s} stats={st}")
            yield k, st


@pytest.mark.parametrize("gen", ["uniform", "normal", "pareto"])
def test_2p30(pk, cuda_device, gen):
    x = workloads.GENERATORS[gen](1 << 30, 3, cuda_device)
    for k, st in run_config(pk, x, [32, 1024, 1 << 19]):
        assert st["path"] in (pk.PATH_FILTER, pk.PATH_TIE) or st["attempts"] > 1
    del x
    torch.cuda.empty_cache()


def test_2p26_normal(pk, cuda_device):
    x = workloads.normal(1 << 26, 2, cuda_device)
    list(run_config(pk, x, [32, 1024, 32768], seeds=(1, 2, 3)))


@pytest.mark.parametrize("gen", ["ulps_below_one", "levels16", "sorted_normal"])
def test_tie_stress_2p28(pk, cuda_device, gen):
    x = workloads.GENERATORS[gen](1 << 28, 4, cuda_device)
    for k, st in run_config(pk, x, [4096]):
        if gen != "sorted_normal":
            assert st["path"] == pk.PATH_TIE  # tau lands on the k-th value, R >> M
    del x
    torch.cuda.empty_cache()


def test_sae_selection(pk, cuda_device):
    x = workloads.sae_preacts(5, cuda_device)
    assert x.numel() == 50_331_648
    list(run_config(pk, x, [131_072]))


def test_batched_64_rows(pk, cuda_device):
    x = workloads.normal_rows(64, 1 << 24, 6, cuda_device)
    vals, idx, sts = pk.topk_batched(x, 32, 1e-3, 77)
    h = x.cpu().numpy()
    for r in range(64):
        rv, ri = topk_partition(np.ascontiguousarray(h[r]), 32)
        assert_same(vals[r], idx[r], rv, ri, f"row {r}")
    assert all(s["path"] == pk.PATH_FILTER for s in sts) or any(s["attempts"] > 1 for s in sts)
