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


@pytest.mark.parametrize("k", [32, 1024, 1 << 19])
def test_bench_protocol_async_2p30(pk, cuda_device, k):
    """The call the benchmark times, in its launch configuration: 20
    profk_topk_async calls in flight on the 2^30 standard-normal input (the
    bench's input seed), each with its own output buffers, completed by
    profk_wait in order; every call's values (bits), indices and order equal
    the oracle's."""
    x = workloads.normal(1 << 30, 1, cuda_device)
    rv, ri = topk_partition(x.cpu().numpy(), k)
    calls = 20
    outs = [(torch.empty(k, dtype=torch.float32, device=cuda_device),
             torch.empty(k, dtype=torch.int64, device=cuda_device)) for _ in range(calls)]
    pending = [pk.topk_async(x, k, 1e-3, 1000 + s, out=outs[s]) for s in range(calls)]
    for s, p in enumerate(pending):
        v, i, st = p.wait()
        assert_same(v, i, rv, ri, f"async call {s} k={k} stats={st}")
        assert st["path"] in (pk.PATH_FILTER, pk.PATH_TIE) or st["attempts"] > 1
    del x
    torch.cuda.empty_cache()
