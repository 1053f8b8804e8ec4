"""The refinement's sort paths for k > 8192, each against the oracle.

The sort of a row's candidate keys counts them into buckets sized from the
data and then sorts every bucket of at most 256 keys with one warp, or, when
some bucket holds more (a value repeated hundreds to thousands of times among
the candidates), whole-bucket ranges of up to 8191 keys with one CTA; beyond
4096 copies of one value it falls back to the radix passes.  An "atom" of c
copies of one large value planted in a normal row puts all c copies in one
bucket, so c = 0, 1000, 3000 and 6000 take the three paths in turn; the
exact path (every key of the row sorted for k) and the filter path (the
buffer sorted) are both covered."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from oracle.topk import topk_sort

pytestmark = pytest.mark.gpu


def with_atom(n, copies, value, seed, device):
    x = workloads.normal(n, seed, device)
    if copies:
        g = torch.Generator(device=device)
        g.manual_seed(seed + 77)
        pos = torch.randperm(n, generator=g, device=device)[:copies]
        x[pos] = value
    return x


@pytest.mark.parametrize("copies", [0, 1000, 3000, 6000])
@pytest.mark.parametrize("k", [10_000, 60_000])
def test_filter_path_sort_with_atom(pk, cuda_device, copies, k):
    n = 1 << 22
    x = with_atom(n, copies, 3.0, 31, cuda_device)
    vals, idx, st = pk.topk(x, k, 1e-3, 5)
    ov, oi = topk_sort(x.cpu().numpy(), k)
    assert_same(vals, idx, ov, oi, f"atom of {copies} copies, k={k}, stats={st}")


@pytest.mark.parametrize("copies", [0, 1000, 3000, 6000])
def test_exact_path_sort_with_atom(pk, cuda_device, copies):
    n, k = 600_000, 30_000
    x = with_atom(n, copies, 2.5, 32, cuda_device)
    vals, idx = pk.exact(x, k)
    ov, oi = topk_sort(x.cpu().numpy(), k)
    assert_same(vals, idx, ov, oi, f"exact path, atom of {copies} copies")


def test_atom_of_signed_zeros(pk, cuda_device):
    # -0.0 and +0.0 are one value for the order: 3000 of each mixed, ordered by index.
    n, k = 1 << 20, 200_000
    x = workloads.normal(n, 33, cuda_device).abs()
    g = torch.Generator(device=cuda_device)
    g.manual_seed(9)
    pos = torch.randperm(n, generator=g, device=cuda_device)[:6000]
    x[pos[:3000]] = 0.0
    x[pos[3000:]] = -0.0
    x[x > 0.1] = 0.0  # k reaches far into the zeros (a tie at the k boundary)
    vals, idx, st = pk.topk(x, k, 1e-3, 6)
    ov, oi = topk_sort(x.cpu().numpy(), k)
    assert_same(vals, idx, ov, oi, f"signed zeros, stats={st}")
