"""Each step of the CUDA path against the oracle, through the C-ABI.

Sizes span several tiles of every kernel plus a ragged tail; edge cases cover
ties, +-0, +-inf, NaN, tau = -inf / +inf and the buffer overflow."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same, decode_keys
from oracle import philox as PX
from oracle import profk as PK
from oracle.topk import topk_sort

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,S,seed,row,attempt", [
    (1 << 22, 32768, 1, 0, 0), (1 << 22, 32768, 2, 5, 3), (1000003, 4099, 77, 1, 0), (64, 32, 9, 0, 0),
    (1 << 30, 105985, 3, 0, 0), (3 * (1 << 20) + 17, 131072, 4, 2, 1), (50331648, 131072, 8, 0, 0),
    # more than 1024 positions per CTA of the persistent form: the step-by-step kernel
    (1 << 24, 400_000, 5, 3, 2), (1 << 20, 1 << 19, 6, 0, 0), ((1 << 21) + 5, 300_001, 7, 1, 4),
    # the whole row (a permutation of it), tiny rows, and rows of one element
    (5000, 5000, 10, 0, 0), (3, 2, 11, 1, 1), (1, 1, 12, 0, 0), ((1 << 32) - 5, 1000, 13, 0, 0)])
@pytest.mark.parametrize("form", ["auto", "steps", "lists"])
def test_sample_matches_oracle(pk, cuda_device, n, S, seed, row, attempt, form):
    """Every kernel form draws the oracle's sample, index by index in order
    (rows off the power-of-two grid walk the permutation's cycles); the lists
    form takes S up to 2^19."""
    pk.set_option(pk.OPT_SAMPLER, {"auto": pk.SAMPLER_AUTO, "steps": pk.SAMPLER_STEPS, "lists": pk.SAMPLER_LISTS}[form])
    x = workloads.uniform(n, seed, cuda_device)
    sidx, svals = pk.sample(x, S, seed, row, attempt)
    ref = PX.sample_indices(n, S, seed, row, attempt)
    got = sidx.cpu().numpy()
    assert np.array_equal(got, ref)
    assert torch.equal(svals, x[sidx])


def _vals(kind, S, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return rng.standard_normal(S).astype(np.float32)
    if kind == "ties":
        return rng.integers(-3, 4, S).astype(np.float32)
    pool = np.float32([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, 2.5e-40, -2.5e-40])  # subnormals too
    return pool[rng.integers(0, pool.size, S)]


@pytest.mark.parametrize("kind", ["normal", "ties", "specials"])
@pytest.mark.parametrize("S", [1, 7, 4096, 32768, 131072])
def test_threshold_matches_oracle(pk, cuda_device, kind, S):
    v = _vals(kind, S, S)
    tv = torch.from_numpy(v).to(cuda_device)
    for t in sorted({1, min(2, S), max(1, S // 3), S}):
        got = float(pk.threshold(tv, t).item())
        ref = float(PK.threshold(v, t))
        assert got == ref, (t, got, ref)


@pytest.mark.parametrize("n", [1, 3, 4, 1000, 16384, 16385, 65536 * 3 + 5, (1 << 22) + 7])
def test_filter_counts_and_buffer(pk, cuda_device, n):
    x = workloads.normal(n, n, cuda_device)
    h = x.cpu().numpy()
    for q in (0.0, 0.5, 0.99, 0.9999):
        tau = np.float32(np.quantile(h, q)) if n > 1 else np.float32(h[0])
        for M in (0, 5, 10 ** 6):
            keys, counts = pk.filter_pass(x, float(tau), M)
            vals, idx, R, R_gt = PK.filter_pass(h, tau, 10 ** 9)
            c = counts.cpu().numpy()
            assert (int(c[0]), int(c[1]), int(c[2])) == (R, R_gt, 0)
            if M >= R:
                ok, gi = decode_keys(keys[:R])
                order = np.argsort(gi)
                assert np.array_equal(gi[order], idx)
            elif M > 0:
                _, gi = decode_keys(keys)
                assert np.unique(gi).size == M and np.all(h[gi] >= tau)


def test_filter_edge_thresholds_and_nan(pk, cuda_device):
    n = 100_003
    x = workloads.normal(n, 5, cuda_device)
    keys, counts = pk.filter_pass(x, float("-inf"), 10)
    assert counts.cpu().tolist() == [n, n, 0]
    keys, counts = pk.filter_pass(x, float("inf"), 10)
    assert counts.cpu().tolist() == [0, 0, 0]
    y = x.clone()
    y[[0, 777, n - 1]] = float("nan")
    y[5] = float("inf")
    keys, counts = pk.filter_pass(y, float("inf"), 10)
    assert counts.cpu().tolist() == [1, 0, 3]
    z = torch.tensor([-0.0, 0.0, -0.0, -1.0, 1.0], device=cuda_device)
    keys, counts = pk.filter_pass(z, 0.0, 10)
    assert counts.cpu().tolist() == [4, 1, 0]
    keys, counts = pk.filter_pass(z, -0.0, 10)
    assert counts.cpu().tolist() == [4, 1, 0]


@pytest.mark.parametrize("n,k", [(200_000, 1), (200_000, 100), (200_000, 8192), (300_000, 8193), (300_000, 40000)])
def test_refine_matches_oracle(pk, cuda_device, n, k):
    x = workloads.levels16(n, k, cuda_device) if k % 2 else workloads.normal(n, k, cuda_device)
    h = x.cpu().numpy()
    tau = float(np.partition(h, n - k - 1000)[n - k - 1000]) if n > k + 1000 else float(h.min())
    keys, counts = pk.filter_pass(x, tau, n)
    R = int(counts[0].item())
    assert R >= k
    v, i = pk.refine(keys[:R].contiguous(), k, x)
    bvals, bidx, R2, _ = PK.filter_pass(h, np.float32(tau), n)
    rv, ri = PK.refine(bvals, bidx, k)
    assert_same(v, i, rv, ri, "refine")


@pytest.mark.parametrize("n,k", [(1, 1), (5, 5), (1000, 1), (1000, 1000), (65537, 9000), (1 << 20, 17),
                                 ((1 << 20) + 3, 1 << 15),
                                 # one CTA per row: placed by counting (k <= 512) or sorted, ragged tails
                                 (1 << 16, 512), ((1 << 17) + 2, 513), (65537, 2048), (200_003, 100)])
@pytest.mark.parametrize("kind", ["normal", "levels16", "specials"])
def test_exact_matches_oracle(pk, cuda_device, n, k, kind):
    if kind == "specials":
        rng = np.random.default_rng(n)
        pool = np.float32([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, 1e-45, 3.0])
        h = pool[rng.integers(0, pool.size, n)]
        x = torch.from_numpy(h).to(cuda_device)
    else:
        x = workloads.GENERATORS[kind](n, n + k, cuda_device)
        h = x.cpu().numpy()
    v, i = pk.exact(x, k)
    assert_same(v, i, *topk_sort(h, k), f"exact {kind} n={n} k={k}")


def test_exact_rejects_nan(pk, cuda_device):
    x = workloads.normal(5000, 1, cuda_device)
    x[1234] = float("nan")
    with pytest.raises(pk.ProfkError) as e:
        pk.exact(x, 10)
    assert e.value.code == -3


def test_exact_unaligned_input(pk, cuda_device):
    """profk_exact on a row that does not start on a 16-byte boundary: the
    selection reads it element by element and the result is the same."""
    base = workloads.normal((1 << 20) + 8, 41, cuda_device)
    x = base[1:(1 << 20) + 1]  # 4 bytes past an aligned start
    assert x.data_ptr() % 16 == 4
    for k in (10, 5000):
        vals, idx = pk.exact(x, k)
        assert_same(vals, idx, *topk_sort(x.cpu().numpy(), k), f"unaligned exact k={k}")
