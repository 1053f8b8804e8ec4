"""Pins of the oracle's exact top-k (definition) to brute force and closed forms."""
import numpy as np
import pytest

import workloads
from oracle.topk import same_result, topk_chunked, topk_partition, topk_rows, topk_sort

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def brute_force(x, k):
    """Repeated argmax; a strict '>' keeps the lower index among equal values."""
    rem = list(range(len(x)))
    out = []
    for _ in range(k):
        best = rem[0]
        for i in rem[1:]:
            if float(x[i]) > float(x[best]):
                best = i
        out.append(best)
        rem.remove(best)
    idx = np.array(out, dtype=np.int64)
    return x[idx], idx


def tie_heavy(rng, n):
    pool = np.array([0.0, -0.0, 1.5, -1.5, np.inf, -np.inf, 3.25, 7.0], dtype=np.float32)
    return pool[rng.integers(0, pool.size, n)]


@pytest.mark.parametrize("seed", range(12))
def test_sort_and_partition_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 120))
    x = tie_heavy(rng, n) if seed % 2 else rng.standard_normal(n).astype(np.float32)
    for k in sorted({1, n, max(1, n // 3), int(rng.integers(1, n + 1))}):
        bv, bi = brute_force(x, k)
        sv, si = topk_sort(x, k)
        pv, pi = topk_partition(x, k)
        assert same_result(sv, si, bv, bi)
        assert same_result(pv, pi, bv, bi)
        for chunks in (1, 3, 7):
            assert same_result(*topk_chunked(x, k, workers=2, chunks=chunks), bv, bi)


def test_zero_signs_are_equal_and_bits_are_kept():
    x = np.array([-0.0, 0.0, -0.0, -1.0], dtype=np.float32)
    v, i = topk_sort(x, 3)
    assert list(i) == [0, 1, 2]
    assert list(v.view(np.uint32)) == [0x80000000, 0x00000000, 0x80000000]


def test_nan_is_rejected():
    x = np.array([1.0, np.nan, 2.0], dtype=np.float32)
    with pytest.raises(ValueError):
        topk_sort(x, 1)
    with pytest.raises(ValueError):
        topk_partition(x, 1)


def test_partition_matches_sort_on_medium_inputs():
    for seed, gen in enumerate(["uniform", "levels16", "ulps_below_one", "pareto", "sorted_normal"]):
        x = workloads.GENERATORS[gen](50_000, seed, "cpu").numpy()
        for k in (1, 17, 4096, 50_000):
            assert same_result(*topk_sort(x, k), *topk_partition(x, k)), (gen, k)


def test_chunked_matches_sort_on_medium_inputs():
    # Ties straddling chunk boundaries (16 levels, the 256 ulps below 1.0), k
    # larger than a chunk, and more chunks than threads.
    for seed, gen in enumerate(["levels16", "ulps_below_one", "normal", "sorted_normal"]):
        x = workloads.GENERATORS[gen](50_001, seed, "cpu").numpy()
        for k in (1, 17, 4096, 20_000, 50_001):
            for workers, chunks in ((4, None), (3, 16)):
                assert same_result(*topk_sort(x, k), *topk_chunked(x, k, workers, chunks)), (gen, k, chunks)


def test_closed_form_ulps_below_one():
    # Tie stress (a): the k largest are the first k indices holding bits 0x3F7FFFFF.
    x = workloads.ulps_below_one(1 << 16, 3, "cpu").numpy()
    k = 64
    top = np.flatnonzero(x.view(np.uint32) == 0x3F7FFFFF)
    assert top.size >= k
    v, i = topk_sort(x, k)
    assert np.array_equal(i, top[:k])
    assert np.all(v.view(np.uint32) == 0x3F7FFFFF)


def test_closed_form_levels16():
    # Tie stress (b): the first k indices of the top level 15/16.
    x = workloads.levels16(1 << 16, 4, "cpu").numpy()
    k = 1024
    top = np.flatnonzero(x == np.float32(15 / 16))
    v, i = topk_sort(x, k)
    assert np.array_equal(i, top[:k])


def test_closed_form_sorted_ascending():
    # Tie stress (c): indices n-1, n-2, ... with equal-value runs in ascending index order.
    x = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 2.0, 3.0], dtype=np.float32)
    v, i = topk_sort(x, 5)
    assert list(i) == [6, 3, 4, 5, 1]
    x = workloads.sorted_normal(10_000, 5, "cpu").numpy()
    v, i = topk_sort(x, 100)
    n = x.size
    expect = []
    j = n - 1
    while len(expect) < 100:
        s = j
        while s > 0 and x[s - 1] == x[j]:
            s -= 1
        expect.extend(range(s, j + 1))
        j = s - 1
    assert list(i) == expect[:100]


def test_rows():
    x = workloads.normal_rows(3, 1000, 9, "cpu").numpy()
    v, i = topk_rows(x, 10)
    for r in range(3):
        assert same_result(v[r], i[r], *brute_force(x[r], 10))
