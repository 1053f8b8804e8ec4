"""Pins of the oracle's generator and sampler.

Philox4x64-10 is checked against numpy's independent implementation
(numpy.random.Philox, which advances its 256-bit counter by one before each
block); Lemire's method exhaustively on 8-bit words; the sampler's subset law
against the uniform distribution on all S-subsets.
"""
import itertools
import math

import numpy as np
import pytest
from scipy import stats

from oracle import philox as PX


def numpy_philox_block(ctr, key):
    c = list(ctr)
    # numpy generates block (counter + 1); step the counter back by one.
    for w in range(4):
        if c[w] > 0:
            c[w] -= 1
            break
        c[w] = (1 << 64) - 1
    bg = np.random.Philox(counter=np.array(c, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
    return [int(v) for v in bg.random_raw(4)]


@pytest.mark.parametrize("ctr,key", [
    ((1, 0, 0, 0), (0, 0)),
    ((5, 3, 0, 0), (1234, 0)),
    ((123456789, 2, 7, 0), (2**63 + 5, 77)),
    ((2**64 - 1, 2**64 - 1, 3, 9), (2**64 - 1, 2**64 - 1)),
    ((0, 1, 0, 0), (99, 1)),
])
def test_philox_matches_numpy(ctr, key):
    assert PX.philox4x64_scalar(ctr, key) == numpy_philox_block(ctr, key)


def test_vectorised_philox_matches_scalar():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 2**63, size=(4, 64), dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    k0, k1 = 0xDEADBEEFCAFEF00D, 42
    out = PX.philox4x64(c[0], c[1], c[2], c[3], k0, k1)
    for j in range(64):
        ref = PX.philox4x64_scalar([int(c[w, j]) for w in range(4)], (k0, k1))
        assert [int(out[w][j]) for w in range(4)] == ref


def test_mulhilo64_exact():
    rng = np.random.default_rng(1)
    a = np.concatenate([rng.integers(0, 2**64 - 1, 200, dtype=np.uint64, endpoint=True),
                        np.array([0, 1, 2**32, 2**64 - 1, 2**63], dtype=np.uint64)])
    b = np.concatenate([rng.integers(0, 2**64 - 1, 200, dtype=np.uint64, endpoint=True),
                        np.array([2**64 - 1, 2**64 - 1, 2**32 - 1, 2**64 - 1, 3], dtype=np.uint64)])
    hi, lo = PX.mulhilo64(a, b)
    for x, y, h, l in zip(a, b, hi, lo):
        p = int(x) * int(y)
        assert int(h) == p >> 64 and int(l) == p & (2**64 - 1)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 7, 100, 129, 200, 255, 256])
def test_lemire_is_exactly_uniform_on_8bit_words(n):
    counts = np.zeros(n, dtype=np.int64)
    for w in range(256):
        v = PX.lemire_accept(w, n, bits=8)
        if v is not None:
            counts[v] += 1
    assert np.all(counts == 256 // n)


def test_lemire_64bit_rejection_zone():
    # n = 3: 2^64 mod 3 = 1, so exactly the words with w*3 mod 2^64 == 0 (w = 0) are rejected.
    assert PX.lemire_accept(0, 3) is None
    assert PX.lemire_accept(1, 3) == 0
    assert PX.lemire_accept(2**64 - 1, 3) == 2


def sequential_sample(n, S, seed, row=0, attempt=0):
    """Independent restatement: draw one at a time, skip repeats, stop at S."""
    out, seen, i = [], set(), 0
    while len(out) < S:
        j = 0
        while True:
            w = PX.philox4x64_scalar((i >> 2, attempt, j, 0), (seed, row))[i & 3]
            v = PX.lemire_accept(w, n)
            if v is not None:
                break
            j += 1
        if v not in seen:
            seen.add(v)
            out.append(v)
        i += 1
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("n,S,seed,row,attempt", [(1000, 50, 1, 0, 0), (37, 20, 5, 3, 2), (2**20, 300, 77, 1, 0),
                                                  (10, 10, 4, 0, 1)])
def test_sampler_matches_sequential_definition(n, S, seed, row, attempt):
    assert np.array_equal(PX.sample_indices(n, S, seed, row, attempt), sequential_sample(n, S, seed, row, attempt))


def test_draws_many_match_single():
    a = PX.draw_values_many(12345, [3, 9, 2**40], 2, 1, 500)
    for j, sd in enumerate([3, 9, 2**40]):
        assert np.array_equal(a[j], PX.draw_values(12345, sd, 2, 1, 0, 500))


def test_sample_is_a_uniform_subset():
    n, S, seeds = 8, 3, 14000
    subsets = {c: i for i, c in enumerate(itertools.combinations(range(n), S))}
    u = PX.draw_values_many(n, np.arange(seeds), 0, 0, 64)
    counts = np.zeros(len(subsets), dtype=np.int64)
    for r in range(seeds):
        _, first = np.unique(u[r], return_index=True)
        assert first.size >= S
        s = tuple(sorted(u[r][np.sort(first)[:S]]))
        counts[subsets[s]] += 1
    chi2 = stats.chisquare(counts)
    assert chi2.pvalue > 1e-4, chi2
    assert math.comb(n, S) == len(subsets)


def test_attempts_and_rows_give_different_streams():
    a = PX.sample_indices(1 << 20, 100, 5, 0, 0)
    b = PX.sample_indices(1 << 20, 100, 5, 0, 1)
    c = PX.sample_indices(1 << 20, 100, 5, 1, 0)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
