"""Pins of the oracle's generator and sampler.

Philox4x64-10 (numpy and C forms) is checked against numpy's independent
implementation (numpy.random.Philox, which advances its 256-bit counter by one
before each block).  The sampler's permutation is checked to be a bijection
(exhaustively on small domains), its C form equal to the numpy one element by
element, and its samples against the uniform law on S-subsets: the subset
frequencies, the position of each index, and the independence of rows and
attempts.  The Monte-Carlo test of Lemma 1 (tests/test_oracle_theory.py)
checks the law of the threshold rank it induces.
"""
import itertools
import math

import numpy as np
import pytest
from scipy import stats

from oracle import csample as CS
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


@pytest.mark.parametrize("ctr,key", [((1, 0, 0, 0), (0, 0)), ((5, 3, 0, 0), (1234, 0)),
                                     ((2**64 - 1, 2**64 - 1, 3, 9), (2**64 - 1, 2**64 - 1)),
                                     ((123456789, 2, 7, 0), (2**63 + 5, 77))])
def test_c_philox_matches_numpy(ctr, key):
    assert CS.philox4x64(ctr, key) == numpy_philox_block(ctr, key)


def test_domain_bits():
    for n in range(1, 2000):
        b = PX.domain_bits(n)
        assert b >= 2 and (1 << b) >= n and (b == 2 or (1 << (b - 1)) < n)
    for n in (2**30, 2**30 + 1, 2**32, 3 * 10**9):
        assert PX.domain_bits(n) == math.ceil(math.log2(n))


def test_round_keys_and_mix():
    # The keys are the words of three Philox blocks in order; the C form agrees.
    ks = PX.round_keys(7, 3, 2)
    assert ks == numpy_philox_block((0, 2, 0, 0), (7, 3)) + numpy_philox_block((1, 2, 0, 0), (7, 3)) + \
        numpy_philox_block((2, 2, 0, 0), (7, 3))
    assert CS.round_keys(7, 3, 2) == ks
    # mix64 is the SplitMix64 output function, restated here on Python integers.
    M = (1 << 64) - 1
    for z in (0, 1, 2**63, 0x0123456789ABCDEF, M):
        y = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        y = ((y ^ (y >> 27)) * 0x94D049BB133111EB) & M
        assert int(PX.mix64(np.uint64(z))) == y ^ (y >> 31)


@pytest.mark.parametrize("bits", range(2, 15))
def test_feistel_is_a_bijection(bits):
    x = np.arange(1 << bits, dtype=np.uint64)
    for seed, row, attempt in ((1, 0, 0), (2**63 + 9, 5, 3)):
        keys = PX.round_keys(seed, row, attempt)
        y = PX.feistel(x, bits, keys)
        assert np.array_equal(np.sort(y), x)
        assert not np.array_equal(y, x)
        for v in (0, 1, (1 << bits) - 1):
            assert CS.feistel(v, bits, keys) == int(y[v])


@pytest.mark.parametrize("n", list(range(1, 70)) + [100, 255, 256, 257, 1000, 4097, 65537])
def test_permutation_of_every_small_domain(n):
    for seed in (3, 77):
        pi = PX.permute(np.arange(n, dtype=np.uint64), n, seed, 1, 2)
        assert np.array_equal(np.sort(pi), np.arange(n))


@pytest.mark.parametrize("n,S,seed,row,attempt", [(1, 1, 1, 0, 0), (5, 5, 9, 0, 0), (1000, 50, 1, 0, 0),
                                                  (37, 20, 5, 3, 2), (2**20, 3000, 77, 1, 0),
                                                  ((1 << 22) + 3, 2000, 2**64 - 1, 7, 5), (50331648, 1000, 4, 0, 1),
                                                  (2**30, 1500, 11, 0, 0), (3_000_000_000, 700, 12, 2, 3),
                                                  ((1 << 40) - 17, 300, 13, 0, 0)])
def test_c_sampler_matches_numpy_definition(n, S, seed, row, attempt):
    ref = PX.sample_indices_numpy(n, S, seed, row, attempt)
    assert np.array_equal(CS.sample_indices(n, S, seed, row, attempt), ref)
    assert np.array_equal(PX.sample_indices(n, S, seed, row, attempt), ref)
    assert np.unique(ref).size == S and ref.min() >= 0 and ref.max() < n
    for j in (0, S // 2, S - 1):
        assert CS.permute(j, n, seed, row, attempt) == ref[j]


def test_sample_many_matches_single():
    a = CS.sample_many(12345, 500, [3, 9, 2**40], 2, 1)
    for j, sd in enumerate([3, 9, 2**40]):
        assert np.array_equal(a[j], CS.sample_indices(12345, 500, sd, 2, 1))


@pytest.mark.parametrize("n,S", [(8, 3), (6, 2), (5, 5)])
def test_sample_is_a_uniform_subset(n, S):
    # Every S-subset equally likely over the seeds (chi-square), and the
    # sample's order a uniform order of the subset for S = 2.
    seeds = 20_000
    subsets = {c: i for i, c in enumerate(itertools.combinations(range(n), S))}
    u = CS.sample_many(n, S, np.arange(seeds))
    counts = np.zeros(len(subsets), dtype=np.int64)
    for r in range(seeds):
        counts[subsets[tuple(sorted(u[r]))]] += 1
    assert math.comb(n, S) == len(subsets)
    if len(subsets) > 1:
        assert stats.chisquare(counts).pvalue > 1e-4
    if S == 2:
        ordered = np.zeros((n, n), dtype=np.int64)
        np.add.at(ordered, (u[:, 0], u[:, 1]), 1)
        off = ordered[~np.eye(n, dtype=bool)]
        assert stats.chisquare(off).pvalue > 1e-4


def test_every_position_is_uniform():
    # Each sample position j takes every index of [0, n) equally often over
    # the seeds, for an n off the power-of-two grid (cycle-walking at work).
    n, S, seeds = 23, 4, 23_000
    u = CS.sample_many(n, S, np.arange(seeds), 3, 0)
    for j in range(S):
        assert stats.chisquare(np.bincount(u[:, j], minlength=n)).pvalue > 1e-4


def test_attempts_and_rows_give_independent_samples():
    # Overlaps of two samples of S from n behave like independent uniform
    # subsets: hypergeometric with mean S^2 / n.
    n, S = 1 << 16, 4096
    base = CS.sample_indices(n, S, 5, 0, 0)
    for other in (CS.sample_indices(n, S, 5, 0, 1), CS.sample_indices(n, S, 5, 1, 0), CS.sample_indices(n, S, 6, 0, 0)):
        overlap = np.intersect1d(base, other).size
        mean, sd = S * S / n, math.sqrt(S * (S / n) * (1 - S / n) * (n - S) / (n - 1))
        assert abs(overlap - mean) < 5 * sd, overlap
