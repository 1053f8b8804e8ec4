"""Monte-Carlo checks of the GPU sampler and filter against the analysis.

10^4 seeds at N = 2^20, k = 64 (S = 32768, t = 9, M = 714):
* on a permutation of 0..N-1 (distinct values) the first-attempt count R has
  the older page's Lemma 1 mean and variance (within 3 standard errors);
* on standard-normal input the first-attempt failures stay within the binomial
  99% bound at eps (18 of 10^4) and agree with the exact Pr(A) + Pr(B) of
  Propositions 2-3.
Each call also returns the exact top-k (checked for a subset of seeds)."""
import math

import numpy as np
import pytest
from scipy import stats

import workloads
from gpu_helpers import assert_same
from oracle import params as P
from oracle.topk import topk_sort

pytestmark = pytest.mark.gpu

N, K, SEEDS = 1 << 20, 64, 10_000


def first_counts(pk, x, seeds):
    R = np.empty(len(seeds), dtype=np.int64)
    att = np.empty(len(seeds), dtype=np.int64)
    ref = topk_sort(x.cpu().numpy(), K)
    for j, s in enumerate(seeds):
        vals, idx, st = pk.topk(x, K, 1e-3, s)
        R[j] = st["R_first"]
        att[j] = st["attempts"]
        if j % 997 == 0:
            assert_same(vals, idx, *ref, f"seed {s}")
    return R, att


def test_lemma1_moments_gpu(pk, cuda_device):
    x = workloads.distinct_shuffled(N, 31, cuda_device)
    S, t, M = P.params(N, K, 1e-3)
    R, _ = first_counts(pk, x, range(5000, 5000 + SEEDS))
    mean, var = P.lemma1_nhg_moments(N, S, t)
    Rf = R.astype(np.float64)
    assert abs(Rf.mean() - mean) <= 3 * math.sqrt(var / SEEDS)
    s2 = Rf.var(ddof=1)
    m4 = np.mean((Rf - Rf.mean()) ** 4)
    assert abs(s2 - var) <= 3 * math.sqrt(max(m4 - s2 * s2, 0.0) / SEEDS)


def test_retry_rate_gpu(pk, cuda_device):
    x = workloads.normal(N, 32, cuda_device)
    S, t, M = P.params(N, K, 1e-3)
    R, att = first_counts(pk, x, range(20000, 20000 + SEEDS))
    fails = int(np.count_nonzero((R < K) | (R > M)))
    assert fails == int(np.count_nonzero(att > 1))
    assert fails <= stats.binom.ppf(0.99, SEEDS, 1e-3)
    assert fails <= stats.binom.ppf(0.999, SEEDS, P.prob_fail(N, K, S, t, M))
