"""Pins of the oracle's Prof-K procedure to the analysis of the pages.

* Exact enumeration over every S-subset of a tiny [N]: the law of R (the older
  page's negative-hypergeometric Lemma 1, Eq 1-2; the corrected page's Lemma 6
  mean) and Propositions 2-3 (exact failure probabilities).
* Monte Carlo with the oracle's own sampler, 10^4 seeds: mean and variance of
  the first-attempt R within 3 standard errors of Lemma 1; the first-attempt
  failure count within the binomial 99% bound at eps and consistent with the
  exact Pr(A) + Pr(B).
* Every control path of the procedure returns the exact top-k.
"""
import itertools
import math
import multiprocessing as mp
from concurrent.futures import ProcessPoolExecutor
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

import workloads
from oracle import params as P
from oracle import profk as PK
from oracle.topk import same_result, topk_sort


def enumerate_R(N, S, t):
    """Distribution of R = rank of the t-th largest sampled element, distinct values."""
    dist = {}
    for sub in itertools.combinations(range(1, N + 1), S):  # ranks, 1 = largest
        R = sorted(sub)[t - 1]
        dist[R] = dist.get(R, 0) + 1
    tot = sum(dist.values())
    return {r: Fraction(c, tot) for r, c in dist.items()}


@pytest.mark.parametrize("N,S,t", [(12, 4, 2), (11, 5, 1), (10, 3, 3), (9, 6, 4)])
def test_rank_law_matches_enumeration(N, S, t):
    d = enumerate_R(N, S, t)
    mean = sum(r * p for r, p in d.items())
    var = sum(r * r * p for r, p in d.items()) - mean * mean
    m_form, v_form = P.lemma1_nhg_moments(N, S, t)
    assert float(mean) == pytest.approx(m_form, rel=1e-12)
    assert float(mean) == pytest.approx(P.mean_rank(N, S, t), rel=1e-12)
    assert float(var) == pytest.approx(v_form, rel=1e-12)
    for r, p in d.items():  # older page, Eq 1
        pmf = Fraction(math.comb(r - 1, t - 1) * math.comb(N - r, S - t), math.comb(N, S))
        assert p == pmf


@pytest.mark.parametrize("N,S,t,k,M", [(12, 4, 2, 3, 6), (11, 5, 1, 2, 4), (10, 3, 3, 4, 9), (12, 6, 2, 1, 2)])
def test_propositions_2_3_match_enumeration(N, S, t, k, M):
    d = enumerate_R(N, S, t)
    p_a = float(sum(p for r, p in d.items() if r < k))
    p_b = float(sum(p for r, p in d.items() if r > M))
    assert P.prob_recall_failure(N, k, S, t) == pytest.approx(p_a, abs=1e-14)
    assert P.prob_overflow(N, S, t, M) == pytest.approx(p_b, abs=1e-14)


def _inputs_small(seed):
    rng = np.random.default_rng(seed)
    n = 4096
    kinds = [rng.standard_normal(n).astype(np.float32),
             np.repeat(np.float32([5.0, 4.0, 3.0]), [3, 900, n - 903]),
             rng.integers(0, 4, n).astype(np.float32),
             np.sort(rng.standard_normal(n).astype(np.float32))]
    return kinds


@pytest.mark.parametrize("seed", range(3))
def test_every_path_is_exact(seed):
    for x in _inputs_small(seed):
        for k in (1, 7, 50):
            ref = topk_sort(x, k)
            for force in ({"S": 256, "t": 3, "M": 400}, {"S": 256, "t": 256, "M": 60},
                          {"S": 256, "t": 1, "M": 50}, {"S": 64, "t": 2}):
                for tie_exit in (True, False):
                    for attempts in (0, 1, 6):
                        v, i, st = PK.profk(x, k, 1e-3, seed * 7 + 1, force=force, tie_exit=tie_exit,
                                            max_attempts=attempts)
                        assert same_result(v, i, *ref), (k, force, tie_exit, attempts, st)
                        if attempts == 0:
                            assert st.path == PK.PATH_FALLBACK


def test_paths_are_reached():
    x = np.repeat(np.float32([5.0, 4.0]), [3, 4093])
    v, i, st = PK.profk(x, 10, 1e-3, 1, force={"S": 256, "t": 5, "M": 100})
    assert st.path == PK.PATH_TIE and same_result(v, i, *topk_sort(x, 10))
    v, i, st = PK.profk(x, 10, 1e-3, 1, force={"S": 256, "t": 5, "M": 100}, tie_exit=False)
    assert st.path == PK.PATH_FALLBACK and st.attempts == 6
    y = np.random.default_rng(2).standard_normal(1 << 16).astype(np.float32)
    v, i, st = PK.profk(y, 64, 1e-3, 3, route=PK.ROUTE_EXACT)
    assert st.path == PK.PATH_EXACT and st.attempts == 0 and same_result(v, i, *topk_sort(y, 64))
    v, i, st = PK.profk(y, 64, 1e-3, 3)  # the method itself, even with S = n / 2
    assert st.path == PK.PATH_FILTER and same_result(v, i, *topk_sort(y, 64))
    v, i, st = PK.profk(y, 16, 1e-3, 3, force={"S": 2048, "t": 4, "M": 500})
    assert st.path == PK.PATH_FILTER and k_le(16, st.R_first, 500)


def k_le(k, R, M):
    return k <= R <= M


# ---------------------------------------------------------------------------
# Monte Carlo on the oracle (N = 2^20, k = 64: S = 32768, t = 9, M = 714).

N_MC, K_MC, SEEDS = 1 << 20, 64, 10_000


def _mc_chunk(args):
    xs, seeds, S, t = args
    return PK.first_attempt_ranks(xs, N_MC, S, t, seeds)


@pytest.fixture(scope="module")
def mc_ranks():
    S, t, M = P.params(N_MC, K_MC, 1e-3)
    distinct = workloads.distinct_shuffled(N_MC, 21, "cpu").numpy()
    normal = workloads.normal(N_MC, 22, "cpu").numpy()
    seeds = list(range(1000, 1000 + SEEDS))
    chunks = [seeds[i:i + 500] for i in range(0, SEEDS, 500)]
    ctx = mp.get_context("spawn")
    with ProcessPoolExecutor(max_workers=min(8, mp.cpu_count()), mp_context=ctx) as ex:
        parts = list(ex.map(_mc_chunk, [([distinct, normal], c, S, t) for c in chunks]))
    R = np.concatenate([p[0] for p in parts], axis=1)
    return dict(S=S, t=t, M=M, R_distinct=R[0], R_normal=R[1])


def test_lemma1_moments_monte_carlo(mc_ranks):
    R = mc_ranks["R_distinct"].astype(np.float64)
    S, t = mc_ranks["S"], mc_ranks["t"]
    mean, var = P.lemma1_nhg_moments(N_MC, S, t)
    n = R.size
    se_mean = math.sqrt(var / n)
    assert abs(R.mean() - mean) <= 3 * se_mean, (R.mean(), mean, se_mean)
    s2 = R.var(ddof=1)
    m4 = np.mean((R - R.mean()) ** 4)
    se_var = math.sqrt(max(m4 - s2 * s2, 0.0) / n)
    assert abs(s2 - var) <= 3 * se_var, (s2, var, se_var)


def test_retry_rate_monte_carlo(mc_ranks):
    R = mc_ranks["R_normal"]
    S, t, M = mc_ranks["S"], mc_ranks["t"], mc_ranks["M"]
    fails = int(np.count_nonzero((R < K_MC) | (R > M)))
    assert fails <= stats.binom.ppf(0.99, SEEDS, 1e-3)  # 18 at eps = 1e-3
    p_exact = P.prob_fail(N_MC, K_MC, S, t, M)
    assert fails <= stats.binom.ppf(0.999, SEEDS, p_exact)
