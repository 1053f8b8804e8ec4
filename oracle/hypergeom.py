"""Hypergeometric law of the sampled counts, in fp64.

Prof-K paper, Section 4, Eq 1-2: X ~ Hypergeometric(N, K, S) counts the
distinguished items among S drawn without replacement from N of which K are
distinguished; F_{N,K,S}(j) = Pr(X <= j) and F^{-1}(p) = min{j : F(j) >= p}.
Lemma 1 identifies X_K = |sample ∩ top-K| with this law.

The pmf is evaluated in log space.  The first term uses
  log Pr(X = 0) = sum_{i<S} log1p(-K / (N - i))      (when S <= N - K),
which keeps full relative precision for N up to 2^32; later terms follow the
ratio Pr(X=j+1)/Pr(X=j) = (K-j)(S-j) / ((j+1)(N-K-S+j+1)).  When S > N - K
the support starts at S-(N-K) and that first term comes from lgamma.
"""
from __future__ import annotations

import math

import numpy as np


def _support(N: int, K: int, S: int):
    return max(0, S - (N - K)), min(K, S)


def _log_pmf_first(N: int, K: int, S: int) -> float:
    lo, _ = _support(N, K, S)
    if lo == 0:
        if K == 0:
            return 0.0
        i = np.arange(S, dtype=np.float64)
        return float(np.sum(np.log1p(-K / (N - i))))
    lc = lambda a, b: math.lgamma(a + 1) - math.lgamma(b + 1) - math.lgamma(a - b + 1)
    return lc(K, lo) + lc(N - K, S - lo) - lc(N, S)


def pmf_upto(N: int, K: int, S: int, j: int) -> np.ndarray:
    """Pr(X = i) for i = 0 .. j (zeros outside the support)."""
    if not (0 <= K <= N and 0 <= S <= N):
        raise ValueError("need 0 <= K, S <= N")
    out = np.zeros(max(j + 1, 0), dtype=np.float64)
    lo, hi = _support(N, K, S)
    if j < lo:
        return out
    lp = _log_pmf_first(N, K, S)
    for i in range(lo, min(j, hi) + 1):
        out[i] = math.exp(lp)
        if i < hi:
            lp += math.log((K - i) * (S - i)) - math.log((i + 1) * (N - K - S + i + 1))
    return out


def cdf(N: int, K: int, S: int, j: int) -> float:
    """F_{N,K,S}(j) = Pr(X <= j)."""
    if j < 0:
        return 0.0
    lo, hi = _support(N, K, S)
    if j >= hi:
        return 1.0
    return float(min(1.0, math.fsum(pmf_upto(N, K, S, j))))


def sf(N: int, K: int, S: int, j: int) -> float:
    """Pr(X > j) = 1 - F(j), summed over the upper terms when that is shorter."""
    lo, hi = _support(N, K, S)
    if j < lo:
        return 1.0
    if j >= hi:
        return 0.0
    return float(max(0.0, 1.0 - math.fsum(pmf_upto(N, K, S, j))))


def quantile(N: int, K: int, S: int, p: float) -> int:
    """F^{-1}_{N,K,S}(p) = min{j in 0..S : F(j) >= p}, p in (0, 1]."""
    if not (0.0 < p <= 1.0):
        raise ValueError("p must be in (0, 1]")
    lo, hi = _support(N, K, S)
    lp = _log_pmf_first(N, K, S)
    acc = []
    for j in range(lo, hi + 1):
        acc.append(math.exp(lp))
        if math.fsum(acc) >= p:
            return j
        if j < hi:
            lp += math.log((K - j) * (S - j)) - math.log((j + 1) * (N - K - S + j + 1))
    return hi
