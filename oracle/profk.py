"""The Prof-K procedure itself, step by step, on the CPU.

Follows the paper's four stages (Section 3 "The Prof-K Algorithm") and its
run-time check (Section 4 "Failure Modes"; Appendix C "The Filter Kernel"):

  1. sample S indices without replacement            (oracle.philox)
  2. tau = t-th largest sampled value
  3. filter: R = |{i : x_i >= tau}|, append those (x_i, i) to a buffer of
     capacity M; the count is exact even when the buffer overflows
  4. refine: exact top-k of the buffer when k <= R <= M; otherwise redraw with
     a fresh sample, and after six failed attempts fall back to an exact top-k
     of the whole input (Section 3, stage 4: "say, six").

One addition that keeps the output exact (a reading, not in the pages): the
filter also counts R_gt = |{i : x_i > tau}|.  If R > M and R_gt < k, then tau
is exactly the k-th largest value (R_gt < k <= R), every threshold that keeps
recall yields R' >= R > M, so every redraw must overflow too; the call then
emits all x_i > tau plus the lowest-index copies of tau ("tie path") at once.
It can be switched off (``tie_exit=False``) to follow the pages literally.

Everything is per row; batched inputs run the procedure row by row with
eps / rows per row (union bound, corrected paper Appendix E.2).

Which calls run the method at all is not the oracle's decision: the caller
passes ``route``.  ROUTE_FILTER runs the four stages above; ROUTE_EXACT
returns the exact top-k without sampling (the result is the same either way;
only the statistics differ).  The rule a library uses to pick the route is an
implementation choice and lives with that library's tests.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import params as P
from . import philox
from .topk import topk_sort

PATH_FILTER = 0
PATH_TIE = 1
PATH_FALLBACK = 2
PATH_EXACT = 3

ROUTE_FILTER = "filter"
ROUTE_EXACT = "exact"


@dataclass
class Stats:
    S: int = 0
    t: int = 0
    M: int = 0
    attempts: int = 0
    path: int = PATH_FILTER
    R_first: int = -1
    R_gt_first: int = -1
    R_final: int = -1
    R_gt_final: int = -1
    taus: list = field(default_factory=list)


def threshold(sampled_values: np.ndarray, t: int) -> np.float32:
    """Stage 2: the t-th largest sampled value (descending sort, 1-based t)."""
    s = np.sort(np.asarray(sampled_values, dtype=np.float32))[::-1]
    return np.float32(s[t - 1])


def filter_counts(x: np.ndarray, tau) -> tuple[int, int]:
    """Stage 3 counts: R = #{x >= tau} and R_gt = #{x > tau} (IEEE compares)."""
    tau = np.float32(tau)
    return int(np.count_nonzero(x >= tau)), int(np.count_nonzero(x > tau))


def filter_pass(x: np.ndarray, tau, M: int):
    """Stage 3: the passers (values, indices in index order) and the counts.

    The pages' buffer receives passers in arrival order and keeps the first M;
    which M survive an overflow is unspecified, so only R and R_gt are defined
    then and the returned passers are None.
    """
    tau = np.float32(tau)
    idx = np.flatnonzero(x >= tau).astype(np.int64)
    R = int(idx.size)
    R_gt = int(np.count_nonzero(x > tau))
    if R > M:
        return None, None, R, R_gt
    return x[idx].copy(), idx, R, R_gt


def refine(buf_vals: np.ndarray, buf_idx: np.ndarray, k: int):
    """Stage 4: exact top-k of the candidate buffer, same order as topk_sort."""
    order = np.lexsort((buf_idx, -np.asarray(buf_vals, dtype=np.float64)))[:k]
    return np.asarray(buf_vals, dtype=np.float32)[order].copy(), np.asarray(buf_idx, dtype=np.int64)[order]


def tie_path(x: np.ndarray, tau, k: int):
    """Exact top-k once tau is known to be the k-th largest value."""
    tau = np.float32(tau)
    gt = np.flatnonzero(x > tau)
    eq = np.flatnonzero(x == tau)[: k - gt.size]
    sel = np.concatenate([gt, eq]).astype(np.int64)
    return refine(x[sel], sel, k)


def profk(x: np.ndarray, k: int, eps: float, seed: int, row: int = 0, *, route: str = ROUTE_FILTER,
          max_attempts: int = 6, mode: int = P.MODE_DEFAULT, tie_exit: bool = True, force=None):
    """One row of Prof-K.  ``route`` (ROUTE_FILTER or ROUTE_EXACT) says whether
    the method runs or the exact selection does (see the module docstring).
    ``force`` may override (S, t, M) as a dict; a forced S recomputes t and M
    from it (the corrected Algorithm 1, t and M steps) unless those are forced
    as well."""
    if route not in (ROUTE_FILTER, ROUTE_EXACT):
        raise ValueError(f"route must be {ROUTE_FILTER!r} or {ROUTE_EXACT!r}")
    x = np.asarray(x, dtype=np.float32)
    if np.isnan(x).any():
        raise ValueError("NaN in input")
    N = x.shape[0]
    st = Stats()
    S, t, M = P.params(N, k, eps, mode)
    if force:
        if "S" in force:  # a forced S gets the fast t and M of that S unless they are forced too
            S = force["S"]
            t, M = P.params_fast(N, k, S, eps)
        t, M = force.get("t", t), force.get("M", M)
    st.S, st.t, st.M = S, t, M
    if route == ROUTE_EXACT:
        st.path = PATH_EXACT
        v, i = topk_sort(x, k)
        return v, i, st
    for a in range(max_attempts):
        sidx = philox.sample_indices(N, S, seed, row, a)
        tau = threshold(x[sidx], t)
        st.taus.append(float(tau))
        vals, idx, R, R_gt = filter_pass(x, tau, M)
        st.attempts = a + 1
        if a == 0:
            st.R_first, st.R_gt_first = R, R_gt
        st.R_final, st.R_gt_final = R, R_gt
        if k <= R <= M:
            st.path = PATH_FILTER
            v, i = refine(vals, idx, k)
            return v, i, st
        if tie_exit and R > M and R_gt < k:
            st.path = PATH_TIE
            v, i = tie_path(x, tau, k)
            return v, i, st
    st.path = PATH_FALLBACK
    v, i = topk_sort(x, k)
    return v, i, st


def first_attempt_ranks(xs, N: int, S: int, t: int, seeds, row: int = 0):
    """R and R_gt of the first attempt for many seeds (Monte-Carlo helper).

    ``xs`` is a list of inputs of length N sharing the same samples: the sample
    depends only on (N, S, seed), so one draw serves every input.  Returns
    int64 arrays of shape (len(xs), len(seeds)) for R and R_gt.
    """
    from . import csample

    seeds = list(seeds)
    R = np.zeros((len(xs), len(seeds)), dtype=np.int64)
    Rg = np.zeros_like(R)
    chunk = 64
    for c0 in range(0, len(seeds), chunk):
        cs = seeds[c0:c0 + chunk]
        sidx = csample.sample_many(N, S, cs, row, 0)
        for j in range(len(cs)):
            for q, x in enumerate(xs):
                tau = threshold(x[sidx[j]], t)
                R[q, c0 + j], Rg[q, c0 + j] = filter_counts(x, tau)
    return R, Rg
