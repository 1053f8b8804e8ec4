"""The library's routing rule as the tests predict it (tests/routing.py), on the CPU.

The GPU tests compare this prediction with the path the library reports; here
its cases are checked against the rule's own statement, and every problem the
rule sends down the filter path is checked to meet the failure budget with
the exact Propositions 2-3 of the corrected paper.
"""
import numpy as np

from oracle import params as P
from oracle import profk as PK
from oracle.topk import same_result, topk_sort
from routing import oracle_profk, route, uses_filter


def filt(N, k, rows=1, eps=1e-3):
    return route(N, k, eps / rows, rows) == PK.ROUTE_FILTER


def test_default_rule_invariants_and_budget():
    for N in (2**20, 2**22, 2**26, 2**30, 50331648, 2**32):
        for k in (1, 2, 32, 1024, 4096, 2**19, N // 64, N // 16, N // 4):
            if k > N:
                continue
            S, t, M = P.params(N, k, 1e-3)
            assert 32768 <= S <= 131072 and 1 <= t <= S and k <= M <= N
            if uses_filter(N, k, S, t, M) and N <= 2**26:
                # every configuration the filter path takes meets the budget
                # (exact Propositions 2-3; kept to N <= 2^26 for the CPU's time)
                assert P.prob_fail(N, k, S, t, M) <= 1e-3


def test_route_cases():
    # A sample of more than 1/8 of the row takes the exact path.
    assert filt(2**20, 64) and filt(2**18, 64)
    assert not filt(2**18 - 4, 64)
    # Dense k stays on the filter path (no cut on k / N) ...
    assert filt(2**20, 2**14 + 1) and filt(2**24, 2**21) and filt(2**26, 2**24)
    # ... until the rules clamp t to S or M to N, as k approaches N.
    assert not filt(2**20, 2**20 - 5) and not filt(2**20, 2**20)
    S, t, M = P.params(2**20, 2**20 - 5, 1e-3)
    assert t == S or M == 2**20
    # Calls of 128 or more rows with k <= 2048: only samples below 1/32 of a row.
    assert filt(2**20, 64, rows=127) and not filt(2**20, 64, rows=128)
    assert filt(2**20 + 4, 2048, rows=1024) and not filt(2**20, 2048, rows=1024)
    assert filt(2**20, 2049, rows=1024)
    assert filt(2**24, 32, rows=64) and filt(2**24, 32, rows=4096)
    # Forced parameters always run the method.
    assert route(1000, 10, 1e-3, force={"S": 64}) == PK.ROUTE_FILTER


def test_oracle_call_follows_the_route():
    rng = np.random.default_rng(5)
    small = rng.standard_normal(1 << 16).astype(np.float32)  # S = 32768 > n / 8: exact
    v, i, st = oracle_profk(small, 64, 1e-3, 3)
    assert st.path == PK.PATH_EXACT and same_result(v, i, *topk_sort(small, 64))
    big = rng.standard_normal(1 << 20).astype(np.float32)
    v, i, st = oracle_profk(big, 64, 1e-3, 3)
    assert st.path == PK.PATH_FILTER and st.attempts == 1 and same_result(v, i, *topk_sort(big, 64))
