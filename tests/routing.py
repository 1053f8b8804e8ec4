"""The library's routing rule, as the tests predict it, and the oracle call that uses it.

Which calls skip sampling is a choice of the library, not of the pages: the
oracle takes the route as an argument, and this helper supplies the route the
library is expected to take.  The GPU tests check it against the path the
library reports (``stats.path``), and ``tests/test_routing.py`` checks its
cases on the CPU.

The rule (the library's reading of the corrected paper, Appendix B, which keeps
the method at the floor sample size for dense k):

* the exact path when the sample would exceed n/8 (a sample that large is
  itself a pass over the row);
* the exact path when the parameter rules were clamped (t = S or M = n, which
  happens as k approaches n), because the budget cannot be met there;
* in calls of 128 rows or more with k <= 2048, the exact path also when the
  sample is n/32 or more (drawing 1/32 of every row by random access costs more
  than selecting each short row exactly in one CTA; measured on a GB300);
* the sample-and-filter path otherwise.
"""
from oracle import params as P
from oracle import profk as PK


def uses_filter(N: int, k: int, S: int, t: int, M: int, rows: int = 1) -> bool:
    if 8 * S > N or t >= S or M >= N:
        return False
    return not (rows >= 128 and 32 * S >= N and k <= 2048)


def route(N: int, k: int, eps_row: float, rows: int = 1, mode: int = P.MODE_DEFAULT, force=None) -> str:
    """The library's route for one row of a call of ``rows`` rows; forced
    parameters always run the method."""
    if force:
        return PK.ROUTE_FILTER
    S, t, M = P.params(N, k, eps_row, mode)
    return PK.ROUTE_FILTER if uses_filter(N, k, S, t, M, rows) else PK.ROUTE_EXACT


def oracle_profk(x, k, eps, seed, row=0, rows=1, *, mode=P.MODE_DEFAULT, force=None, **kw):
    """oracle.profk.profk on one row, on the route the library takes for it.
    ``eps`` is the row's own budget (the call's eps / rows)."""
    r = route(len(x), k, eps, rows, mode, force)
    return PK.profk(x, k, eps, seed, row, route=r, mode=mode, force=force, **kw)
