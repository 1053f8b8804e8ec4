"""Parameter rules (S, t, M) of Prof-K, in fp64.

Two versions of the paper disagree here; both are written out so that tests can
hold each to its own page.

Corrected version ("Prof-K: Probabilistic One-Pass Filtering for Efficient
Top-k Selection", arXiv HTML):
  * Theorem 4 (exact optimal parameters): t* = F^{-1}_{N,k-1,S}(1-eps_A) + 1,
    M* = min{M >= k : F_{N,M,S}(t*-1) <= eps_B};  Propositions 2-3 give the
    exact failure probabilities.
  * Algorithm 1 (fast approximate parameters), Appendix B Eq 9-12: Acklam's
    inverse normal, the Cornish-Fisher threshold rank (mu >= 15), the Poisson
    quantile (mu < 15) and the Wilson-Hilferty buffer capacity.
  * Proposition 7: S1 = (z/r)^(2/3) (kN)^(1/3), S2 = (kappa N / r)^(1/2).

Older version (same title, mirrored page):
  * Lemma 2 normal approximation, Eq 6 threshold rank, Corollary 4 buffer
    size M = k + z sqrt(k(N-k)/S (1-S/N)) with z = z_A + z_B, Theorem 5
    S* = (z tau_B log k / (2 tau_A))^(2/3) (k(N-k))^(1/3), and its Algorithm 1
    (S clamped to [32768, 131072], "t <- 1 if alpha S < -ln(eps/2)").

Default rule used by the library (a reading, because the two versions conflict):
S from the older version's Theorem 5 with its clamp, rounding and log2 (its
Algorithm 1, its sample-size step), and t, M from the corrected Algorithm 1 (its t and M steps)
with z = Phi^{-1}(1 - eps/2), then 1 <= t <= S and k <= M <= N.  The older
t-rule sets t = 1 exactly where recall failure is likely (its own text derives
the bound in the wrong direction), so it is kept only as a named function and
an optional mode.  A third mode keeps that S and takes the exact optimal t and
M of the corrected Theorem 4 (``params_exact``, pinned to Table 3).  A fourth
follows the corrected Algorithm 1 throughout, its sample size included
(Proposition 7 with a cost ratio r(k) calibrated on a GB300; the paper's own
RTX 3060 calibration reproduces Table 3's S column).

What pins each function (tests/test_oracle_params.py unless named):
  norm_ppf                    scipy's ndtri within Acklam's stated 1.15e-9
  prob_recall_failure,
  prob_overflow, prob_fail    enumeration of every S-subset of a tiny [N]
                              (tests/test_oracle_theory.py); Table 3's failure
                              probabilities
  params_exact                Table 3's t* and M* columns (21 rows)
  threshold_rank_fast,
  params_fast                 Table 3's t and M columns; k = 1 gives t = 1
  buffer_capacity_fast        Table 3's M column; scipy's exact Gamma quantile
                              (3 % high at t = 1, Appendix B, closing with t)
  sample_size_prop7           Proposition 7's bracket around the numerical
                              minimiser of the Eq 13 cost
  sample_size_corrected,
  inv_r_rtx3060               Table 3's S column with the paper's r(k)
  params_corrected            its two steps
  inv_r_gb300                 a measured calibration (its fit is tested in
                              tests/test_calibrate_fit.py); parity unpinned
                              by the pages, which fix only the form
  lemma1_nhg_moments,
  mean_rank                   enumeration (Eq 1-2; Lemma 6)
  lemma2_normal               converges to Lemma 1's moments like 1/S at
                              fixed S/N (Eq 3-4 as a limit)
  t_eq6                       the smallest t meeting Eq 5's normal tail bound
  m_cor4                      Eq 8 and Eq 11 (M = c k) algebra
  s_thm5                      the numerical minimiser of Eq 13 with
                              Corollary 4's M at f = 1 (Theorem 5)
  s_star_scaling              the page's "S* ~ 4,600 at N = 1e9, k = 100"
  sample_size_old             that minimiser rounded and clamped to
                              [32768, 131072] (older Algorithm 1)
  params_old                  Eq 6 / Eq 8 / Eq 11 at a point above the t = 1
                              cut, and both sides of the cut at -ln(eps/2)
  params                      composition of the above (the library's modes
                              equal it: tests/test_abi.py)
"""
from __future__ import annotations

import math

from . import hypergeom

# ---------------------------------------------------------------------------
# Inverse standard normal: P. J. Acklam's rational approximation (relative
# error below 1.15e-9), as the corrected paper prescribes (Appendix B).
# Coefficients from Acklam's published algorithm.
_A = (-3.969683028665376e+01, 2.209460984245205e+02, -2.759285104469687e+02,
      1.383577518672690e+02, -3.066479806614716e+01, 2.506628277459239e+00)
_B = (-5.447609879822406e+01, 1.615858368580409e+02, -1.556989798598866e+02,
      6.680131188771972e+01, -1.328068155288572e+01)
_C = (-7.784894002430293e-03, -3.223964580411365e-01, -2.400758277161838e+00,
      -2.549732539343734e+00, 4.374664141464968e+00, 2.938163982698783e+00)
_D = (7.784695709041462e-03, 3.224671290700398e-01, 2.445134137142996e+00,
      3.754408661907416e+00)
_P_LOW = 0.02425


def norm_ppf(p: float) -> float:
    """Phi^{-1}(p) for p in (0, 1) by Acklam's three-region rational fit."""
    if not (0.0 < p < 1.0):
        raise ValueError("p must be in (0, 1)")
    if p < _P_LOW:
        q = math.sqrt(-2.0 * math.log(p))
        return ((((((_C[0] * q + _C[1]) * q + _C[2]) * q + _C[3]) * q + _C[4]) * q + _C[5])
                / ((((_D[0] * q + _D[1]) * q + _D[2]) * q + _D[3]) * q + 1.0))
    if p > 1.0 - _P_LOW:
        q = math.sqrt(-2.0 * math.log1p(-p))
        return -((((((_C[0] * q + _C[1]) * q + _C[2]) * q + _C[3]) * q + _C[4]) * q + _C[5])
                 / ((((_D[0] * q + _D[1]) * q + _D[2]) * q + _D[3]) * q + 1.0))
    q = p - 0.5
    r = q * q
    return ((((((_A[0] * r + _A[1]) * r + _A[2]) * r + _A[3]) * r + _A[4]) * r + _A[5]) * q
            / (((((_B[0] * r + _B[1]) * r + _B[2]) * r + _B[3]) * r + _B[4]) * r + 1.0))


# ---------------------------------------------------------------------------
# Corrected version: exact analysis.

def prob_recall_failure(N: int, k: int, S: int, t: int) -> float:
    """Proposition 2: Pr(R < k) = 1 - F_{N,k-1,S}(t-1)."""
    return hypergeom.sf(N, k - 1, S, t - 1)


def prob_overflow(N: int, S: int, t: int, M: int) -> float:
    """Proposition 3: Pr(R > M) = F_{N,M,S}(t-1)."""
    return hypergeom.cdf(N, M, S, t - 1)


def prob_fail(N: int, k: int, S: int, t: int, M: int) -> float:
    """Eq 8: Pr(A or B) = Pr(R < k) + Pr(R > M) (disjoint because M >= k)."""
    return prob_recall_failure(N, k, S, t) + prob_overflow(N, S, t, M)


def params_exact(N: int, k: int, S: int, eps: float, eps_a: float | None = None,
                 eps_b: float | None = None):
    """Theorem 4: exact optimal (t*, M*) for a given S; default split eps/2."""
    eps_a = eps / 2 if eps_a is None else eps_a
    eps_b = eps / 2 if eps_b is None else eps_b
    t = hypergeom.quantile(N, k - 1, S, 1.0 - eps_a) + 1
    lo, hi = k, N  # G(M) = F_{N,M,S}(t-1) is nonincreasing in M and G(N) = 0
    while lo < hi:
        mid = (lo + hi) // 2
        if hypergeom.cdf(N, mid, S, t - 1) <= eps_b:
            hi = mid
        else:
            lo = mid + 1
    return t, lo


def threshold_rank_fast(N: int, k: int, S: int, eps: float) -> int:
    """Corrected Algorithm 1, the t step: Eq 10 (Cornish-Fisher) or Eq 11 (Poisson)."""
    z = norm_ppf(1.0 - eps / 2)
    mu = (k - 1) * S / N
    if mu >= 15:
        sigma = math.sqrt(mu * (1.0 - (k - 1) / N) * (N - S) / (N - 1))
        return math.ceil(mu + z * sigma + (z * z - 1.0) / 6.0) + 1
    p = math.exp(-mu)
    c = p
    j = 0
    while c < 1.0 - eps / 2:
        j += 1
        p = p * mu / j
        c = c + p
    return j + 1


def buffer_capacity_fast(N: int, S: int, t: int, eps: float) -> int:
    """Corrected Algorithm 1, the M step: Eq 12, Wilson-Hilferty quantile of Gamma(t,1)."""
    z = norm_ppf(1.0 - eps / 2)
    h = 1.0 / (9.0 * t)
    return math.ceil((N + 1) / (S + 1) * t * (1.0 - h + z * math.sqrt(h)) ** 3)


def params_fast(N: int, k: int, S: int, eps: float):
    """Corrected Algorithm 1 (t and M steps) for a given S, then 1 <= t <= S and k <= M <= N."""
    t = min(max(threshold_rank_fast(N, k, S, eps), 1), S)
    M = min(max(buffer_capacity_fast(N, S, t, eps), k), N)
    return t, M


def mean_rank(N: int, S: int, t: int) -> float:
    """Lemma 6: E[R] = (N+1) t / (S+1)."""
    return (N + 1) * t / (S + 1)


def sample_size_prop7(N: int, k: int, eps: float, r: float):
    """Proposition 7 candidates (S1, S2) for cost ratio r; kappa = z^2 + 1/2.

    Pinned by Proposition 7's bracket (the cost's minimiser lies between
    max(S1, S2) and 2^(2/3) times it) and, through sample_size_corrected, by
    the corrected page's Table 3 S column: exact on the rows the floor, the cap
    or n/128 set, within 5 % on those S1 or S2 set (the printed two-digit
    coefficients of r(k) are rounded).
    """
    z = norm_ppf(1.0 - eps / 2)
    kappa = z * z + 0.5
    S1 = (z / r) ** (2.0 / 3.0) * (k * N) ** (1.0 / 3.0)
    S2 = math.sqrt(kappa * N / r)
    return S1, S2


# Bounds of the corrected rule: the fixed-cost floor S_min = 2^14 (Appendix E.1,
# "the fixed-cost floor"), S_max = 2^18 (Table 3 tops out there at N = 2^31).
S_MIN_CORRECTED = 1 << 14
S_MAX_CORRECTED = 1 << 18


def inv_r_rtx3060(k: int):
    """The paper's calibration of 1/r(k) on its RTX 3060 (Appendix E.1):
    0.59 log2 k - 4.3 for k > 2^7; None (r = infinity) below."""
    return 0.59 * math.log2(k) - 4.3 if k > (1 << 7) else None


# The same fit on a GB300 (this library's kernels, an S sweep over n = 2^22..2^30,
# k = 2^5..2^19): the buffer cost per element barely grows with k there, the
# refinement being latency-bound, so the line is nearly flat.
GB300_INV_R_SLOPE = 0.0033
GB300_INV_R_INTERCEPT = 0.41


def inv_r_gb300(k: int):
    """1/r(k) calibrated on a GB300 in the paper's form: a + b log2 k for k > 2^7."""
    return GB300_INV_R_SLOPE * math.log2(k) + GB300_INV_R_INTERCEPT if k > (1 << 7) else None


def sample_size_corrected(N: int, k: int, eps: float, inv_r=inv_r_gb300, s_min: int = S_MIN_CORRECTED,
                          s_max: int = S_MAX_CORRECTED) -> int:
    """Corrected Algorithm 1, its sample-size steps (lines 1-4) with Proposition 7:
    z = Phi^{-1}(1 - eps/2), kappa = z^2 + 1/2, S = clip(floor(max(S1, S2)), S_min, S_max),
    S_min when r = infinity or k/N > 2^-10; then at most N/128.

    The cap N/128 is a reading: Table 3 uses S = 8,192 = N/128 for every k at
    N = 2^20, below the floor, and no other row reaches N/128.
    """
    ir = inv_r(k)
    if ir is None or ir <= 0.0 or k > N / 1024.0:
        S = s_min
    else:
        S1, S2 = sample_size_prop7(N, k, eps, 1.0 / ir)
        S = min(max(math.floor(max(S1, S2)), s_min), s_max)
    return max(1, min(S, N // 128))


def params_corrected(N: int, k: int, eps: float, inv_r=inv_r_gb300):
    """Corrected Algorithm 1 in full: the sample-size steps, then its t and M steps."""
    S = sample_size_corrected(N, k, eps, inv_r)
    t, M = params_fast(N, k, S, eps)
    return S, t, M


# ---------------------------------------------------------------------------
# Older version: closed forms.

def lemma2_normal(N: int, S: int, t: int):
    """Lemma 2 (Eq 4): R ~ Normal(N q, N^2 q (1-q) f / S), q = t/S, f = 1 - S/N."""
    q = t / S
    f = 1.0 - S / N
    return N * q, N * N * q * (1.0 - q) * f / S


def lemma1_nhg_moments(N: int, S: int, t: int):
    """Older Lemma 1 (Eq 2): mean and variance of the negative hypergeometric R."""
    mean = (N + 1) * t / (S + 1)
    var = t * (S - t + 1) * (N + 1) * (N - S) / ((S + 1) ** 2 * (S + 2))
    return mean, var


def t_eq6(N: int, k: int, S: int, z_a: float) -> int:
    """Eq 6: t = ceil(S alpha + z_A sqrt(S alpha (1-alpha) f))."""
    alpha = k / N
    f = 1.0 - S / N
    return math.ceil(S * alpha + z_a * math.sqrt(S * alpha * (1.0 - alpha) * f))


def m_cor4(N: int, k: int, S: int, z: float) -> float:
    """Corollary 4 (Eq 12): M = k + z sqrt(k (N-k) / S * (1 - S/N)), z = z_A + z_B."""
    return k + z * math.sqrt(k * (N - k) / S * (1.0 - S / N))


def s_thm5(N: int, k: int, z: float, cost_ratio: float = 1.0, log=math.log2) -> float:
    """Theorem 5 (Eq 14): S* = (z (tau_B/tau_A) log k / 2)^(2/3) (k (N-k))^(1/3)."""
    return (z * cost_ratio * log(k) / 2.0) ** (2.0 / 3.0) * (k * (N - k)) ** (1.0 / 3.0)


def s_star_scaling(N: int, k: int) -> float:
    """Theorem 5's k << N scaling S* ~ (k (N-k))^(1/3) with unit prefactor."""
    return (k * (N - k)) ** (1.0 / 3.0)


S_MIN_OLD = 32768
S_MAX_OLD = 131072


def sample_size_old(N: int, k: int, eps: float, s_min: int = S_MIN_OLD,
                    s_max: int = S_MAX_OLD, cost_ratio: float = 1.0) -> int:
    """Older Algorithm 1, the sample-size step: z = 2 Phi^{-1}(1-eps/2), S* with log2, round, clamp."""
    z = 2.0 * norm_ppf(1.0 - eps / 2)
    s = s_thm5(N, k, z, cost_ratio) if k > 1 else 0.0
    return int(min(s_max, max(s_min, math.floor(s + 0.5))))


def params_old(N: int, k: int, eps: float, s_min: int = S_MIN_OLD, s_max: int = S_MAX_OLD,
               cost_ratio: float = 1.0):
    """Older Algorithm 1, literally (all of its steps), through the named
    closed forms: z = z_A + z_B with z_A = z_B = Phi^{-1}(1 - eps/2); S from
    Theorem 5 (sample_size_old); t = max(1, Eq 6 with z_A); M = the ceiling of
    Corollary 4 with z; and t = 1 when alpha S < -ln(eps/2)."""
    z_half = norm_ppf(1.0 - eps / 2)
    z = 2.0 * z_half
    S = sample_size_old(N, k, eps, s_min, s_max, cost_ratio)
    t = max(1, t_eq6(N, k, S, z_half))
    M = math.ceil(m_cor4(N, k, S, z))
    if (k / N) * S < -math.log(eps / 2):
        t = 1
    return S, t, M


# ---------------------------------------------------------------------------
# The library's rule.

MODE_DEFAULT = 0
MODE_OLD = 1
MODE_EXACT = 2
MODE_CORRECTED = 3


def params(N: int, k: int, eps: float, mode: int = MODE_DEFAULT):
    """(S, t, M) as the library computes them (see the module docstring)."""
    if mode == MODE_OLD:
        S, t, M = params_old(N, k, eps)
        S = min(S, N)
        return S, min(max(t, 1), S), min(max(M, k), N)
    if mode == MODE_CORRECTED:  # the corrected Algorithm 1 throughout, GB300 calibration
        return params_corrected(N, k, eps)
    S = min(sample_size_old(N, k, eps), N)
    if mode == MODE_EXACT:  # Theorem 4 at that S
        t, M = params_exact(N, k, S, eps)
        return S, min(max(t, 1), S), min(max(M, k), N)
    t, M = params_fast(N, k, S, eps)
    return S, t, M

