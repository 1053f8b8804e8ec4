// Parameter selection (S, t, M) of Prof-K, host fp64.
//
// Sources ("Prof-K: Probabilistic One-Pass Filtering for Efficient Top-k
// Selection"; two versions of the page exist and are cited separately):
//  * older version, Theorem 5 (Eq 14) and its Algorithm 1, the sample-size step:
//      z = 2 Phi^{-1}(1 - eps/2),  S* = (z log2(k) / 2)^(2/3) (k (n-k))^(1/3),
//      S = clamp(round(S*), 32768, 131072);
//  * corrected version, Algorithm 1, the t and M steps (Appendix B, Eq 9-12), with
//    z = Phi^{-1}(1 - eps/2) by Acklam's rational approximation:
//      mu = (k-1) S / n;
//      mu >= 15: t = ceil(mu + z sigma + (z^2 - 1)/6) + 1,
//                sigma^2 = mu (1 - (k-1)/n) (n - S)/(n - 1)      (Eq 10)
//      mu <  15: t = 1 + min{j : Poisson(mu) cdf(j) >= 1 - eps/2} (Eq 11)
//      M = ceil((n+1)/(S+1) t (1 - h + z sqrt(h))^3), h = 1/(9t)  (Eq 12)
//  * older version, Algorithm 1 literally (Eq 6 t, Corollary 4 M, and t = 1
//    when (k/n) S < -ln(eps/2)) as the optional mode.
//  * corrected version, Algorithm 1 throughout (mode 3): its sample-size steps
//    with Proposition 7, kappa = z^2 + 1/2,
//      S1 = (z r(k)^-1)^(2/3) (k n)^(1/3),  S2 = (kappa n / r(k))^(1/2),
//      S = clip(floor(max(S1, S2)), 2^14, 2^18), 2^14 when r = infinity or
//      k/n > 2^-10, then at most n/128 (Table 3 uses n/128 at n = 2^20);
//    the cost ratio in the paper's form 1/r(k) = a log2 k + b for k > 2^7
//    (r = infinity below), with a and b fitted on a GB300 from an S sweep
//    of whole calls (Appendix E.1's procedure).
// The default mixes the two because the older t-rule sets t = 1 exactly where
// recall failure is likely; the corrected version replaces it.
#include <cmath>
#include <cstdint>

#include "params.h"

namespace profk {

double inv_norm_cdf(double p) {
  // P. J. Acklam's algorithm: a rational function of p - 1/2 in the central
  // region and of sqrt(-2 log(tail)) in the tails.
  static const double a[6] = {-3.969683028665376e+01, 2.209460984245205e+02, -2.759285104469687e+02,
                              1.383577518672690e+02,  -3.066479806614716e+01, 2.506628277459239e+00};
  static const double b[5] = {-5.447609879822406e+01, 1.615858368580409e+02, -1.556989798598866e+02,
                              6.680131188771972e+01,  -1.328068155288572e+01};
  static const double c[6] = {-7.784894002430293e-03, -3.223964580411365e-01, -2.400758277161838e+00,
                              -2.549732539343734e+00, 4.374664141464968e+00,  2.938163982698783e+00};
  static const double d[4] = {7.784695709041462e-03, 3.224671290700398e-01, 2.445134137142996e+00,
                              3.754408661907416e+00};
  const double plow = 0.02425;
  if (p < plow) {
    const double q = std::sqrt(-2.0 * std::log(p));
    return (((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) /
           ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1.0);
  }
  if (p > 1.0 - plow) {
    const double q = std::sqrt(-2.0 * std::log1p(-p));
    return -(((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) /
           ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1.0);
  }
  const double q = p - 0.5, r = q * q;
  return (((((a[0] * r + a[1]) * r + a[2]) * r + a[3]) * r + a[4]) * r + a[5]) * q /
         (((((b[0] * r + b[1]) * r + b[2]) * r + b[3]) * r + b[4]) * r + 1.0);
}

int64_t sample_size_thm5(int64_t n, int64_t k, double eps) {
  const double z = 2.0 * inv_norm_cdf(1.0 - eps / 2.0);
  double s = 0.0;
  if (k > 1) {
    const double kk = static_cast<double>(k), nn = static_cast<double>(n);
    s = std::pow(z * std::log2(kk) / 2.0, 2.0 / 3.0) * std::pow(kk * (nn - kk), 1.0 / 3.0);
  }
  double r = std::floor(s + 0.5);
  if (r < 32768.0) r = 32768.0;
  if (r > 131072.0) r = 131072.0;
  return static_cast<int64_t>(r);
}

int64_t threshold_rank_fast(int64_t n, int64_t k, int64_t S, double eps) {
  const double z = inv_norm_cdf(1.0 - eps / 2.0);
  const double N = static_cast<double>(n);
  const double mu = static_cast<double>(k - 1) * static_cast<double>(S) / N;
  if (mu >= 15.0) {
    const double sigma = std::sqrt(mu * (1.0 - static_cast<double>(k - 1) / N) * (N - static_cast<double>(S)) / (N - 1.0));
    return static_cast<int64_t>(std::ceil(mu + z * sigma + (z * z - 1.0) / 6.0)) + 1;
  }
  double p = std::exp(-mu), c = p;
  int64_t j = 0;
  while (c < 1.0 - eps / 2.0) {
    ++j;
    p = p * mu / static_cast<double>(j);
    c = c + p;
    if (j > 100000) break;  // unreachable for mu < 15; keeps the loop finite
  }
  return j + 1;
}

int64_t buffer_capacity_fast(int64_t n, int64_t S, int64_t t, double eps) {
  const double z = inv_norm_cdf(1.0 - eps / 2.0);
  const double h = 1.0 / (9.0 * static_cast<double>(t));
  const double w = 1.0 - h + z * std::sqrt(h);
  return static_cast<int64_t>(std::ceil((static_cast<double>(n) + 1.0) / (static_cast<double>(S) + 1.0) *
                                        static_cast<double>(t) * w * w * w));
}

static int64_t clamp64(int64_t v, int64_t lo, int64_t hi) { return v < lo ? lo : (v > hi ? hi : v); }

// ---- Exact optimal (t*, M*) for a given S: Theorem 4 of the corrected
// version (Section 4), with the failure budget split eps/2 + eps/2.
// X ~ Hypergeometric(N, K, S) counts the distinguished items among S drawn
// without replacement from N, K of them distinguished.  The first pmf term
// comes from log-binomials in extended precision, the next ones from the
// ratio Pr(X = j+1) / Pr(X = j) = (K-j)(S-j) / ((j+1)(N-K-S+j+1)).
namespace {

long double log_choose(long double a, long double b) {
  return std::lgamma(a + 1.0L) - std::lgamma(b + 1.0L) - std::lgamma(a - b + 1.0L);
}

// Walks the pmf upwards from the bottom of the support.
struct HyperWalk {
  int64_t N, K, S, j, hi;
  double lp;  // log Pr(X = j)
  HyperWalk(int64_t n, int64_t kk, int64_t s) : N(n), K(kk), S(s) {
    j = s - (n - kk) > 0 ? s - (n - kk) : 0;
    hi = kk < s ? kk : s;
    lp = static_cast<double>(log_choose(static_cast<long double>(K), static_cast<long double>(j)) +
                             log_choose(static_cast<long double>(N - K), static_cast<long double>(S - j)) -
                             log_choose(static_cast<long double>(N), static_cast<long double>(S)));
  }
  double pmf() const { return std::exp(lp); }
  void next() {
    lp += std::log(static_cast<double>(K - j)) + std::log(static_cast<double>(S - j)) -
          std::log(static_cast<double>(j + 1)) - std::log(static_cast<double>(N - K - S + j + 1));
    ++j;
  }
};

// Pr(X <= x).
double hyper_cdf(int64_t N, int64_t K, int64_t S, int64_t x) {
  HyperWalk w(N, K, S);
  if (x < w.j) return 0.0;
  if (x >= w.hi) return 1.0;
  double c = 0.0;
  for (;; w.next()) {
    c += w.pmf();
    if (w.j == x) break;
  }
  return c < 1.0 ? c : 1.0;
}

// min { x : Pr(X <= x) >= p }.
int64_t hyper_quantile(int64_t N, int64_t K, int64_t S, double p) {
  HyperWalk w(N, K, S);
  double c = 0.0;
  for (;; w.next()) {
    c += w.pmf();
    if (c >= p || w.j >= w.hi) return w.j;
  }
}

}  // namespace

void exact_params(int64_t n, int64_t k, int64_t S, double eps, int64_t* t, int64_t* M) {
  // t*: the smallest t with Pr(fewer than t of the top k - 1 are sampled) ...
  // i.e. t - 1 = the (1 - eps/2)-quantile of X_{k-1}; M*: the smallest M
  // with Pr(X_M <= t - 1) <= eps/2 (nonincreasing in M, zero at M = n).
  *t = hyper_quantile(n, k - 1, S, 1.0 - eps / 2.0) + 1;
  int64_t lo = k, hi = n;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (hyper_cdf(n, mid, S, *t - 1) <= eps / 2.0)
      hi = mid;
    else
      lo = mid + 1;
  }
  *M = lo;
}

// 1/r(k) of the corrected rule, fitted on a GB300: the buffer selection's cost
// per element barely grows with k on this GPU (its refinement is bound by
// latency, not by the number of keys), so the line is nearly flat.
constexpr double kInvRSlope = 0.0033, kInvRIntercept = 0.41;

int64_t sample_size_corrected(int64_t n, int64_t k, double eps) {
  const int64_t s_min = int64_t(1) << 14, s_max = int64_t(1) << 18;
  const double nn = static_cast<double>(n), kk = static_cast<double>(k);
  int64_t S = s_min;
  if (k > (1 << 7) && kk <= nn / 1024.0) {
    const double inv_r = kInvRSlope * std::log2(kk) + kInvRIntercept;
    if (inv_r > 0.0) {
      const double z = inv_norm_cdf(1.0 - eps / 2.0);
      const double kappa = z * z + 0.5;
      const double S1 = std::pow(z * inv_r, 2.0 / 3.0) * std::cbrt(kk * nn);
      const double S2 = std::sqrt(kappa * nn * inv_r);
      const double s = std::floor(std::max(S1, S2));
      S = s < static_cast<double>(s_min) ? s_min : (s > static_cast<double>(s_max) ? s_max : static_cast<int64_t>(s));
    }
  }
  if (S > n / 128) S = n / 128;
  return S < 1 ? 1 : S;
}

Params compute_params(int64_t n, int64_t k, double eps, int mode) {
  Params p{};
  if (mode == 3) {
    const int64_t S = sample_size_corrected(n, k, eps);
    const int64_t t = clamp64(threshold_rank_fast(n, k, S, eps), 1, S);
    p.S = S;
    p.t = t;
    p.M = clamp64(buffer_capacity_fast(n, S, t, eps), k, n);
    return p;
  }
  if (mode == 1) {
    const double z = 2.0 * inv_norm_cdf(1.0 - eps / 2.0);
    const double N = static_cast<double>(n), K = static_cast<double>(k);
    const double alpha = K / N;
    int64_t S = sample_size_thm5(n, k, eps);
    if (S > n) S = n;
    const double f = 1.0 - static_cast<double>(S) / N;
    const double Sd = static_cast<double>(S);
    int64_t t = static_cast<int64_t>(std::ceil(Sd * alpha + z / 2.0 * std::sqrt(Sd * alpha * (1.0 - alpha) * f)));
    if (t < 1) t = 1;
    int64_t M = static_cast<int64_t>(std::ceil(K + z * std::sqrt(K * (N - K) / Sd * f)));
    if (alpha * Sd < -std::log(eps / 2.0)) t = 1;
    p.S = S;
    p.t = clamp64(t, 1, S);
    p.M = clamp64(M, k, n);
    return p;
  }
  int64_t S = sample_size_thm5(n, k, eps);
  if (S > n) S = n;
  if (mode == 2) {
    int64_t t = 1, M = n;
    exact_params(n, k, S, eps, &t, &M);
    p.S = S;
    p.t = clamp64(t, 1, S);
    p.M = clamp64(M, k, n);
    return p;
  }
  const int64_t t = clamp64(threshold_rank_fast(n, k, S, eps), 1, S);
  const int64_t M = clamp64(buffer_capacity_fast(n, S, t, eps), k, n);
  p.S = S;
  p.t = t;
  p.M = M;
  return p;
}

bool uses_filter(const Params& P, int64_t n, int64_t k, int64_t rows) {
  // The sample at most n/8, and parameters that can meet the budget (t and M
  // below their clamps S and n, which they reach as k approaches n).  No cut
  // on k/n: sampling measured 4-6 times faster than the exact path for
  // k/n = 1/32 .. 1/8, and the corrected paper keeps the method there.
  if (8 * P.S > n || P.t >= P.S || P.M >= n) return false;
  // Many short rows: a sample of 1/32 of each row or more, drawn by random
  // access, costs more than selecting each row exactly inside one CTA.
  if (rows >= 128 && 32 * P.S >= n && k <= 2048) return false;
  return true;
}

}  // namespace profk
