// Host parameter rules of Prof-K (see params.cpp).
#pragma once

#include <cstdint>

namespace profk {

struct Params {
  int64_t S, t, M;
};

double inv_norm_cdf(double p);
int64_t sample_size_thm5(int64_t n, int64_t k, double eps);
// Corrected Algorithm 1, its sample-size steps (Proposition 7, GB300 cost ratio).
int64_t sample_size_corrected(int64_t n, int64_t k, double eps);
int64_t threshold_rank_fast(int64_t n, int64_t k, int64_t S, double eps);
int64_t buffer_capacity_fast(int64_t n, int64_t S, int64_t t, double eps);
// Theorem 4 (corrected version): exact optimal t and M for a given S.
void exact_params(int64_t n, int64_t k, int64_t S, double eps, int64_t* t, int64_t* M);
// mode 0: default rule, mode 1: the older version's Algorithm 1 literally,
// mode 2: S as in mode 0 with the exact t and M of Theorem 4,
// mode 3: the corrected Algorithm 1 throughout (its own sample size).
Params compute_params(int64_t n, int64_t k, double eps, int mode);
// Sample-and-filter when S <= n/8, t < S and M < n, and, for calls of 128 or
// more rows with k <= 2048, only when S < n/32; otherwise the exact path runs.
bool uses_filter(const Params& P, int64_t n, int64_t k, int64_t rows = 1);

}  // namespace profk
