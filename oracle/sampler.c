/* The oracle's sampler in plain C: test infrastructure only.
 *
 * The same definition as oracle/philox.py (which states it in full and
 * cites its sources): the sample of S indices from [0, n) is pi(0), ...,
 * pi(S-1), where pi is a twelve-round Feistel network on [0, 2^b),
 * b = max(2, ceil(log2 n)), with round function f_i(R) = mix(R xor K_i)
 * (mix: the SplitMix64 output function; K_0 .. K_11: the words of the
 * Philox4x64-10 blocks (q, attempt, 0, 0), q = 0, 1, 2, under the key
 * (seed, row)), cycle-walked into [0, n).  Philox4x64-10 follows Salmon,
 * Moraes, Dror and Shaw (SC'11).  Written for clarity: exact 128-bit
 * products through unsigned __int128, one scalar at a time.  Only the tests
 * and the Monte-Carlo checks call it; the CUDA library shares none of it. */
#include <stdint.h>

typedef unsigned __int128 u128;

void oracle_philox4x64_10(const uint64_t ctr[4], uint64_t k0, uint64_t k1, uint64_t out[4]) {
  uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B97F4A7C15ull; /* golden ratio */
      k1 += 0xBB67AE8584CAA73Bull; /* sqrt(3) - 1 */
    }
    const u128 p0 = (u128)0xD2E7470EE14C6C93ull * c0;
    const u128 p1 = (u128)0xCA5A826395121157ull * c2;
    const uint64_t d0 = (uint64_t)(p1 >> 64) ^ c1 ^ k0;
    const uint64_t d1 = (uint64_t)p1;
    const uint64_t d2 = (uint64_t)(p0 >> 64) ^ c3 ^ k1;
    const uint64_t d3 = (uint64_t)p0;
    c0 = d0;
    c1 = d1;
    c2 = d2;
    c3 = d3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

int oracle_domain_bits(uint64_t n) {
  int b = 0;
  while (b < 64 && ((uint64_t)1 << b) < n) ++b;
  return b < 2 ? 2 : b;
}

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

void oracle_round_keys(uint64_t seed, uint64_t row, uint64_t attempt, uint64_t keys[12]) {
  for (uint64_t q = 0; q < 3; ++q) {
    const uint64_t ctr[4] = {q, attempt, 0, 0};
    oracle_philox4x64_10(ctr, seed, row, keys + 4 * q);
  }
}

uint64_t oracle_feistel(uint64_t x, int bits, const uint64_t keys[12]) {
  int w = bits / 2; /* width of the low part entering the round */
  for (int i = 0; i < 12; ++i) {
    const int wl = bits - w;
    const uint64_t right = x & (((uint64_t)1 << w) - 1);
    const uint64_t left = x >> w;
    x = (right << wl) | (left ^ (mix64(right ^ keys[i]) & (((uint64_t)1 << wl) - 1)));
    w = wl;
  }
  return x;
}

static uint64_t permute_keys(uint64_t j, uint64_t n, const uint64_t keys[12]) {
  const int b = oracle_domain_bits(n);
  uint64_t x = oracle_feistel(j, b, keys);
  while (x >= n) x = oracle_feistel(x, b, keys);
  return x;
}

uint64_t oracle_permute(uint64_t j, uint64_t n, uint64_t seed, uint64_t row, uint64_t attempt) {
  uint64_t keys[12];
  oracle_round_keys(seed, row, attempt, keys);
  return permute_keys(j, n, keys);
}

/* out[0..S) = pi(0), ..., pi(S-1); 0 on success, -1 unless 1 <= S <= n. */
int oracle_sample(uint64_t n, uint64_t S, uint64_t seed, uint64_t row, uint64_t attempt, int64_t* out) {
  if (S < 1 || S > n) return -1;
  uint64_t keys[12];
  oracle_round_keys(seed, row, attempt, keys);
  for (uint64_t j = 0; j < S; ++j) out[j] = (int64_t)permute_keys(j, n, keys);
  return 0;
}

/* The samples of many seeds: out[s * S + j] for seeds[s]. */
int oracle_sample_many(uint64_t n, uint64_t S, const uint64_t* seeds, int64_t nseeds, uint64_t row,
                       uint64_t attempt, int64_t* out) {
  for (int64_t s = 0; s < nseeds; ++s)
    if (oracle_sample(n, S, seeds[s], row, attempt, out + s * (int64_t)S) != 0) return -1;
  return 0;
}
