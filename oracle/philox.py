"""Counter-based random numbers and the without-replacement sampler.

Prof-K's first stage draws S indices uniformly *without replacement* from
[N] (paper, Section 3 "The Prof-K Algorithm", stage 1 "Sampling"; Section 4
"Notation and Conventions": the sample is a uniformly random S-subset).  The
pages do not say how the subset is drawn.  The reading taken here, shared with
the CUDA library only as a written definition (no code is shared):

Permutation.  For a call with user seed ``seed``, batch row ``row`` and
attempt ``attempt`` (0 for the first pass, +1 per redraw), a keyed
pseudo-random permutation pi of [0, n) is built in two steps.

  1. Round keys K_0 .. K_11: the twelve words of the Philox4x64-10 blocks
     with counters (q, attempt, 0, 0), q = 0, 1, 2, under the key (seed, row),
     in order.
  2. A Feistel network E on [0, 2^b), b = max(2, ceil(log2 n)), of twelve
     rounds.  The state x is split into a high part L and a low part R of
     width w (w = floor(b/2) in round 0); round i maps it to
         x' = (R << (b - w)) | (L xor (f_i(R) mod 2^(b - w)))
     and the next round splits at w' = b - w.  Every round is invertible, so
     E permutes [0, 2^b).  The round function is f_i(R) = mix(R xor K_i),
     mix being the SplitMix64 output function (Steele, Lea and Flood, "Fast
     splittable pseudorandom number generators", OOPSLA 2014):
         z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
         z *= 0x94D049BB133111EB; z ^= z >> 31     (mod 2^64).
  3. Cycle-walking into [0, n): pi(j) = the first of E(j), E(E(j)), ... that
     is below n.  Because E is a permutation and j < n, the walk returns to
     [0, n), and pi is a permutation of [0, n) (Black and Rogaway, "Ciphers
     with arbitrary finite domains", CT-RSA 2002).  Since 2^b < 2n, a walk
     takes fewer than two steps on average.

Sample.  The sample is pi(0), pi(1), ..., pi(S-1): S distinct indices by
construction, in that order.  With enough rounds of a well-mixing round
function the set is a uniform S-subset to the precision the analysis needs;
twelve rounds are where the subset law passes a chi-square test even on
domains of 3 to 8 elements (four rounds of the same kind fail there), and the
tests also check the positions of the indices and Lemma 1 by Monte Carlo.

Philox4x64-10 is the generator of Salmon, Moraes, Dror and Shaw, "Parallel
random numbers: as easy as 1, 2, 3" (SC'11): ten rounds of two 64x64->128
multiplications, with the key bumped by two Weyl constants between rounds.

This module writes the definition out in numpy (slow, vectorised); the same
definition in plain C (oracle/sampler.c, through oracle.csample) serves the
Monte-Carlo tests, which need about 10^9 round-function calls, and the tests
require the two to agree element by element.
"""
from __future__ import annotations

import numpy as np

# Constants of Philox4x64 as published by Salmon et al. (SC'11).
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15  # golden ratio
PHILOX_W1 = 0xBB67AE8584CAA73B  # sqrt(3) - 1
_MASK64 = (1 << 64) - 1
_M32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def philox4x64_scalar(ctr, key, rounds: int = 10):
    """Reference Philox4x64 on Python integers (exact 128-bit products)."""
    c = [int(v) & _MASK64 for v in ctr]
    k0, k1 = (int(v) & _MASK64 for v in key)
    for r in range(rounds):
        if r:
            k0 = (k0 + PHILOX_W0) & _MASK64
            k1 = (k1 + PHILOX_W1) & _MASK64
        p0 = PHILOX_M0 * c[0]
        p1 = PHILOX_M1 * c[2]
        c = [(p1 >> 64) ^ c[1] ^ k0, p1 & _MASK64, (p0 >> 64) ^ c[3] ^ k1, p0 & _MASK64]
    return c


def mulhilo64(a, b):
    """64x64 -> (hi, lo) 128-bit product of uint64 arrays, by 32-bit halves."""
    a = np.asarray(a, dtype=np.uint64)
    b = np.asarray(b, dtype=np.uint64)
    a0, a1 = a & _M32, a >> _S32
    b0, b1 = b & _M32, b >> _S32
    p00 = a0 * b0
    p01 = a0 * b1
    p10 = a1 * b0
    p11 = a1 * b1
    mid = (p00 >> _S32) + (p01 & _M32) + (p10 & _M32)
    lo = (p00 & _M32) | ((mid & _M32) << _S32)
    hi = p11 + (p01 >> _S32) + (p10 >> _S32) + (mid >> _S32)
    return hi, lo


def philox4x64(c0, c1, c2, c3, k0, k1, rounds: int = 10):
    """Vectorised Philox4x64 over broadcastable uint64 arrays."""
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint64) for v in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64)
    k1 = np.asarray(k1, dtype=np.uint64)
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(c0, c1, c2, c3, k0, k1)
    w0, w1 = np.uint64(PHILOX_W0), np.uint64(PHILOX_W1)
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    with np.errstate(over="ignore"):
        for r in range(rounds):
            if r:
                k0 = k0 + w0
                k1 = k1 + w1
            hi0, lo0 = mulhilo64(m0, c0)
            hi1, lo1 = mulhilo64(m1, c2)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


FEISTEL_ROUNDS = 12
MIX_M1 = 0xBF58476D1CE4E5B9  # SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014)
MIX_M2 = 0x94D049BB133111EB


def domain_bits(n: int) -> int:
    """b = max(2, ceil(log2 n)): the Feistel network permutes [0, 2^b), 2^b >= n."""
    return max(2, (int(n) - 1).bit_length())


def round_keys(seed: int, row: int, attempt: int) -> list:
    """K_0 .. K_11: the words of Philox4x64-10 blocks (q, attempt, 0, 0), q = 0, 1, 2."""
    keys = []
    for q in range((FEISTEL_ROUNDS + 3) // 4):
        keys += philox4x64_scalar((q, attempt, 0, 0), (seed, row))
    return keys[:FEISTEL_ROUNDS]


def mix64(z):
    """The SplitMix64 output function on uint64 arrays (products mod 2^64)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX_M2)
        return z ^ (z >> np.uint64(31))


def feistel(x, bits: int, keys) -> np.ndarray:
    """E(x) for every x of a uint64 array: the rounds of the module docstring."""
    x = np.asarray(x, dtype=np.uint64).copy()
    w = bits // 2
    for k in keys:
        wl = bits - w
        right = x & np.uint64((1 << w) - 1)
        left = x >> np.uint64(w)
        f = mix64(right ^ np.uint64(k))
        x = (right << np.uint64(wl)) | (left ^ (f & np.uint64((1 << wl) - 1)))
        w = wl
    return x


def permute(j, n: int, seed: int, row: int = 0, attempt: int = 0) -> np.ndarray:
    """pi(j) for every j (all < n): E applied until the value falls below n."""
    j = np.asarray(j, dtype=np.uint64)
    if j.size and int(j.max()) >= n:
        raise ValueError("need j < n")
    b = domain_bits(n)
    keys = round_keys(seed, row, attempt)
    out = feistel(j, b, keys)
    walking = np.flatnonzero(out >= np.uint64(n))
    while walking.size:
        out[walking] = feistel(out[walking], b, keys)
        walking = walking[out[walking] >= np.uint64(n)]
    return out.astype(np.int64)


def sample_indices_numpy(n: int, S: int, seed: int, row: int = 0, attempt: int = 0) -> np.ndarray:
    """The sample pi(0), ..., pi(S-1) (int64[S]), by the numpy definition."""
    if not (1 <= S <= n):
        raise ValueError("need 1 <= S <= n")
    return permute(np.arange(S, dtype=np.uint64), n, seed, row, attempt)


def sample_indices(n: int, S: int, seed: int, row: int = 0, attempt: int = 0) -> np.ndarray:
    """The sample pi(0), ..., pi(S-1) (int64[S]), by the C form of the same
    definition (oracle/sampler.c), which the tests hold equal to the numpy one."""
    from . import csample

    return csample.sample_indices(n, S, seed, row, attempt)
