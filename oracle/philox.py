"""Counter-based random numbers and the without-replacement sampler.

Prof-K's first stage draws S indices uniformly *without replacement* from
[N] (paper, Section 3 "The Prof-K Algorithm", stage 1 "Sampling"; Section 4
"Notation and Conventions": the sample is a uniformly random S-subset).  The
pages do not say how the subset is drawn.  The reading taken here, shared with
the CUDA library only as a written definition (no code is shared):

Draw stream.  For a call with user seed ``seed``, batch row ``row`` and
attempt ``attempt`` (0 for the first pass, +1 per redraw), draw number i
(i = 0, 1, 2, ...) is produced as follows.  Rejection round j starts at 0.

  1. w = Philox4x64-10(counter=(i // 4, attempt, j, 0), key=(seed, row))[i % 4]
  2. Lemire's bounded integer: m = w * n as a 128-bit product; let lo be its
     low 64 bits.  If lo < (2^64 - n) mod n the word is rejected: j += 1 and
     go to 1.  Otherwise the draw is u_i = m >> 64, uniform on [0, n).

Sample.  The sample is the first S *distinct* values of u_0, u_1, ..., in order
of first appearance.  Rejecting repeats while drawing i.i.d. uniform indices
yields every ordered S-tuple of distinct indices with probability
1 / (n (n-1) ... (n-S+1)), so the set is a uniform S-subset, as the analysis
requires.

Philox4x64-10 is the generator of Salmon, Moraes, Dror and Shaw, "Parallel
random numbers: as easy as 1, 2, 3" (SC'11): ten rounds of two 64x64->128
multiplications, with the key bumped by two Weyl constants between rounds.
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


def lemire_accept(w: int, n: int, bits: int = 64):
    """Lemire's multiply-shift bounded integer for one word of ``bits`` bits.

    Returns the value in [0, n) or None when the word is rejected.  ``bits`` is
    a parameter only so that tests can check the method exhaustively on small
    words; the sampler uses 64.
    """
    full = 1 << bits
    m = w * n
    lo = m & (full - 1)
    if lo < (full - n) % n:
        return None
    return m >> bits


def draw_values(n: int, seed: int, row: int, attempt: int, start: int, stop: int) -> np.ndarray:
    """Draws u_start .. u_{stop-1} of the stream defined in the module docstring."""
    if not (1 <= n <= (1 << 32)):
        raise ValueError("n must be in [1, 2^32]")
    if stop <= start:
        return np.empty(0, dtype=np.int64)
    b0, b1 = start >> 2, ((stop - 1) >> 2) + 1
    blocks = np.arange(b0, b1, dtype=np.uint64)
    w = np.stack(philox4x64(blocks, attempt, 0, 0, seed, row), axis=1).reshape(-1)
    w = w[start - 4 * b0: stop - 4 * b0]
    hi, lo = mulhilo64(w, np.uint64(n))
    thr = np.uint64(((1 << 64) - n) % n)
    out = hi.astype(np.int64)
    for p in np.flatnonzero(lo < thr):
        i = start + int(p)
        j = 1
        while True:
            word = philox4x64_scalar((i >> 2, attempt, j, 0), (seed, row))[i & 3]
            v = lemire_accept(word, n)
            if v is not None:
                out[p] = v
                break
            j += 1
    return out


def draw_values_many(n: int, seeds, row: int, attempt: int, stop: int) -> np.ndarray:
    """Draws u_0 .. u_{stop-1} for many seeds at once (int64[len(seeds), stop])."""
    seeds = np.asarray(seeds, dtype=np.uint64).reshape(-1, 1)
    nb = (stop + 3) >> 2
    blocks = np.arange(nb, dtype=np.uint64).reshape(1, -1)
    w = np.stack(philox4x64(blocks, attempt, 0, 0, seeds, row), axis=2).reshape(seeds.shape[0], -1)[:, :stop]
    hi, lo = mulhilo64(w, np.uint64(n))
    thr = np.uint64(((1 << 64) - n) % n)
    out = hi.astype(np.int64)
    for r, p in zip(*np.nonzero(lo < thr)):
        i, j = int(p), 1
        while True:
            word = philox4x64_scalar((i >> 2, attempt, j, 0), (int(seeds[r, 0]), row))[i & 3]
            v = lemire_accept(word, n)
            if v is not None:
                out[r, p] = v
                break
            j += 1
    return out


def sample_indices(n: int, S: int, seed: int, row: int = 0, attempt: int = 0) -> np.ndarray:
    """The first S distinct draws, in order of first appearance (int64[S])."""
    if not (1 <= S <= n):
        raise ValueError("need 1 <= S <= n")
    D = S + 64
    while True:
        u = draw_values(n, seed, row, attempt, 0, D)
        _, first = np.unique(u, return_index=True)
        if first.size >= S:
            return u[np.sort(first)[:S]]
        D *= 2
