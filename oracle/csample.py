"""ctypes access to the oracle's sampler in plain C (oracle/sampler.c).

TEST INFRASTRUCTURE ONLY, like the rest of oracle/.  The library is compiled
here with gcc on first use (or by the build entry point) into oracle/_build/;
it shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "sampler.c"
LIB = HERE / "_build" / "liboracle_sampler.so"

_lib = None


def build() -> Path:
    """Compiles sampler.c when the library is missing or older than it."""
    if LIB.exists() and LIB.stat().st_mtime >= SRC.stat().st_mtime:
        return LIB
    LIB.parent.mkdir(exist_ok=True)
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp")
    subprocess.run(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", str(SRC), "-o", str(tmp)], check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        h = C.CDLL(str(build()))
        u64, i64 = C.c_uint64, C.c_int64
        h.oracle_philox4x64_10.argtypes = [C.POINTER(u64), u64, u64, C.POINTER(u64)]
        h.oracle_philox4x64_10.restype = None
        h.oracle_feistel.argtypes = [u64, C.c_int, C.POINTER(u64)]
        h.oracle_feistel.restype = u64
        h.oracle_round_keys.argtypes = [u64, u64, u64, C.POINTER(u64)]
        h.oracle_round_keys.restype = None
        h.oracle_permute.argtypes = [u64, u64, u64, u64, u64]
        h.oracle_permute.restype = u64
        h.oracle_domain_bits.argtypes = [u64]
        h.oracle_domain_bits.restype = C.c_int
        h.oracle_sample.argtypes = [u64, u64, u64, u64, u64, C.POINTER(i64)]
        h.oracle_sample.restype = C.c_int
        h.oracle_sample_many.argtypes = [u64, u64, C.POINTER(u64), i64, u64, u64, C.POINTER(i64)]
        h.oracle_sample_many.restype = C.c_int
        _lib = h
    return _lib


def philox4x64(ctr, key):
    c = (C.c_uint64 * 4)(*[int(v) & (2**64 - 1) for v in ctr])
    o = (C.c_uint64 * 4)()
    _load().oracle_philox4x64_10(c, int(key[0]) & (2**64 - 1), int(key[1]) & (2**64 - 1), o)
    return [int(v) for v in o]


def round_keys(seed: int, row: int, attempt: int) -> list:
    k = (C.c_uint64 * 12)()
    _load().oracle_round_keys(int(seed) & (2**64 - 1), row, attempt, k)
    return [int(v) for v in k]


def feistel(x: int, bits: int, keys) -> int:
    k = (C.c_uint64 * 12)(*[int(v) for v in keys])
    return int(_load().oracle_feistel(x, bits, k))


def permute(j: int, n: int, seed: int, row: int = 0, attempt: int = 0) -> int:
    return int(_load().oracle_permute(j, n, seed, row, attempt))


def sample_indices(n: int, S: int, seed: int, row: int = 0, attempt: int = 0) -> np.ndarray:
    if not (1 <= S <= n):
        raise ValueError("need 1 <= S <= n")
    out = np.empty(S, dtype=np.int64)
    rc = _load().oracle_sample(n, S, int(seed) & (2**64 - 1), row, attempt,
                               out.ctypes.data_as(C.POINTER(C.c_int64)))
    if rc != 0:
        raise ValueError("need 1 <= S <= n")
    return out


def sample_many(n: int, S: int, seeds, row: int = 0, attempt: int = 0) -> np.ndarray:
    """The samples of every seed (int64[len(seeds), S])."""
    sd = np.ascontiguousarray(np.asarray(seeds, dtype=np.uint64))
    out = np.empty((sd.size, S), dtype=np.int64)
    rc = _load().oracle_sample_many(n, S, sd.ctypes.data_as(C.POINTER(C.c_uint64)), sd.size, row, attempt,
                                    out.ctypes.data_as(C.POINTER(C.c_int64)))
    if rc != 0:
        raise ValueError("need 1 <= S <= n")
    return out
