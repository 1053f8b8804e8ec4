"""ctypes declarations of the C-ABI in include/profk.h (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "lib" / "libprofk.so"

PROFK_OK = 0
PROFK_ERR_INVALID = -1
PROFK_ERR_CUDA = -2
PROFK_ERR_NAN = -3
PROFK_ERR_UNSUPPORTED = -4
PROFK_ERR_DEVICE_TIMEOUT = -5
PROFK_ERR_SCRATCH = -6

PATH_FILTER, PATH_TIE, PATH_FALLBACK, PATH_EXACT = 0, 1, 2, 3
PARAMS_DEFAULT, PARAMS_OLD, PARAMS_EXACT, PARAMS_CORRECTED = 0, 1, 2, 3

OPT_PARAM_MODE = 0
OPT_MAX_ATTEMPTS = 1
OPT_TIE_EXIT = 2
OPT_FORCE_S = 3
OPT_FORCE_T = 4
OPT_FORCE_M = 5
OPT_TIMING = 6
OPT_FILTER_CTAS_PER_SM = 7
OPT_PDL = 8
OPT_MAX_SEGMENT = 9
OPT_SAMPLER = 10
SAMPLER_AUTO, SAMPLER_GRID, SAMPLER_STEPS, SAMPLER_LISTS = 0, 1, 2, 3
OPT_WAIT_TEST = 11
OPT_SPECULATIVE = 12
OPT_PREFIX_TEST = 13
WAIT_TEST_OFF, WAIT_TEST_SAMPLER, WAIT_TEST_REFINE, WAIT_TEST_SORT = 0, 1, 2, 3
OPT_DEFAULTS = {0: 0, 1: 6, 2: 1, 3: 0, 4: 0, 5: 0, 6: 0, 7: 0, 8: 1, 9: 0, 10: 0, 11: 0, 12: 0, 13: 0}


class ProfkStats(C.Structure):
    _fields_ = [
        ("S", C.c_int64), ("t", C.c_int64), ("M", C.c_int64),
        ("R_first", C.c_int64), ("R_gt_first", C.c_int64),
        ("R_final", C.c_int64), ("R_gt_final", C.c_int64),
        ("tau_first", C.c_float), ("tau_final", C.c_float),
        ("attempts", C.c_int32), ("path", C.c_int32),
        ("draw_doublings", C.c_int32), ("cuda_error", C.c_int32),
        ("aux_bytes", C.c_uint64),
        ("filter_ms", C.c_float), ("launches", C.c_int32),
    ]

    def as_dict(self) -> dict:
        return dict(zip(_STATS_NAMES, _STATS_FMT.unpack(bytes(self))))


_STATS_NAMES = tuple(name for name, _ in ProfkStats._fields_)
_STATS_FMT = __import__("struct").Struct("=7q2f4iQfi")
assert _STATS_FMT.size == C.sizeof(ProfkStats)


class ProfkError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (status {code})")
        self.code = code


_lib = None

_SIGS = {
    "profk_topk": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_double, C.c_uint64,
                             C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(ProfkStats)]),
    "profk_topk_batched": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_double,
                                     C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(ProfkStats)]),
    "profk_params": (C.c_int, [C.c_int64, C.c_int64, C.c_double, C.c_int,
                               C.POINTER(C.c_int64), C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "profk_workspace_size": (C.c_size_t, [C.c_int64, C.c_int64, C.c_int64, C.c_double]),
    "profk_set_workspace": (C.c_int, [C.c_void_p, C.c_size_t]),
    "profk_topk_async": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_double, C.c_uint64, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.POINTER(C.c_void_p)]),
    "profk_topk_batched_async": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_double,
                                           C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p,
                                           C.POINTER(C.c_void_p)]),
    "profk_wait": (C.c_int, [C.c_void_p, C.c_void_p]),
    "profk_set_option": (C.c_int, [C.c_int, C.c_int64]),
    "profk_get_option": (C.c_int64, [C.c_int]),
    "profk_strerror": (C.c_char_p, [C.c_int]),
    "profk_sample": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_uint64, C.c_int64, C.c_int32,
                               C.c_void_p, C.c_void_p, C.c_void_p]),
    "profk_threshold": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_void_p]),
    "profk_filter": (C.c_int, [C.c_void_p, C.c_int64, C.c_float, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "profk_refine": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int64, C.c_void_p,
                               C.c_void_p, C.c_void_p]),
    "profk_exact": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "profk_last_stage_ms": (C.c_int, [C.POINTER(C.c_float), C.c_int]),
    "profk_topk_noalloc": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_double, C.c_uint64,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(ProfkStats)]),
}


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
        h = C.CDLL(str(LIB_PATH))
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def check(code: int) -> None:
    if code != PROFK_OK:
        raise ProfkError(code, lib().profk_strerror(code).decode())
