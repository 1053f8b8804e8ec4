"""The C-ABI library without a GPU: it builds, loads, exports every declared
symbol, and its host-only entry points (parameters, options, argument checks)
agree with the oracle.  No call here launches device work."""
import ctypes as C
import re
from pathlib import Path

import pytest

from oracle import params as P

HEADER = Path(__file__).resolve().parent.parent / "include" / "profk.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(profk_[a-z_]+)\s*\(", text)))


def test_header_declares_the_method(pk):
    names = declared_functions()
    for must in ("profk_topk", "profk_topk_batched", "profk_params", "profk_workspace_size",
                 "profk_set_option", "profk_get_option", "profk_strerror", "profk_sample",
                 "profk_threshold", "profk_filter", "profk_refine", "profk_exact", "profk_set_workspace",
                 "profk_topk_async", "profk_topk_batched_async", "profk_wait"):
        assert must in names


def test_library_exports_every_declared_symbol(pk):
    lib = pk.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_params_match_oracle(pk, mode):
    # The oracle's exact search (mode 2) is slow, so it gets a smaller grid.
    Ns = (1 << 20, 1 << 22, 1 << 26, 1 << 28, 1 << 30, 50331648, 1 << 24, 3_000_000_000, 1 << 32)
    ks = (1, 2, 32, 64, 1024, 4096, 32768, 131072, 1 << 19)
    if mode == 2:
        Ns, ks = (1 << 20, 1 << 26, 1 << 30, 3_000_000_000), (1, 32, 1024, 131072)
    for N in Ns:
        for k in ks:
            for eps in (1e-3, 1e-3 / 64, 0.05):
                if k > N:
                    continue
                assert pk.params(N, k, eps, mode) == P.params(N, k, eps, mode), (N, k, eps, mode)


def test_options_roundtrip_and_validation(pk):
    assert pk.get_option(pk.OPT_MAX_ATTEMPTS) == 6
    pk.set_option(pk.OPT_MAX_ATTEMPTS, 2)
    assert pk.get_option(pk.OPT_MAX_ATTEMPTS) == 2
    with pytest.raises(pk.ProfkError):
        pk.set_option(99, 1)
    with pytest.raises(pk.ProfkError):
        pk.set_option(pk.OPT_PARAM_MODE, 5)
    pk.set_option(pk.OPT_PARAM_MODE, 2)  # the exact Theorem 4 mode
    with pytest.raises(pk.ProfkError):
        pk.set_option(pk.OPT_FORCE_S, -1)
    assert pk.get_option(pk.OPT_SAMPLER) == pk.SAMPLER_AUTO
    for form in (pk.SAMPLER_GRID, pk.SAMPLER_STEPS, pk.SAMPLER_LISTS, pk.SAMPLER_AUTO):
        pk.set_option(pk.OPT_SAMPLER, form)
        assert pk.get_option(pk.OPT_SAMPLER) == form
    for bad in (-1, 4):
        with pytest.raises(pk.ProfkError):
            pk.set_option(pk.OPT_SAMPLER, bad)


def test_strerror(pk):
    lib = pk.lib()
    for code in range(-6, 1):
        assert lib.profk_strerror(code) and lib.profk_strerror(code) != b"unknown status"
    assert b"NaN" in lib.profk_strerror(-3)
    assert b"scratch" in lib.profk_strerror(-6)


def test_invalid_arguments_are_rejected_before_any_device_work(pk):
    lib = pk.lib()
    st = pk.ProfkStats()
    assert lib.profk_topk(None, 10, 1, 1e-3, 0, None, None, None, C.byref(st)) == -1
    fake = C.c_void_p(256)  # never dereferenced: the arguments fail validation first
    assert lib.profk_topk(fake, 10, 0, 1e-3, 0, fake, fake, None, None) == -1
    assert lib.profk_topk(fake, 10, 11, 1e-3, 0, fake, fake, None, None) == -1
    assert lib.profk_topk(fake, 10, 1, 0.0, 0, fake, fake, None, None) == -1
    assert lib.profk_topk(fake, 10, 1, 1.0, 0, fake, fake, None, None) == -1
    assert lib.profk_topk(fake, 1 << 40, 1, 1e-3, 0, fake, fake, None, None) == -4
    assert lib.profk_topk(C.c_void_p(258), 10, 1, 1e-3, 0, fake, fake, None, None) == -4
    assert lib.profk_topk_batched(fake, 0, 10, 10, 1, 1e-3, 0, fake, fake, None, None) == -1
    assert lib.profk_topk_batched(fake, 2, 10, 9, 1, 1e-3, 0, fake, fake, None, None) == -1
    # x must be a float pointer (4-byte aligned); any row stride ld >= n is taken.
    assert lib.profk_topk_batched(C.c_void_p(258), 2, 10, 10, 1, 1e-3, 0, fake, fake, None, None) == -4
    assert lib.profk_sample(fake, 10, 11, 0, 0, 0, fake, fake, None) == -1  # S > n
    assert lib.profk_threshold(fake, 10, 11, fake, None) == -1
    assert lib.profk_refine(fake, 5, 6, fake, 10, fake, fake, None) == -1
    assert lib.profk_exact(fake, 10, 11, fake, fake, None) == -1
    S, t, M = C.c_int64(), C.c_int64(), C.c_int64()
    assert lib.profk_params(10, 11, 1e-3, 0, C.byref(S), C.byref(t), C.byref(M)) == -1


def test_workspace_is_O_M_plus_S(pk):
    small = pk.workspace_size(1, 1 << 26, 1024)
    big = pk.workspace_size(1, 1 << 30, 1024)
    assert 0 < big < 16 << 20  # megabytes, not a fraction of the 4 GiB input
    assert big < 16 * small
    assert pk.workspace_size(1, 10, 11) == 0


def test_set_workspace_validation(pk):
    lib = pk.lib()
    assert lib.profk_set_workspace(C.c_void_p(256 + 8), 1 << 20) == -1  # not 256-byte aligned
    assert lib.profk_set_workspace(None, 0) == 0
    assert lib.profk_set_workspace(C.c_void_p(1 << 20), 0) == 0  # zero bytes: back to the pool


def test_async_argument_checks(pk):
    lib = pk.lib()
    h = C.c_void_p(7)
    fake = C.c_void_p(256)
    assert lib.profk_topk_async(None, 10, 1, 1e-3, 0, fake, fake, None, C.byref(h)) == -1
    assert not h.value  # no call was created
    assert lib.profk_topk_async(fake, 10, 1, 1e-3, 0, fake, fake, None, None) == -1
    assert lib.profk_topk_batched_async(C.c_void_p(258), 2, 10, 10, 1, 1e-3, 0, fake, fake, None, C.byref(h)) == -4
    assert lib.profk_wait(None, None) == -1


def test_long_row_workspace_size(pk):
    # A row beyond the split point needs the larger of its segment calls plus
    # 12 bytes per merged candidate.  The plan: P = ceil(n / 2^32) segments of
    # ceil(n / P) rounded up to a multiple of 4, the last one possibly shorter;
    # equal segments go through one batched call, a shorter last one alone.
    round256 = lambda v: (v + 255) // 256 * 256
    k = 1 << 18
    n = 4_300_000_000  # two equal segments: one batched call of two rows
    seg = n // 2
    cand = 2 * k
    assert pk.workspace_size(1, n, k, 1e-3) == (round256(pk.workspace_size(2, seg, k, 1e-3))
                                                 + round256(4 * cand) + round256(8 * cand))
    n = 4_300_000_004  # ceil(n / 2) = 2,150,000,002 -> 2,150,000,004; the tail has 2,150,000,000
    seg, tail = 2_150_000_004, 2_150_000_000
    need = max(pk.workspace_size(1, seg, k, 1e-3 / 2), pk.workspace_size(1, tail, k, 1e-3 / 2))
    assert pk.workspace_size(1, n, k, 1e-3) == round256(need) + round256(4 * cand) + round256(8 * cand)
    assert pk.workspace_size(1, 1 << 40, 1, 1e-3) == 0


def test_noalloc_argument_and_size_checks(pk):
    # The entry point that allocates nothing refuses, before any device work:
    # bad arguments, rows beyond 2^32 elements or not float-aligned, and problems whose
    # workspace does not fit its fixed scratch (k = n = 2^23 takes the exact
    # route and needs 8 x 2^23 bytes of selection keys, beyond 32 MiB).
    from streaming_selection_primitive_gb300 import _abi
    lib = pk.lib()
    fake = C.c_void_p(256)
    st = pk.ProfkStats()
    assert lib.profk_topk_noalloc(None, 10, 1, 1e-3, 0, fake, fake, None, C.byref(st)) == _abi.PROFK_ERR_INVALID
    assert lib.profk_topk_noalloc(fake, 10, 11, 1e-3, 0, fake, fake, None, None) == _abi.PROFK_ERR_INVALID
    assert lib.profk_topk_noalloc(fake, (1 << 32) + 4, 1, 1e-3, 0, fake, fake, None, None) == \
        _abi.PROFK_ERR_UNSUPPORTED
    assert lib.profk_topk_noalloc(C.c_void_p(258), 100, 1, 1e-3, 0, fake, fake, None, None) == \
        _abi.PROFK_ERR_UNSUPPORTED
    assert lib.profk_topk_noalloc(fake, 1 << 23, 1 << 23, 1e-3, 0, fake, fake, None, None) == \
        _abi.PROFK_ERR_SCRATCH


def test_wait_test_option(pk):
    # The test setting of the bounded device waits: off by default, one of the
    # three persistent kernels, nothing else.
    assert pk.get_option(pk.OPT_WAIT_TEST) == pk.WAIT_TEST_OFF
    for v in (pk.WAIT_TEST_SAMPLER, pk.WAIT_TEST_REFINE, pk.WAIT_TEST_SORT, pk.WAIT_TEST_OFF):
        pk.set_option(pk.OPT_WAIT_TEST, v)
        assert pk.get_option(pk.OPT_WAIT_TEST) == v
    for bad in (4, -1):
        with pytest.raises(pk.ProfkError):
            pk.set_option(pk.OPT_WAIT_TEST, bad)


def test_speculative_option(pk):
    # Attempts enqueued after the first: off by default, 0 .. 8.
    assert pk.get_option(pk.OPT_SPECULATIVE) == 0
    for v in (8, 1, 0):
        pk.set_option(pk.OPT_SPECULATIVE, v)
        assert pk.get_option(pk.OPT_SPECULATIVE) == v
    for bad in (9, -1):
        with pytest.raises(pk.ProfkError):
            pk.set_option(pk.OPT_SPECULATIVE, bad)


def test_prefix_test_option(pk):
    # The test setting of the grid refinement's prefix check: off by default,
    # 1 .. 33 (the number of trusted low bits of the filter's record, plus one).
    assert pk.get_option(pk.OPT_PREFIX_TEST) == 0
    for v in (1, 9, 33, 0):
        pk.set_option(pk.OPT_PREFIX_TEST, v)
        assert pk.get_option(pk.OPT_PREFIX_TEST) == v
    for bad in (34, -1):
        with pytest.raises(pk.ProfkError):
            pk.set_option(pk.OPT_PREFIX_TEST, bad)
