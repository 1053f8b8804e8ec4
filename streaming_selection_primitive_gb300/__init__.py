"""Prof-K exact top-k selection on GB300: Python binding of libprofk.so.

Every step runs in the library's CUDA kernels; this module only marshals
arguments.  PyTorch supplies device memory and the current CUDA stream.  There
is no CPU fallback: a missing library or a non-CUDA tensor raises.

    import streaming_selection_primitive_gb300 as pk
    vals, idx, stats = pk.topk(x, k=1024, eps=1e-3, seed=0)   # x: 1-D float32 CUDA tensor
"""
from __future__ import annotations

import ctypes as C

from . import _abi
from ._abi import (OPT_FILTER_CTAS_PER_SM, OPT_FORCE_M, OPT_FORCE_S, OPT_FORCE_T, OPT_MAX_ATTEMPTS,
                   OPT_MAX_SEGMENT, OPT_PARAM_MODE, OPT_PDL, OPT_PREFIX_TEST, OPT_SAMPLER, OPT_SPECULATIVE, OPT_TIE_EXIT,
                   OPT_TIMING, OPT_WAIT_TEST, WAIT_TEST_OFF, WAIT_TEST_REFINE, WAIT_TEST_SAMPLER, WAIT_TEST_SORT, PARAMS_CORRECTED,
                   PARAMS_DEFAULT, PARAMS_EXACT, SAMPLER_AUTO, SAMPLER_GRID, SAMPLER_LISTS, SAMPLER_STEPS,
                   PARAMS_OLD, PATH_EXACT, PATH_FALLBACK, PATH_FILTER, PATH_TIE, ProfkError, ProfkStats)

__all__ = ["topk", "topk_batched", "topk_noalloc", "params", "workspace_size", "set_option", "get_option", "reset_options",
           "sample", "threshold", "filter_pass", "refine", "exact", "last_stage_ms", "ProfkError", "ProfkStats",
           "lib"]


def lib():
    return _abi.lib()


def _torch():
    import torch
    return torch


def _stream_handle(stream=None, device=None) -> int:
    """Raw cudaStream_t of `stream`, else of the current stream of `device`."""
    if stream is not None:
        return int(stream.cuda_stream)
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None and device is not None:
        return int(raw(device.index if device.index is not None else torch.cuda.current_device()))
    return int(torch.cuda.current_stream().cuda_stream)


def _need_cuda_f32(x, name="x"):
    torch = _torch()
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32:
        raise TypeError(f"{name} must be a float32 CUDA tensor")


def params(n: int, k: int, eps: float = 1e-3, mode: int = PARAMS_DEFAULT):
    """(S, t, M) as the library computes them (host arithmetic, no GPU needed)."""
    S, t, M = C.c_int64(), C.c_int64(), C.c_int64()
    _abi.check(lib().profk_params(int(n), int(k), float(eps), int(mode), C.byref(S), C.byref(t), C.byref(M)))
    return S.value, t.value, M.value


def workspace_size(rows: int, n: int, k: int, eps: float = 1e-3) -> int:
    return int(lib().profk_workspace_size(int(rows), int(n), int(k), float(eps)))


_user_workspace = None  # keeps the caller's buffer alive while it is registered


def set_workspace(buf=None):
    """Use the CUDA tensor `buf` (any dtype, contiguous, 256-byte aligned) as the
    workspace of this thread's topk / topk_batched calls; None returns to the
    library's memory pool.  A call that needs more than buf's bytes raises
    ProfkError (PROFK_ERR_SCRATCH)."""
    global _user_workspace
    if buf is None:
        _abi.check(lib().profk_set_workspace(None, 0))
        _user_workspace = None
        return
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("the workspace must be a contiguous CUDA tensor")
    _abi.check(lib().profk_set_workspace(buf.data_ptr(), buf.numel() * buf.element_size()))
    _user_workspace = buf


def set_option(option: int, value: int) -> None:
    _abi.check(lib().profk_set_option(int(option), int(value)))


def get_option(option: int) -> int:
    return int(lib().profk_get_option(int(option)))


def reset_options() -> None:
    for o, v in _abi.OPT_DEFAULTS.items():
        set_option(o, v)


STAGES = ("sample", "threshold", "filter", "refine", "readback", "call_wall")


def last_stage_ms() -> dict:
    """Stage times of this thread's last timed call (PROFK_OPT_TIMING on)."""
    buf = (C.c_float * 6)()
    m = lib().profk_last_stage_ms(buf, 6)
    return {STAGES[i]: buf[i] for i in range(max(m, 0))}


def topk(x, k: int, eps: float = 1e-3, seed: int = 0, out=None, stream=None):
    """Exact top-k of a 1-D float32 CUDA tensor: (values, int64 indices, stats dict)."""
    torch = _torch()
    _need_cuda_f32(x)
    if x.dim() != 1 or not x.is_contiguous():
        raise ValueError("x must be 1-D and contiguous")
    n = x.numel()
    if out is None:
        vals = torch.empty(k, dtype=torch.float32, device=x.device)
        idx = torch.empty(k, dtype=torch.int64, device=x.device)
    else:
        vals, idx = out
    st = ProfkStats()
    code = lib().profk_topk(x.data_ptr(), n, int(k), float(eps), int(seed) & (2**64 - 1), vals.data_ptr(),
                            idx.data_ptr(), _stream_handle(stream, x.device), C.byref(st))
    _abi.check(code)
    return vals, idx, st.as_dict()


def topk_noalloc(x, k: int, eps: float = 1e-3, seed: int = 0, out=None, stream=None):
    """topk through profk_topk_noalloc: the call itself allocates no device or
    pinned memory (the library's fixed scratch array serves it; calls that
    overlap on one device race on that array).  Pass ``out`` = (values, indices)
    to keep this wrapper from allocating the outputs too."""
    torch = _torch()
    _need_cuda_f32(x)
    if x.dim() != 1 or not x.is_contiguous():
        raise ValueError("x must be 1-D and contiguous")
    if out is None:
        vals = torch.empty(k, dtype=torch.float32, device=x.device)
        idx = torch.empty(k, dtype=torch.int64, device=x.device)
    else:
        vals, idx = out
    st = ProfkStats()
    code = lib().profk_topk_noalloc(x.data_ptr(), x.numel(), int(k), float(eps), int(seed) & (2**64 - 1),
                                    vals.data_ptr(), idx.data_ptr(), _stream_handle(stream, x.device), C.byref(st))
    _abi.check(code)
    return vals, idx, st.as_dict()


def topk_batched(x, k: int, eps: float = 1e-3, seed: int = 0, out=None, stream=None, stats: bool = True):
    """Exact top-k of each row of a 2-D float32 CUDA tensor (row stride x.stride(0)).
    Returns (values, indices, per-row stats dicts, or None when stats=False)."""
    torch = _torch()
    _need_cuda_f32(x)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    rows, n = x.shape
    if out is None:
        vals = torch.empty((rows, k), dtype=torch.float32, device=x.device)
        idx = torch.empty((rows, k), dtype=torch.int64, device=x.device)
    else:
        vals, idx = out
    sts = (ProfkStats * rows)() if stats else None
    code = lib().profk_topk_batched(x.data_ptr(), rows, n, x.stride(0), int(k), float(eps),
                                    int(seed) & (2**64 - 1), vals.data_ptr(), idx.data_ptr(),
                                    _stream_handle(stream, x.device), sts)
    _abi.check(code)
    return vals, idx, ([s.as_dict() for s in sts] if stats else None)


class Pending:
    """An asynchronous call (topk_async / topk_batched_async).  wait() completes
    it exactly once and returns (values, indices, stats); it keeps the input and
    the outputs alive until then."""

    def __init__(self, handle, x, vals, idx, rows, batched):
        self._h, self._x, self.vals, self.idx, self.rows, self.batched = handle, x, vals, idx, rows, batched

    def wait(self):
        if self._h is None:
            raise RuntimeError("this call was already waited for")
        sts = (ProfkStats * self.rows)()
        code = lib().profk_wait(self._h, sts)
        self._h, self._x = None, None
        _abi.check(code)
        if self.batched:
            return self.vals, self.idx, [s.as_dict() for s in sts]
        return self.vals, self.idx, sts[0].as_dict()

    def __del__(self):
        if getattr(self, "_h", None) is not None:
            lib().profk_wait(self._h, None)


def topk_async(x, k: int, eps: float = 1e-3, seed: int = 0, out=None, stream=None) -> Pending:
    """Asynchronous topk: enqueues the call and returns a Pending; see Pending.wait."""
    torch = _torch()
    _need_cuda_f32(x)
    if x.dim() != 1 or not x.is_contiguous():
        raise ValueError("x must be 1-D and contiguous")
    if out is None:
        vals = torch.empty(k, dtype=torch.float32, device=x.device)
        idx = torch.empty(k, dtype=torch.int64, device=x.device)
    else:
        vals, idx = out
    h = C.c_void_p()
    _abi.check(lib().profk_topk_async(x.data_ptr(), x.numel(), int(k), float(eps), int(seed) & (2**64 - 1),
                                      vals.data_ptr(), idx.data_ptr(), _stream_handle(stream, x.device),
                                      C.byref(h)))
    return Pending(h, x, vals, idx, 1, False)


def topk_batched_async(x, k: int, eps: float = 1e-3, seed: int = 0, out=None, stream=None) -> Pending:
    """Asynchronous topk_batched: enqueues the call and returns a Pending."""
    torch = _torch()
    _need_cuda_f32(x)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    rows, n = x.shape
    if out is None:
        vals = torch.empty((rows, k), dtype=torch.float32, device=x.device)
        idx = torch.empty((rows, k), dtype=torch.int64, device=x.device)
    else:
        vals, idx = out
    h = C.c_void_p()
    _abi.check(lib().profk_topk_batched_async(x.data_ptr(), rows, n, x.stride(0), int(k), float(eps),
                                              int(seed) & (2**64 - 1), vals.data_ptr(), idx.data_ptr(),
                                              _stream_handle(stream, x.device), C.byref(h)))
    return Pending(h, x, vals, idx, rows, True)


def sample(x, S: int, seed: int, row: int = 0, attempt: int = 0, stream=None):
    """Step 1 alone: the sample's indices (int64, draw order) and values."""
    torch = _torch()
    _need_cuda_f32(x)
    sidx = torch.empty(S, dtype=torch.int64, device=x.device)
    svals = torch.empty(S, dtype=torch.float32, device=x.device)
    _abi.check(lib().profk_sample(x.data_ptr(), x.numel(), int(S), int(seed) & (2**64 - 1), int(row),
                                  int(attempt), sidx.data_ptr(), svals.data_ptr(), _stream_handle(stream)))
    return sidx, svals


def threshold(vals, t: int, stream=None):
    """Step 2 alone: the t-th largest of a float32 CUDA tensor, as a 1-element tensor."""
    torch = _torch()
    _need_cuda_f32(vals, "vals")
    out = torch.empty(1, dtype=torch.float32, device=vals.device)
    _abi.check(lib().profk_threshold(vals.data_ptr(), vals.numel(), int(t), out.data_ptr(),
                                     _stream_handle(stream)))
    return out


def filter_pass(x, tau: float, M: int, stream=None):
    """Step 3 alone: (candidate keys[M] as int64 bit patterns, counts[3] = R, R_gt, NaNs)."""
    torch = _torch()
    _need_cuda_f32(x)
    keys = torch.zeros(max(int(M), 1), dtype=torch.int64, device=x.device)
    counts = torch.zeros(3, dtype=torch.int64, device=x.device)
    _abi.check(lib().profk_filter(x.data_ptr(), x.numel(), float(tau), int(M), keys.data_ptr(),
                                  counts.data_ptr(), _stream_handle(stream)))
    return keys[: int(M)], counts


def refine(keys, k: int, x, stream=None):
    """Step 4 alone: exact top-k of candidate keys (profk_filter encoding)."""
    torch = _torch()
    _need_cuda_f32(x)
    vals = torch.empty(k, dtype=torch.float32, device=x.device)
    idx = torch.empty(k, dtype=torch.int64, device=x.device)
    _abi.check(lib().profk_refine(keys.data_ptr(), keys.numel(), int(k), x.data_ptr(), x.numel(),
                                  vals.data_ptr(), idx.data_ptr(), _stream_handle(stream)))
    return vals, idx


def exact(x, k: int, stream=None):
    """Exact top-k without sampling (the fallback)."""
    torch = _torch()
    _need_cuda_f32(x)
    vals = torch.empty(k, dtype=torch.float32, device=x.device)
    idx = torch.empty(k, dtype=torch.int64, device=x.device)
    _abi.check(lib().profk_exact(x.data_ptr(), x.numel(), int(k), vals.data_ptr(), idx.data_ptr(),
                                 _stream_handle(stream)))
    return vals, idx
