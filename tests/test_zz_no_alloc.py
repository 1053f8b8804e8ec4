"""profk_topk_noalloc, the entry point that allocates nothing.

Some callers cannot allocate on the call path: a latency-bounded serving loop
(an allocation can synchronize or stall the device), a plugin whose host owns
all device memory through its own allocator, a process whose pool already holds
nearly all of the GPU.  profk_topk_noalloc serves them from a fixed scratch
array reserved when the library loads.  This test calls it through the C-ABI,
twice in a row per problem (the second call finds the first call's leftovers in
the shared scratch), and requires the same bit-exact result as profk_topk.

Kept in a file that pytest collects last, so that a failure here cannot stop a
run before the other tests; it also passes when run alone in a fresh process.
"""
import ctypes as C

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

SCRATCH_ERR = -6


def noalloc_fn(pk):
    fn = pk.lib().profk_topk_noalloc
    fn.restype = C.c_int
    fn.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_double, C.c_uint64, C.c_void_p, C.c_void_p,
                   C.c_void_p, C.POINTER(pk.ProfkStats)]
    return fn


def call_noalloc(pk, fn, x, k, eps, seed):
    vals = torch.empty(k, dtype=torch.float32, device=x.device)
    idx = torch.empty(k, dtype=torch.int64, device=x.device)
    st = pk.ProfkStats()
    code = fn(x.data_ptr(), x.numel(), k, eps, seed, vals.data_ptr(), idx.data_ptr(),
              torch.cuda.current_stream().cuda_stream, C.byref(st))
    torch.cuda.synchronize()
    return code, vals, idx, st


@pytest.mark.parametrize("gen,n,k", [("normal", 1 << 24, 1024), ("uniform", (1 << 22) + 3, 32),
                                     ("levels16", 1 << 22, 100), ("normal", 1 << 16, 64)])
def test_noalloc_matches_profk_topk_twice(pk, cuda_device, gen, n, k):
    fn = noalloc_fn(pk)
    x = workloads.GENERATORS[gen](n, 3, cuda_device)
    ref_v, ref_i, ref_st = pk.topk(x, k, 1e-3, 17)
    torch.cuda.synchronize()
    for call in range(2):
        code, v, i, st = call_noalloc(pk, fn, x, k, 1e-3, 17)
        assert code == 0, code
        assert torch.equal(v.view(torch.int32), ref_v.view(torch.int32)), f"values differ on call {call}"
        assert torch.equal(i, ref_i), f"indices differ on call {call}"
        assert (st.path, st.attempts, st.R_first) == (ref_st["path"], ref_st["attempts"], ref_st["R_first"])
        assert st.aux_bytes == 0


def test_noalloc_rejects_problems_beyond_its_scratch(pk, cuda_device):
    fn = noalloc_fn(pk)
    n = 1 << 23  # k = n takes the exact path and needs 8 * 2^23 = 64 MiB of sort keys
    x = workloads.normal(n, 4, cuda_device)
    code, _, _, _ = call_noalloc(pk, fn, x, n, 1e-3, 1)
    assert code == SCRATCH_ERR
    assert b"scratch" in pk.lib().profk_strerror(SCRATCH_ERR)
