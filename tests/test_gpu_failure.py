"""A bounded device wait that runs out: the failure path of the persistent kernels.

Every grid barrier and look-back of the persistent kernels (the sampler's grid
form, the grid refinement, the buffer sort) is a bounded wait.  With
PROFK_OPT_WAIT_TEST the first grid barrier of one of them waits for one CTA
more than its launch has, a count no CTA completes, with a bound of 4096
polls.  Each CTA's wait then runs out (or sees that another CTA's did), the
CTA leaves without writing, and the kernels after it skip the row.  The call
must return PROFK_ERR_DEVICE_TIMEOUT with its outputs untouched, and the next
call must be exact again.  With attempts enqueued after the first
(PROFK_OPT_SPECULATIVE), the row that reported the error is settled and the
later attempts must leave it, and its error, alone.  Nothing here faults,
traps or hangs the GPU: every wait ends by its own bound.
"""
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from routing import oracle_profk

pytestmark = pytest.mark.gpu

SENTINEL_V, SENTINEL_I = 12345.0, -7


@pytest.mark.parametrize("which,n,k", [("sampler", 1 << 24, 32),       # t = 3: the candidate lists' wait
                                       ("sampler", 1 << 24, 1024),     # t = 9: the passes' grid barriers
                                       ("refine", 1 << 24, 1024), ("sort", 1 << 24, 1 << 15)])
@pytest.mark.parametrize("api", ["sync", "async"])
@pytest.mark.parametrize("spec", [0, 3])
def test_wait_that_runs_out_is_reported(pk, cuda_device, which, n, k, api, spec):
    x = workloads.normal(n, 7, cuda_device)
    vals = torch.full((k,), SENTINEL_V, dtype=torch.float32, device=cuda_device)
    idx = torch.full((k,), SENTINEL_I, dtype=torch.int64, device=cuda_device)
    code = {"sampler": pk.WAIT_TEST_SAMPLER, "refine": pk.WAIT_TEST_REFINE, "sort": pk.WAIT_TEST_SORT}[which]
    pk.set_option(pk.OPT_SPECULATIVE, spec)
    pk.set_option(pk.OPT_WAIT_TEST, code)
    with pytest.raises(pk.ProfkError) as e:
        if api == "sync":
            pk.topk(x, k, 1e-3, 3, out=(vals, idx))
        else:
            pk.topk_async(x, k, 1e-3, 3, out=(vals, idx)).wait()
    assert e.value.code == -5  # PROFK_ERR_DEVICE_TIMEOUT
    torch.cuda.synchronize()
    assert bool((vals == SENTINEL_V).all()) and bool((idx == SENTINEL_I).all()), "outputs were written"
    # The next call is exact again.
    pk.set_option(pk.OPT_WAIT_TEST, pk.WAIT_TEST_OFF)
    v, i, st = pk.topk(x, k, 1e-3, 3)
    ov, oi, ost = oracle_profk(x.cpu().numpy(), k, 1e-3, 3)
    assert_same(v, i, ov, oi, f"after the timed-out {which} call")
    assert st["path"] == ost.path and st["R_first"] == ost.R_first

