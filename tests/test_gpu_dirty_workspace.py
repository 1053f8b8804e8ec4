"""Calls on a workspace that holds anything, against the oracle.

The library allocates its workspace from the stream-ordered pool (or takes
the caller's buffer) and never clears it as a whole: every step must set up,
before it reads them, the counters, flags and control words it uses.  Here
each configuration runs on a caller-owned workspace filled first with ones
and then with random bytes; the results, paths and attempts must be the
oracle procedure's.  The configurations reach the sampler forms (one grid
launch with t <= 8 and with t > 8, the per-chunk lists, the step-by-step
form), the tie exit, the radix refinement of large k, batched rows, redraws
left to the device, a redraw before the exact fallback, and the fallback with
no attempt at all.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import assert_same
from routing import oracle_profk

pytestmark = pytest.mark.gpu

# name: (generator, rows, n, k, eps, options, oracle keywords)
CONFIGS = {
    "grid_t_small": ("normal", 1, 1 << 22, 32, 1e-3, {}, {}),
    "grid_t_large": ("normal", 1, 1 << 22, 4096, 1e-3, {}, {}),
    "tie_exit": ("levels16", 1, 1 << 22, 4096, 1e-3, {}, {}),
    "radix_refine": ("normal", 1, 1 << 22, 40000, 1e-3, {}, {}),
    "lists_rows": ("normal", 24, 1 << 18, 64, 1e-3, {"sampler": 3}, {}),
    "steps": ("uniform", 1, 1 << 22, 100, 1e-3, {"sampler": 2}, {}),
    "speculative": ("normal", 3, 1 << 20, 1000, 1e-3, {"spec": 3, "S": 2048, "t": 1}, {"force": {"S": 2048, "t": 1}}),
    "redraw_then_fallback": ("normal", 2, 1 << 20, 500, 1e-3, {"max_attempts": 1, "S": 4096, "t": 4096, "M": 600},
                             {"force": {"S": 4096, "t": 4096, "M": 600}, "max_attempts": 1}),
    "no_attempt": ("sorted_normal", 4, 1 << 20, 3000, 0.5, {"max_attempts": 0}, {"max_attempts": 0}),
}


def set_options(pk, o):
    pk.set_option(pk.OPT_SAMPLER, o.get("sampler", 0))
    pk.set_option(pk.OPT_SPECULATIVE, o.get("spec", 0))
    pk.set_option(pk.OPT_MAX_ATTEMPTS, o.get("max_attempts", 6))
    pk.set_option(pk.OPT_FORCE_S, o.get("S", 0))
    pk.set_option(pk.OPT_FORCE_T, o.get("t", 0))
    pk.set_option(pk.OPT_FORCE_M, o.get("M", 0))


@pytest.mark.parametrize("fill", ["ones", "random"])
@pytest.mark.parametrize("name", list(CONFIGS))
def test_dirty_workspace(pk, cuda_device, name, fill):
    gen, rows, n, k, eps, opts, okw = CONFIGS[name]
    x = workloads.GENERATORS[gen](rows * n, 41, cuda_device).view(rows, n)
    need = pk.workspace_size(rows, n, k, eps)
    if fill == "ones":
        buf = torch.full((need,), 0xFF, dtype=torch.uint8, device=cuda_device)
    else:
        g = torch.Generator(device=cuda_device).manual_seed(7)
        buf = torch.randint(0, 256, (need,), dtype=torch.uint8, device=cuda_device, generator=g)
    set_options(pk, opts)
    pk.set_workspace(buf)
    try:
        if rows == 1:
            v, i, st = pk.topk(x[0], k, eps, 5)
            v, i, sts = v[None], i[None], [st]
        else:
            v, i, sts = pk.topk_batched(x, k, eps, 5)
    finally:
        pk.set_workspace(None)
    h = x.cpu().numpy()
    for r in range(rows):
        if rows == 1:
            ov, oi, ost = oracle_profk(h[0], k, eps, 5, **okw)
        else:
            ov, oi, ost = oracle_profk(np.ascontiguousarray(h[r]), k, eps / rows, 5, row=r, rows=rows, **okw)
        assert_same(v[r], i[r], ov, oi, f"{name} {fill} row {r}")
        assert (sts[r]["path"], sts[r]["attempts"], sts[r]["R_first"]) == (ost.path, ost.attempts, ost.R_first), \
            (name, fill, r, sts[r])
