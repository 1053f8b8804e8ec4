"""Seeded synthetic inputs for Prof-K (shared by tests, smoke and bench).

This module only generates data; it holds none of the method's arithmetic, so
both the CUDA path and the CPU oracle can be fed from it.  Every generator
takes a seed and a device; on CUDA the values come from PyTorch's
counter-based Philox generator, on the CPU from PyTorch's CPU generator (the
two differ; each run compares the GPU result and the oracle on the same
tensor).

Shapes and distributions follow the workloads of "Prof-K: Probabilistic
One-Pass Filtering for Efficient Top-k Selection" (Section 5 and Appendix E:
standard-normal float32 vectors; uniform and heavy-tailed inputs; inputs whose
values share leading bits; batched rows; the BatchTopK SAE selection), at the
sizes listed in ``CONFIGS``.
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def uniform(n: int, seed: int, device="cuda") -> torch.Tensor:
    """i.i.d. Uniform[0, 1) float32."""
    return torch.rand(n, generator=_gen(seed, device), device=device, dtype=torch.float32)


def normal(n: int, seed: int, device="cuda") -> torch.Tensor:
    """i.i.d. standard normal float32."""
    return torch.randn(n, generator=_gen(seed, device), device=device, dtype=torch.float32)


def pareto(n: int, seed: int, device="cuda", alpha: float = 1.5, xm: float = 1.0) -> torch.Tensor:
    """Pareto(alpha, x_m) by inversion, x = x_m (1 - u)^(-1/alpha); heavy-tailed."""
    u = uniform(n, seed, device)
    return xm * torch.pow(1.0 - u, -1.0 / alpha)


def ulps_below_one(n: int, seed: int, device="cuda", frac: float = 0.999) -> torch.Tensor:
    """Tie stress (a): with probability `frac` a value uniform over the 256 float32
    ulps just below 1.0 (bits 0x3F7FFF00 .. 0x3F7FFFFF), else Uniform[0, 1)."""
    g = _gen(seed, device)
    pick = torch.rand(n, generator=g, device=device) < frac
    bits = 0x3F7FFF00 + torch.randint(0, 256, (n,), generator=g, device=device, dtype=torch.int32)
    u = torch.rand(n, generator=g, device=device, dtype=torch.float32)
    return torch.where(pick, bits.view(torch.float32), u)


def levels16(n: int, seed: int, device="cuda") -> torch.Tensor:
    """Tie stress (b): values from 16 levels j/16, j = 0..15, equally likely."""
    j = torch.randint(0, 16, (n,), generator=_gen(seed, device), device=device, dtype=torch.int32)
    return j.to(torch.float32) / 16.0


def sorted_normal(n: int, seed: int, device="cuda") -> torch.Tensor:
    """Tie stress (c): the standard-normal input sorted ascending."""
    return torch.sort(normal(n, seed, device)).values


def distinct_shuffled(n: int, seed: int, device="cuda") -> torch.Tensor:
    """A random permutation of 0..n-1 as float32 (all values distinct, n <= 2^24)."""
    if n > (1 << 24):
        raise ValueError("n <= 2^24 keeps every value exact in float32")
    return torch.randperm(n, generator=_gen(seed, device), device=device).to(torch.float32)


def normal_rows(rows: int, n: int, seed: int, device="cuda") -> torch.Tensor:
    """Batched rows of i.i.d. standard normals, shape (rows, n)."""
    return torch.randn(rows, n, generator=_gen(seed, device), device=device, dtype=torch.float32)


def sae_preacts(seed: int, device="cuda", batch: int = 4096, d_in: int = 512, d_dict: int = 12288) -> torch.Tensor:
    """BatchTopK SAE selection input: ReLU(X W + b) flattened.

    X ~ N(0, 1) of shape batch x d_in, W ~ N(0, 1/d_in) of shape d_in x d_dict,
    b ~ N(0, 0.01) (variance; std 0.1).  Computed in float32 without TF32.
    4096 x 12288 = 50,331,648 values, about half of them exactly zero.
    """
    g = _gen(seed, device)
    X = torch.randn(batch, d_in, generator=g, device=device, dtype=torch.float32)
    W = torch.randn(d_in, d_dict, generator=g, device=device, dtype=torch.float32) * math.sqrt(1.0 / d_in)
    b = torch.randn(d_dict, generator=g, device=device, dtype=torch.float32) * 0.1
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        pre = torch.relu(X @ W + b)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return pre.reshape(-1).contiguous()


GENERATORS = {
    "uniform": uniform,
    "normal": normal,
    "pareto": pareto,
    "ulps_below_one": ulps_below_one,
    "levels16": levels16,
    "sorted_normal": sorted_normal,
}

# The benchmark workloads: name -> (generator, n, list of k, eps).
CONFIGS = {
    "uniform_2^22": ("uniform", 1 << 22, [32], 1e-3),
    "normal_2^26": ("normal", 1 << 26, [32, 1024, 32768], 1e-3),
    "uniform_2^30": ("uniform", 1 << 30, [32, 1024, 1 << 19], 1e-3),
    "normal_2^30": ("normal", 1 << 30, [32, 1024, 1 << 19], 1e-3),
    "pareto_2^30": ("pareto", 1 << 30, [32, 1024, 1 << 19], 1e-3),
    "ulps_below_one_2^28": ("ulps_below_one", 1 << 28, [4096], 1e-3),
    "levels16_2^28": ("levels16", 1 << 28, [4096], 1e-3),
    "sorted_normal_2^28": ("sorted_normal", 1 << 28, [4096], 1e-3),
}
