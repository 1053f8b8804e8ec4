"""Exact top-k: the plain definition, written out.

Problem statement (Prof-K paper, Section 3 "Problem Setup and Algorithm
Overview"): given x in R^N and k >= 1, return the k largest entries of x with
their indices; batched inputs are handled row by row.

Order used everywhere (the pages assume distinct values, Section 4 "Notation and
Conventions", and are silent on ties; the reading taken here):

* values descending under IEEE-754 comparison, so -0.0 == +0.0 and +-inf are
  ordinary values;
* equal values ordered by ascending index;
* NaN is rejected (ValueError).

The returned values keep their original bit patterns (a -0.0 stays -0.0).
"""
from __future__ import annotations

import numpy as np


def _check(x: np.ndarray, k: int) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype != np.float32 or x.ndim != 1:
        raise TypeError("x must be a 1-D float32 array")
    n = x.shape[0]
    if not (1 <= k <= n):
        raise ValueError(f"need 1 <= k <= n, got k={k}, n={n}")
    if np.isnan(x).any():
        raise ValueError("NaN in input")
    return x


def topk_sort(x: np.ndarray, k: int):
    """Definition: full sort of (value desc, index asc), keep the first k.

    ``np.lexsort`` sorts by its last key first: -x ascending (float64, exact
    for float32 input, -0.0 == +0.0), then the index ascending.
    """
    x = _check(x, k)
    n = x.shape[0]
    order = np.lexsort((np.arange(n, dtype=np.int64), -x.astype(np.float64)))
    sel = order[:k].astype(np.int64)
    return x[sel].copy(), sel


def topk_partition(x: np.ndarray, k: int):
    """The same definition, reached in O(N) for inputs too large to sort.

    Let v_k be the k-th largest value (a selection, ``np.partition``).  Under
    the order above, the top-k set is every element strictly greater than v_k
    plus the lowest-index elements equal to v_k, as many as are needed to make
    k.  Those k elements are then sorted by the same rule as ``topk_sort``.
    Tests pin this against ``topk_sort`` on inputs with ties, +-0 and +-inf.
    """
    x = _check(x, k)
    n = x.shape[0]
    vk = np.partition(x, n - k)[n - k]
    gt = np.flatnonzero(x > vk)
    eq = np.flatnonzero(x == vk)[: k - gt.size]
    sel = np.concatenate([gt, eq]).astype(np.int64)
    order = np.lexsort((sel, -x[sel].astype(np.float64)))
    sel = sel[order]
    return x[sel].copy(), sel


def topk_chunked(x: np.ndarray, k: int, workers: int, chunks: int | None = None):
    """The same definition on several host threads, for timing the CPU on large inputs.

    The row is cut into contiguous chunks; each chunk's top-min(k, len) is
    taken by ``topk_partition`` in a thread pool (numpy's selection and sorts
    release the GIL), with the chunk's offset added to its indices; the top k
    of those candidates, by ``topk_sort``'s rule, is the row's top k.  Exact
    because an element among the row's k largest (in the order above) is
    among its own chunk's k largest: every element ahead of it in its chunk is
    also ahead of it in the row.  Tests pin this against ``topk_sort``.
    """
    from concurrent.futures import ThreadPoolExecutor

    x = _check(x, k)
    n = x.shape[0]
    chunks = max(1, min(n, chunks if chunks else workers))
    bounds = [(n * c // chunks, n * (c + 1) // chunks) for c in range(chunks)]

    def one(b):
        lo, hi = b
        v, i = topk_partition(x[lo:hi], min(k, hi - lo))
        return v, i + lo

    with ThreadPoolExecutor(max_workers=max(1, workers)) as ex:
        parts = list(ex.map(one, bounds))
    cv = np.concatenate([p[0] for p in parts])
    ci = np.concatenate([p[1] for p in parts])
    order = np.lexsort((ci, -cv.astype(np.float64)))[:k]
    return cv[order].copy(), ci[order]


def topk_rows(x2d: np.ndarray, k: int, method=topk_sort):
    """Batched rows: the definition applied to each row; indices are per row."""
    x2d = np.asarray(x2d)
    vals = np.empty((x2d.shape[0], k), dtype=np.float32)
    idx = np.empty((x2d.shape[0], k), dtype=np.int64)
    for r in range(x2d.shape[0]):
        vals[r], idx[r] = method(np.ascontiguousarray(x2d[r]), k)
    return vals, idx


def same_result(v1, i1, v2, i2) -> bool:
    """Bit-exact equality of two (values, indices) results, order included."""
    v1 = np.asarray(v1, dtype=np.float32)
    v2 = np.asarray(v2, dtype=np.float32)
    return (v1.shape == v2.shape
            and np.array_equal(v1.view(np.uint32), v2.view(np.uint32))
            and np.array_equal(np.asarray(i1, dtype=np.int64), np.asarray(i2, dtype=np.int64)))
