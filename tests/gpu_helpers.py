"""Helpers shared by the GPU parity tests."""
import numpy as np

from oracle.topk import same_result


def assert_same(vals, idx, ref_vals, ref_idx, what=""):
    v = vals.detach().cpu().numpy()
    i = idx.detach().cpu().numpy()
    if not same_result(v, i, ref_vals, ref_idx):
        bad = np.flatnonzero((v.view(np.uint32) != np.asarray(ref_vals, np.float32).view(np.uint32))
                             | (i != ref_idx))
        j = int(bad[0]) if bad.size else -1
        raise AssertionError(f"{what}: mismatch at {bad.size} of {v.size} positions; first {j}: "
                             f"gpu ({v[j] if j >= 0 else None}, {i[j] if j >= 0 else None}) vs "
                             f"oracle ({ref_vals[j] if j >= 0 else None}, {ref_idx[j] if j >= 0 else None})")


def decode_keys(keys_i64):
    """profk_filter keys -> (order keys, indices)."""
    u = keys_i64.detach().cpu().numpy().view(np.uint64)
    return (u >> np.uint64(32)).astype(np.uint32), (~(u & np.uint64(0xFFFFFFFF))).astype(np.uint32).astype(np.int64) & 0xFFFFFFFF
