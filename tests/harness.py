"""Comparison helpers shared by the oracle pin tests and the GPU parity tests.

The rules they apply:
  * indices: bit-exact, except draws the oracle marks as lying within 1e-6 * total of a leaf
    (or rank) boundary; every mismatch must be such a draw, and mismatches must stay under
    0.01% of all draws;
  * internal sums: within 1e-6 relative (the trees are built to agree exactly);
  * IS weights: within 1e-5 relative;
  * gathered rows, actions, rewards, dones: byte-exact.
"""
from __future__ import annotations

import math

import numpy as np

IDX_MISMATCH_CAP = 1e-4   # 0.01% of draws
SUM_RTOL = 1e-6
W_RTOL = 1e-5


def tree_identity_violations(leaves: np.ndarray, sums: np.ndarray, mins: np.ndarray) -> dict:
    """Count nodes i in [1, n) where S[i] != S[2i] + S[2i+1] or M[i] != min(M[2i], M[2i+1]),
    taking leaves as binary64 sums and empty (0) leaves as +inf mins."""
    n = len(leaves)
    if n < 2:
        return {"sum": 0, "min": 0}
    full_s = np.concatenate([sums.astype(np.float64), leaves.astype(np.float64)])
    leaf_m = np.where(leaves > 0, leaves, np.float32(np.inf)).astype(np.float32)
    full_m = np.concatenate([mins.astype(np.float32), leaf_m])
    i = np.arange(1, n)
    bad_s = full_s[i] != (full_s[2 * i] + full_s[2 * i + 1])
    bad_m = full_m[i] != np.minimum(full_m[2 * i], full_m[2 * i + 1])
    return {"sum": int(bad_s.sum()), "min": int(bad_m.sum())}


def exact_total(leaves: np.ndarray) -> float:
    """The correctly rounded sum of the binary32 leaves (math.fsum)."""
    return math.fsum(float(x) for x in leaves.astype(np.float64))


def compare_indices(got: np.ndarray, want: np.ndarray, near: np.ndarray) -> dict:
    got = np.asarray(got, dtype=np.int64)
    want = np.asarray(want, dtype=np.int64)
    near = np.asarray(near, dtype=bool)
    mism = got != want
    return {
        "draws": int(len(want)),
        "mismatch": int(mism.sum()),
        "unexcused": int((mism & ~near).sum()),
        "near": int(near.sum()),
    }


def assert_indices(got, want, near, what="indices"):
    r = compare_indices(got, want, near)
    assert r["unexcused"] == 0, f"{what}: {r['unexcused']} mismatches away from a boundary: {r}"
    assert r["mismatch"] <= IDX_MISMATCH_CAP * r["draws"] or r["mismatch"] == 0, (
        f"{what}: excused mismatches over 0.01% of draws: {r}")
    return r


def rel_err(a, b) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    denom = np.maximum(np.abs(b), np.finfo(np.float64).tiny)
    return np.abs(a - b) / denom


def assert_sums_close(got, want, what="sums"):
    e = rel_err(got, want)
    assert np.all(e <= SUM_RTOL), f"{what}: max rel err {e.max():.3e}"


def assert_weights_close(got, want, mask=None, what="IS weights"):
    e = rel_err(got, want)
    if mask is not None:
        e = e[mask]
    assert e.size == 0 or np.all(e <= W_RTOL), f"{what}: max rel err {e.max():.3e}"


def f32_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between positive binary32 arrays."""
    ai = np.asarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, dtype=np.float32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)
