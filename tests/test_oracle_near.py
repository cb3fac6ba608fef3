"""Pins for the oracle's near-boundary flag: the rule that decides which GPU/oracle index
mismatches the parity bar excuses ("Putting prioritized replay's segment tree on a GPU", The
Race Condition Worth Writing Down: a bit-for-bit oracle; the 1e-6 * total rule of the parity
bar).

The flag of a draw says that its mass m lies within 1e-6 * T of an end of the chosen slot's
extent [C(i-1), C(i)), or that the walk fell off the end.  Here the expected flag is computed a
different way: from the cumulative sums (numpy cumsum, exact on integer leaves) the chosen slot
is `searchsorted(C, m, side="right")`, and the flag is whether the distance from m to the
nearest of ALL boundaries {0, C(0), ..., C(s-1)} is below 1e-6 * T, with T the exact total
(math.fsum) -- no descent, no leftover mass, no per-mode code.  Masses are placed on every
boundary, one ulp either side, 0.5e-6 T and 2e-6 T either side, at the midpoints of the extents
and past the end, in every mode (tree, flat, uniform, rank).

The last test builds copies of the oracle with one known mistake planted in the rule (an
absolute tolerance, a fall-off not counted, the upper distance taken against the next leaf, the
upper end not tested) and checks that these pins reject each of them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

from rl_infra_gb300 import workloads as wl

REL_TOL = 1e-6


def _expected(C: np.ndarray, s: int, T: float, m: float):
    """Slot and flag from the cumulative sums C (inclusive, length s) by the nearest-boundary
    distance."""
    i = int(np.searchsorted(C, m, side="right"))
    if i >= s:
        return s - 1, True
    bounds = np.concatenate([[0.0], C])
    return i, bool(np.min(np.abs(bounds - m)) < REL_TOL * T)


def _masses(C: np.ndarray, T: float, picks) -> list:
    tol = REL_TOL * T
    out = [0.0, T / 2]
    prev = 0.0
    for i in picks:
        c = float(C[i])
        out += [c, np.nextafter(c, -np.inf), np.nextafter(c, np.inf), c - 0.5 * tol, c + 0.5 * tol,
                c - 2 * tol, c + 2 * tol, (prev + c) / 2]
        prev = c
    out += [np.nextafter(T, -np.inf), T, T + 0.5 * tol, T + 5 * tol]
    return [m for m in out if m >= 0.0]


def _check(o, C, s, T, masses, rank_order=None):
    """Mismatches between the oracle's locate step and the independent expectation."""
    bad = []
    for m in masses:
        want_i, want_near = _expected(C, s, T, m)
        slot, _, near = o.locate(m)
        want_slot = int(rank_order[want_i]) if rank_order is not None else want_i
        if slot != want_slot or near != want_near:
            bad.append((float(m), slot, near, want_slot, want_near))
    return bad


def _int_leaves(g, n):
    """Integer leaves (exact sums): mostly 1..1000, a few of 10^6, some runs of ones."""
    v = g.integers(1, 1000, n).astype(np.float64)
    v[g.choice(n, max(1, n // 16), replace=False)] = 1e6
    v[n // 3: n // 3 + 5] = 1.0
    return v.astype(np.float32)


def _tree_case(orc, plant, capacity, fill, seed):
    g = wl.rng(seed, 1)
    raw = _int_leaves(g, fill)
    raw[-1] = 1e6                         # a wide last extent, so a fall-off is not near by distance
    o = orc.Oracle(capacity, 0, 0, alpha=1.0, eps=1e-6, mode=orc.PROPORTIONAL, with_ring=False, plant=plant)
    o.add(raw_prio=raw, count=fill)
    L = o.leaves()[:fill].astype(np.float64)
    assert np.array_equal(L, raw.astype(np.float64))     # alpha = 1: the leaves are the raw values
    C = np.cumsum(L)
    T = math.fsum(L)
    assert C[-1] == T and o.total() == T
    picks = sorted(set(range(0, fill, max(1, fill // 40))) | {fill - 2, fill - 1, fill // 3, fill // 3 + 2})
    bad = _check(o, C, fill, T, _masses(C, T, picks))
    o.close()
    return bad


def _flat_case(orc, plant, fill, seed):
    g = wl.rng(seed, 2)
    raw = _int_leaves(g, fill)
    o = orc.Oracle(fill + 7, 0, 0, alpha=1.0, eps=1e-6, mode=orc.FLAT, with_ring=False, plant=plant)
    o.add(raw_prio=raw, count=fill)
    L = raw.astype(np.float64)
    C = np.cumsum(L)
    T = math.fsum(L)
    picks = sorted(set(range(0, fill, max(1, fill // 40))) | {fill - 1})
    bad = _check(o, C, fill, T, _masses(C, T, picks))
    o.close()
    return bad


def _uniform_case(orc, plant, fill):
    o = orc.Oracle(fill + 3, 0, 0, alpha=0.6, eps=1e-6, mode=orc.UNIFORM, with_ring=False, plant=plant)
    o.add(raw_prio=np.ones(fill, np.float32), count=fill)
    C = np.arange(1, fill + 1, dtype=np.float64)
    T = float(fill)
    picks = sorted(set(range(0, fill, max(1, fill // 40))) | {fill - 1})
    masses = _masses(C, T, picks) + [T + 0.5, T + 0.25]   # past the end, mid-slot: not near by distance
    bad = _check(o, C, fill, T, masses)
    o.close()
    return bad


def _rank_case(orc, plant, fill, alpha, seed):
    g = wl.rng(seed, 3)
    raw = (g.integers(1, 50, fill)).astype(np.float32)   # ties: order by slot within a key
    o = orc.Oracle(fill, 0, 0, alpha=alpha, eps=1e-6, mode=orc.RANK, with_ring=False, plant=plant)
    o.add(raw_prio=raw, count=fill)
    order = np.lexsort((np.arange(fill), -raw.astype(np.float64)))
    cdf = o.cdf()
    C = cdf[1:fill + 1]
    T = float(cdf[fill])
    picks = sorted(set(range(0, fill, max(1, fill // 40))) | {fill - 1})
    bad = _check(o, C, fill, T, _masses(C, T, picks), rank_order=order)
    o.close()
    return bad


def _all_cases(orc, plant=0) -> dict:
    return {
        "tree 64/64": _tree_case(orc, plant, 64, 64, 1),
        "tree 50/64 (fall-off into padding)": _tree_case(orc, plant, 50, 50, 2),
        "tree 1000/700": _tree_case(orc, plant, 1000, 700, 3),
        "flat 300": _flat_case(orc, plant, 300, 4),
        "uniform 1000": _uniform_case(orc, plant, 1000),
        "uniform 37": _uniform_case(orc, plant, 37),
        "rank 500 alpha 0.7": _rank_case(orc, plant, 500, 0.7, 5),
        "rank 64 alpha 0": _rank_case(orc, plant, 64, 0.0, 6),
    }


def test_near_flag_at_placed_masses(orc):
    bad = {k: v for k, v in _all_cases(orc).items() if v}
    assert not bad, bad


def test_sampled_near_flags_match_the_distance_rule(orc):
    """The flags orc_sample returns, on its own drawn masses, against the same independent rule,
    in every mode; the leaves are chosen so that both flagged and unflagged draws occur."""
    for mode in (orc.PROPORTIONAL, orc.FLAT, orc.UNIFORM, orc.RANK):
        g = wl.rng(11, mode)
        fill = 3000
        raw = _int_leaves(g, fill)
        o = orc.Oracle(4096, 0, 0, alpha=1.0 if mode != orc.RANK else 0.6, eps=1e-6, mode=mode,
                       with_ring=False, seed=mode)
        o.add(raw_prio=raw, count=fill)
        if mode in (orc.PROPORTIONAL, orc.FLAT):
            C, order = np.cumsum(raw.astype(np.float64)), None
        elif mode == orc.UNIFORM:
            C, order = np.arange(1, fill + 1, dtype=np.float64), None
        else:
            C, order = o.cdf()[1:fill + 1], np.lexsort((np.arange(fill), -raw.astype(np.float64)))
        T = float(C[-1])
        flags = []
        for _ in range(4):
            s = o.sample(1000, 0.4, gather=False)
            for j in range(1000):
                i, near = _expected(C, fill, T, s["mass"][j])
                want = int(order[i]) if order is not None else i
                assert s["idx"][j] == want and bool(s["near"][j]) == near, (mode, j, s["mass"][j])
                flags.append(near)
        assert 0 < sum(flags) < len(flags), (mode, sum(flags))
        o.close()


@pytest.mark.parametrize("plant,what", [(1, "absolute tolerance 1e-6"), (2, "fall-off not counted"),
                                        (3, "upper distance against the next leaf"),
                                        (4, "upper end not tested")])
def test_planted_mistakes_in_the_rule_are_caught(orc, plant, what):
    bad = {k: v for k, v in _all_cases(orc, plant).items() if v}
    assert bad, f"a planted mistake ({what}) passed every near-boundary pin"
