"""Pins for the oracle: each check ties it to something other than itself (a hand-worked
example, a closed form, an exact sum, a library routine, brute force or a statistical law), so
that a dropped term, a wrong sign or index or a swapped operand fails one of them."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
from scipy import stats

from tests import harness
from rl_infra_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _buffer(orc, raw, alpha=1.0, capacity=None, d=0, dp=None, mode=0, seed=0, eps=1e-6):
    raw = np.asarray(raw, dtype=np.float32)
    cap = capacity or len(raw)
    o = orc.Oracle(cap, d, dp if dp is not None else d, alpha=alpha, eps=eps, mode=mode,
                   seed=seed, with_ring=False)
    o.add(raw_prio=raw, count=len(raw))
    return o


# -- Philox4x32-10 ------------------------------------------------------------------------

def test_philox_uniform_chi_square(orc):
    u = np.array([orc.uniform53(7, j, c, 0) for c in range(64) for j in range(4096)])
    assert np.all((u >= 0.0) & (u < 1.0))
    # 53-bit construction: u * 2^53 is an integer
    assert np.all(np.floor(u * 2.0**53) == u * 2.0**53)
    counts, _ = np.histogram(u, bins=256, range=(0.0, 1.0))
    p = stats.chisquare(counts).pvalue
    assert p > 1e-4, p
    # the test has power: a 5% density tilt of the same sample is rejected
    tilted = np.clip(u + 0.05 * u * (1 - u), 0, 1 - 1e-12)
    assert stats.chisquare(np.histogram(tilted, bins=256, range=(0, 1))[0]).pvalue < 1e-6


def test_philox_bit_balance_and_avalanche(orc):
    rng = np.random.default_rng(3)
    outs = np.array([orc.philox4x32_10([i, 5, 0, 9], [0xDEAD, 0xBEEF]) for i in range(8192)],
                    dtype=np.uint64)
    bits = ((outs[:, :, None] >> np.arange(32, dtype=np.uint64)) & 1).reshape(-1, 128)
    freq = bits.mean(axis=0)
    sigma = 0.5 / math.sqrt(len(outs))
    assert np.all(np.abs(freq - 0.5) < 5.5 * sigma), np.abs(freq - 0.5).max()
    # flipping any single counter or key bit changes about half of the 128 output bits
    dists = []
    for _ in range(200):
        ctr = rng.integers(0, 2**32, size=4, dtype=np.uint64)
        key = rng.integers(0, 2**32, size=2, dtype=np.uint64)
        base = orc.philox4x32_10(ctr, key)
        for b in range(0, 192, 7):
            c2, k2 = ctr.copy(), key.copy()
            if b < 128:
                c2[b // 32] ^= np.uint64(1 << (b % 32))
            else:
                k2[(b - 128) // 32] ^= np.uint64(1 << ((b - 128) % 32))
            other = orc.philox4x32_10(c2, k2)
            dists.append(sum(bin(int(x) ^ int(y)).count("1") for x, y in zip(base, other)))
    assert abs(np.mean(dists) - 64.0) < 1.0, np.mean(dists)
    assert min(dists) > 30


def test_philox_distinct_streams(orc):
    a = [orc.uniform53(0, j, 0, 0) for j in range(64)]
    b = [orc.uniform53(0, j, 1, 0) for j in range(64)]
    c = [orc.uniform53(0, j, 0, 1) for j in range(64)]
    d = [orc.uniform53(1, j, 0, 0) for j in range(64)]
    for x, y in ((a, b), (a, c), (a, d), (b, c)):
        assert len(set(x) & set(y)) == 0


# -- hand-worked example -------------------------------------------------------------------

def test_golden_hand_descent(orc):
    g = json.load(open(os.path.join(GOLDEN, "descent_hand.json")))
    o = _buffer(orc, g["raw_priorities"], alpha=g["alpha"])
    assert o.total() == g["total"]
    assert o.min() == g["min"]
    s = o.sums()
    for k, v in g["node_sums"].items():
        assert s[int(k)] == v
    for mass, leaf in g["descents"]:
        got, rem = o.descend(mass)
        assert got == leaf, (mass, got, leaf)
        assert 0.0 <= rem < g["raw_priorities"][leaf]
    wtab = dict((i, w) for i, w in g["is_weights"])
    out = o.sample(g["total"], g["beta"], gather=False)
    assert len(set(out["idx"].tolist())) == 8  # one stratum per unit of mass: all leaves hit
    for i, w in zip(out["idx"], out["w"]):
        assert abs(w - wtab[int(i)]) <= 1e-7 * wtab[int(i)]


# -- tree structure ------------------------------------------------------------------------

@pytest.mark.parametrize("cap", [1, 2, 3, 1000, 1 << 16])
def test_tree_root_min_identities(orc, cap):
    g = wl.rng(11, cap)
    raw = g.lognormal(0, 1, size=cap).astype(np.float32)
    o = _buffer(orc, raw, alpha=0.6)
    leaves = o.leaves()
    assert np.all(leaves[cap:] == 0)
    assert o.total() == pytest.approx(harness.exact_total(leaves), rel=1e-12)
    assert o.min() == leaves[:cap].min()
    if o.n > 1:
        v = harness.tree_identity_violations(leaves, o.sums(), o.mins())
        assert v == {"sum": 0, "min": 0}


def test_partial_fill_min_ignores_empty_slots(orc):
    o = orc.Oracle(1000, 0, 0, alpha=1.0, with_ring=False)
    raw = np.linspace(5.0, 2.0, 700).astype(np.float32)
    o.add(raw_prio=raw, count=700)
    assert o.size == 700 and o.cursor == 700
    assert o.min() == np.float32(2.0)
    out = o.sample(4096, 0.4, gather=False)
    assert out["idx"].max() < 700


# -- descent against the linear cumulative scan -------------------------------------------

def test_descent_integer_leaves_every_boundary(orc):
    g = wl.rng(5)
    raw = g.integers(1, 10, size=1 << 10).astype(np.float32)
    o = _buffer(orc, raw, alpha=1.0)
    C = np.cumsum(raw.astype(np.float64))  # exact: small integers
    masses = np.concatenate([C[:-1], np.nextafter(C[:-1], -np.inf),
                             np.nextafter(C[:-1], np.inf), g.uniform(0, C[-1], 2000), [0.0]])
    for m in masses:
        want = int(np.searchsorted(C, m, side="right"))  # first i with C_i > m
        got, _ = o.descend(float(m))
        assert got == want, (m, got, want)


def test_descent_real_leaves_away_from_boundaries(orc):
    g = wl.rng(6)
    raw = g.lognormal(0, 1, size=1 << 12).astype(np.float32)
    o = _buffer(orc, raw, alpha=0.6)
    L = o.leaves()
    C = np.cumsum(L.astype(np.float64))
    T = o.total()
    masses = g.uniform(0, T, 20000)
    checked = 0
    for m in masses:
        want = int(np.searchsorted(C, m, side="right"))
        if abs(C[min(want, len(C) - 1)] - m) < 1e-9 * T or (want > 0 and abs(C[want - 1] - m) < 1e-9 * T):
            continue
        got, _ = o.descend(float(m))
        assert got == want
        checked += 1
    assert checked > 19000


def test_descent_equal_leaves_closed_form(orc):
    n = 1 << 12
    o = _buffer(orc, np.full(n, 0.5, np.float32), alpha=1.0)
    assert o.total() == n * 0.5
    g = wl.rng(8)
    for m in np.concatenate([g.uniform(0, n * 0.5, 5000), np.arange(0, n * 0.5, 0.25)]):
        got, _ = o.descend(float(m))
        assert got == math.floor(m / 0.5)


def test_single_filled_slot_always_chosen(orc):
    o = orc.Oracle(1 << 10, 0, 0, alpha=0.6, with_ring=False)
    o.add(raw_prio=np.array([0.3], np.float32), count=1)
    out = o.sample(512, 0.4, gather=False)
    assert np.all(out["idx"] == 0)
    assert np.all(out["w"] == 1.0)


# -- sampling distribution and stratification -----------------------------------------------

def test_stratified_masses_and_call_counter(orc):
    g = wl.rng(9)
    raw = g.uniform(0.01, 1, 1024).astype(np.float32)
    o = _buffer(orc, raw, alpha=0.6)
    T = o.total()
    B = 256
    a = o.sample(B, 0.4, gather=False)
    b = o.sample(B, 0.4, gather=False)
    seg = T / B
    j = np.arange(B)
    for out in (a, b):
        assert np.all(out["mass"] >= j * seg * (1 - 1e-15))
        assert np.all(out["mass"] < (j + 1) * seg * (1 + 1e-15))
    assert not np.array_equal(a["mass"], b["mass"])
    assert o.sample_calls == 2


def test_chi_square_sample_frequencies(orc):
    w = wl.WORKLOADS["tiny"]
    g = wl.rng(0)
    raw = wl.raw_priorities(g, w.capacity, "uniform")
    o = _buffer(orc, raw, alpha=w.alpha)
    counts = np.zeros(w.capacity)
    for _ in range(1000):
        out = o.sample(1024, w.beta, gather=False)
        counts += np.bincount(out["idx"], minlength=w.capacity)
    p = raw.astype(np.float64) ** w.alpha
    p /= p.sum()
    N = counts.sum()
    assert N == 1024 * 1000
    assert stats.chisquare(counts, N * p).pvalue > 1e-4
    # power: the same counts reject alpha = 0.5 (a plausible wrong exponent)
    q = raw.astype(np.float64) ** 0.5
    q /= q.sum()
    assert stats.chisquare(counts, N * q).pvalue < 1e-10


# -- importance-sampling weights ------------------------------------------------------------

def test_is_weights_against_page_formula(orc):
    g = wl.rng(12)
    cap = 3000
    raw = g.lognormal(0, 1, cap).astype(np.float32)
    o = _buffer(orc, raw, alpha=0.6, capacity=4000)  # partly filled, non power of two
    beta = 0.4
    out = o.sample(2048, beta, gather=False)
    L = o.leaves().astype(np.float64)
    T = harness.exact_total(L)
    n = o.size
    P = L[out["idx"]] / T
    pmin = L[:n].min()
    max_w = (n * pmin / T) ** (-beta)
    want = (n * P) ** (-beta) / max_w
    harness.assert_weights_close(out["w"], want)
    assert np.all(out["w"] <= 1.0)


def test_is_weight_one_at_min_leaf_and_beta_zero(orc):
    o = _buffer(orc, [1.0, 2.0, 2.0, 2.0], alpha=1.0)
    out = o.sample(7, 0.4, gather=False)
    assert out["idx"][0] == 0 and out["w"][0] == 1.0
    out = o.sample(64, 0.0, gather=False)
    assert np.all(out["w"] == 1.0)


# -- priority update ------------------------------------------------------------------------

def _model_update(leaves, max_raw, idx, td, size, alpha, eps):
    """Brute-force sequential model: batch order, last writer wins, NaN -> eps,
    +-Inf -> the running maximum at the start of the call."""
    leaves = leaves.copy()
    start = np.float32(max_raw)
    m = np.float32(max_raw)
    skipped = 0
    for i, t in zip(idx, td):
        if i < 0 or i >= size:
            skipped += 1
            continue
        if np.isnan(t):
            raw = np.float32(eps)
        elif np.isinf(t):
            raw = start
        else:
            raw = np.float32(np.float64(abs(np.float32(t))) + eps)
        leaves[i] = np.float32(np.float64(raw) ** alpha)
        m = max(m, raw)
    return leaves, m, skipped


def test_update_against_sequential_model(orc):
    w = wl.WORKLOADS["tiny"]
    g = wl.rng(21)
    raw = wl.raw_priorities(g, w.capacity, "uniform")
    o = _buffer(orc, raw, alpha=w.alpha)
    for rnd in range(10):
        out = o.sample(w.batch, w.beta, gather=False)
        idx = out["idx"].copy()
        td = wl.td_errors(g, w.batch)
        idx[:4] = idx[4:8]                         # duplicates: later positions must win
        if rnd == 3:
            td[0], td[1], td[2] = np.nan, np.inf, -np.inf
            idx[3] = -1                           # skipped
            idx[5] = w.capacity + 7               # skipped
            td[9] = 40.0                          # raises the running maximum
        want, want_max, want_skip = _model_update(o.leaves(), o.max_raw, idx, td, o.size,
                                                  w.alpha, w.eps)
        assert o.update(idx, td) == want_skip
        got = o.leaves()
        assert np.array_equal(got, want)
        assert o.max_raw == want_max
        assert harness.tree_identity_violations(got, o.sums(), o.mins()) == {"sum": 0, "min": 0}
        assert o.total() == pytest.approx(harness.exact_total(got), rel=1e-12)
        assert o.min() == got[: o.size].min()
    assert o.max_raw == pytest.approx(40.0 + 1e-6)


def test_planted_level_race_is_detected(orc):
    """A rebuild that runs every level at once reads children before they are rewritten (the
    bug the segment-tree post describes).  The harness must flag the tree it produces."""
    g = wl.rng(31)
    n = 1 << 10
    raw = g.uniform(0.01, 1, n).astype(np.float32)
    o = _buffer(orc, raw, alpha=0.6)
    old_s = o.sums()
    idx = g.choice(n, 64, replace=False)
    td = wl.td_errors(g, 64)
    o.update(idx, td)
    new_leaves = o.leaves()
    full_old = np.concatenate([old_s, new_leaves.astype(np.float64)])
    racy = old_s.copy()
    i = np.arange(1, n)
    racy[1:] = full_old[2 * i] + full_old[2 * i + 1]  # all levels from pre-update children
    v = harness.tree_identity_violations(new_leaves, racy, o.mins())
    assert v["sum"] > 0
    with pytest.raises(AssertionError):
        harness.assert_sums_close(racy[1:2], o.sums()[1:2])
        assert np.array_equal(racy, o.sums())


# -- insertion, ring wrap and gather --------------------------------------------------------

def test_add_ring_wrap_and_gather(orc):
    cap, d, dp = 10, 3, 5
    o = orc.Oracle(cap, d, dp, alpha=0.6, eps=1e-6, with_ring=True)
    g = wl.rng(41)
    slots = {}
    cursor = 0
    max_raw = np.float32(1.0)
    for count, with_prio in ((3, True), (4, False), (7, True), (25, False)):
        t = wl.transitions(g, count, wl.Workload("t", cap, d, dp, 4, 0.6, 0.4, 1e-6, 1))
        prio = g.uniform(0.5, 3.0, count).astype(np.float32) if with_prio else None
        o.add(t["states"], t["next_states"], t["actions"], t["rewards"], t["dones"], prio)
        start = max_raw
        for k in range(count):
            s = (cursor + k) % cap
            r = prio[k] if prio is not None else start
            slots[s] = (t["states"][k], t["next_states"][k], t["actions"][k], t["rewards"][k],
                        t["dones"][k], np.float32(np.float64(r) ** 0.6))
            max_raw = max(max_raw, np.float32(r))
        cursor = (cursor + count) % cap
        assert o.cursor == cursor
        assert o.size == min(len(slots), cap)
        assert o.max_raw == max_raw
        L = o.leaves()
        for s, row in slots.items():
            assert L[s] == row[5]
        out = o.sample(64, 0.4)
        for j, i in enumerate(out["idx"]):
            st, nx, a, r, dn, _ = slots[int(i)]
            assert np.array_equal(out["states"][j, :d], st)
            assert np.array_equal(out["next_states"][j, :d], nx)
            assert np.all(out["states"][j, d:] == 0) and np.all(out["next_states"][j, d:] == 0)
            assert out["actions"][j] == a and out["rewards"][j] == r and out["dones"][j] == dn


def test_priority_clamps_on_insert(orc):
    o = orc.Oracle(8, 0, 0, alpha=1.0, eps=1e-3, with_ring=False)
    o.add(raw_prio=np.array([np.nan, np.inf, -2.0, 0.0, 1e-5, 7.0, 2.0, np.inf], np.float32),
          count=8)
    L = o.leaves()
    e = np.float32(1e-3)
    assert L.tolist() == [e, 1.0, e, e, e, 7.0, 2.0, 1.0]
    assert o.max_raw == 7.0


def test_errors(orc):
    with pytest.raises(orc.OracleError):
        orc.Oracle(0, 4)
    with pytest.raises(orc.OracleError):
        orc.Oracle(16, 4, 2)
    o = orc.Oracle(16, 0, 0, with_ring=False)
    with pytest.raises(orc.OracleError):
        o.sample(4, 0.4, gather=False)  # empty


# -- rank-based variant ----------------------------------------------------------------------

def test_rank_order_matches_lexsort(orc):
    g = wl.rng(51)
    raw = wl.raw_priorities(g, 5000, "absnormal")
    raw[100:200] = raw[50]  # ties
    o = _buffer(orc, raw, alpha=0.7, mode=1)
    got = o.rank_order()
    want = np.lexsort((np.arange(5000), -raw.astype(np.float64)))
    assert np.array_equal(got, want)


def test_rank_cdf_against_hurwitz_zeta(orc):
    mpmath = pytest.importorskip("mpmath")
    n, alpha = 1 << 20, 0.7
    o = orc.Oracle(n, 0, 0, alpha=alpha, mode=1, with_ring=False)
    cdf = o.cdf()
    assert cdf[0] == 0.0
    for r in (1, 2, 1000, n):
        exact = float(mpmath.zeta(alpha) - mpmath.zeta(alpha, r + 1))
        assert cdf[r] == pytest.approx(exact, rel=1e-12)
    assert np.all(np.diff(cdf) > 0)


def test_rank_sampling_distribution_and_weights(orc):
    g = wl.rng(52)
    n, alpha, beta = 512, 0.7, 0.5
    raw = wl.raw_priorities(g, n, "absnormal")
    o = _buffer(orc, raw, alpha=alpha, mode=1)
    order = o.rank_order()
    rank_of = np.empty(n, np.int64)
    rank_of[order] = np.arange(1, n + 1)
    counts = np.zeros(n)
    for _ in range(400):
        out = o.sample(1024, beta, gather=False)
        r = rank_of[out["idx"]]
        counts += np.bincount(r - 1, minlength=n)
        # page formula: (n P(r))^-beta / max_w with P(r) = r^-alpha / sum_k k^-alpha
        H = float(np.sum(np.arange(1, n + 1, dtype=np.float64) ** -alpha))
        P = r.astype(np.float64) ** -alpha / H
        max_w = (n * (float(n) ** -alpha / H)) ** (-beta)
        harness.assert_weights_close(out["w"], (n * P) ** (-beta) / max_w)
    P = np.arange(1, n + 1, dtype=np.float64) ** -alpha
    P /= P.sum()
    assert stats.chisquare(counts, counts.sum() * P).pvalue > 1e-4
    Q = np.arange(1, n + 1, dtype=np.float64) ** -0.6
    Q /= Q.sum()
    assert stats.chisquare(counts, counts.sum() * Q).pvalue < 1e-10


def test_rank_update_lww(orc):
    o = _buffer(orc, [1.0, 2.0, 3.0, 4.0], alpha=0.7, mode=1)
    o.update(np.array([2, 2, 0, 9], np.int64), np.array([5.0, -6.0, np.nan, 1.0], np.float32))
    raw = o.raw()
    assert raw[2] == np.float32(6.0 + 1e-6)
    assert raw[0] == np.float32(1e-6)
    assert o.max_raw == np.float32(6.0 + 1e-6)
    assert o.rank_order().tolist() == [2, 3, 1, 0]


# -- uniform mode (the plain replay that prioritized replay replaces) --------------------------

def _uniform(orc, size, capacity=None, seed=0, with_ring=False, d=0):
    o = orc.Oracle(capacity or size, d, d, alpha=0.6, mode=orc.UNIFORM, seed=seed,
                   with_ring=with_ring)
    g = wl.rng(size)
    if with_ring:
        t = wl.transitions(g, size, wl.Workload("u", capacity or size, d, d, 4, 0.6, 0.4, 1e-6, 1))
        o.add(t["states"], t["next_states"], t["actions"], t["rewards"], t["dones"],
              g.uniform(0.1, 5, size).astype(np.float32))
    else:
        o.add(raw_prio=g.uniform(0.1, 5, size).astype(np.float32), count=size)
    return o


def test_uniform_one_draw_per_slot_when_batch_equals_size(orc):
    # each stratum is exactly one slot wide, so draw j must land on slot j whatever u_j is
    for size in (1, 7, 1000, 4096):
        o = _uniform(orc, size, capacity=2 * size)
        for _ in range(3):
            out = o.sample(size, 0.4, gather=False)
            assert np.array_equal(out["idx"], np.arange(size))
            assert np.all(out["w"] == 1.0)


def test_uniform_strata_bounds_and_weights(orc):
    # partly filled ring, B neither divides nor is divided by the filled count
    size, B = 1237, 100
    o = _uniform(orc, size, capacity=5000, seed=3)
    assert o.total() == size and o.min() == 1.0
    j = np.arange(B)
    lo = (j * size) // B                     # first slot of stratum j
    hi = -(-((j + 1) * size) // B)           # one past its last (ceil)
    seen = set()
    for _ in range(50):
        out = o.sample(B, 0.7, gather=False)
        assert np.all(out["idx"] >= lo) and np.all(out["idx"] < hi)
        assert np.all(out["idx"] < size)
        assert np.all(out["w"] == 1.0)
        seen.add(out["idx"].tobytes())
    assert len(seen) == 50                   # every call draws afresh


def test_uniform_chi_square(orc):
    size, B, calls = 3000, 256, 2000
    o = _uniform(orc, size, capacity=4096, seed=5)   # 1096 slots never filled
    counts = np.zeros(4096)
    for _ in range(calls):
        counts += np.bincount(o.sample(B, 0.4, gather=False)["idx"], minlength=4096)
    assert counts[size:].sum() == 0
    N = counts.sum()
    assert N == B * calls
    assert stats.chisquare(counts[:size], np.full(size, N / size)).pvalue > 1e-4
    # stratification: per call, the draws below slot k are the strata that end at or below k,
    # plus at most the one stratum that straddles k, so over all calls the prefix counts stay
    # within [calls * f, calls * (f + 1)], f = floor(k * B / size) -- a bound an unstratified or
    # biased sampler breaks
    k = np.arange(1, size + 1)
    f = (k * B) // size
    prefix = np.cumsum(counts[:size])
    assert np.all(prefix >= calls * f) and np.all(prefix <= calls * (f + 1))


def test_uniform_update_changes_nothing(orc):
    a = _uniform(orc, 500, capacity=512, seed=8)
    b = _uniform(orc, 500, capacity=512, seed=8)
    g = wl.rng(1)
    assert a.update(g.integers(0, 500, 300), g.uniform(0, 100, 300).astype(np.float32)) == 0
    assert a.max_raw == b.max_raw and a.total() == b.total() == 500
    for _ in range(3):
        x, y = a.sample(64, 0.4, gather=False), b.sample(64, 0.4, gather=False)
        assert np.array_equal(x["idx"], y["idx"]) and np.array_equal(x["mass"], y["mass"])


def test_uniform_gather_after_wrap(orc):
    cap, d = 37, 5
    o = orc.Oracle(cap, d, d + 3, alpha=0.6, mode=orc.UNIFORM, seed=2, with_ring=True)
    g = wl.rng(77)
    rows = {}
    cursor = 0
    for count in (20, 30, 11):
        t = wl.transitions(g, count, wl.Workload("u", cap, d, d + 3, 4, 0.6, 0.4, 1e-6, 1))
        o.add(t["states"], t["next_states"], t["actions"], t["rewards"], t["dones"])
        for k in range(count):
            rows[(cursor + k) % cap] = (t["states"][k], t["next_states"][k], t["actions"][k],
                                        t["rewards"][k], t["dones"][k])
        cursor = (cursor + count) % cap
    assert o.size == cap
    out = o.sample(cap, 0.4)
    assert np.array_equal(out["idx"], np.arange(cap))
    for j in range(cap):
        st, nx, a, r, dn = rows[j]
        assert np.array_equal(out["states"][j, :d], st) and np.all(out["states"][j, d:] == 0)
        assert np.array_equal(out["next_states"][j, :d], nx) and np.all(out["next_states"][j, d:] == 0)
        assert out["actions"][j] == a and out["rewards"][j] == r and out["dones"][j] == dn


# -- flat mode: cumulative array + binary search, no tree ---------------------------------------

def _twins(orc, raw, capacity=None, alpha=0.6, seed=0):
    """The same buffer twice: proportional (tree descent) and flat (scan + search)."""
    out = []
    for mode in (orc.PROPORTIONAL, orc.FLAT):
        o = orc.Oracle(capacity or len(raw), 0, 0, alpha=alpha, mode=mode, seed=seed, with_ring=False)
        o.add(raw_prio=np.asarray(raw, np.float32), count=len(raw))
        out.append(o)
    return out


def test_flat_equals_tree_on_exact_sums(orc):
    # integer leaves (alpha = 1): every prefix and every node sum is exact, so the tree's descent
    # and the flat search must pick the same leaf for every mass, with the same weights
    g = wl.rng(31)
    raw = g.integers(1, 50, 3000).astype(np.float32)
    tree, flat = _twins(orc, raw, capacity=4096, alpha=1.0, seed=4)
    assert flat.total() == tree.total() == float(raw.astype(np.float64).sum())
    assert flat.min() == tree.min() == raw.min()
    for B in (1, 7, 512, 3000, 6001):
        a, b = tree.sample(B, 0.4, gather=False), flat.sample(B, 0.4, gather=False)
        assert np.array_equal(a["mass"], b["mass"])
        assert np.array_equal(a["idx"], b["idx"])
        assert np.array_equal(a["w"], b["w"])


def test_flat_search_against_numpy_cumsum(orc):
    # real leaves: the flat oracle's index is numpy's sequential cumsum + searchsorted(right)
    g = wl.rng(32)
    raw = g.lognormal(0, 2, 5000).astype(np.float32)
    (flat,) = _twins(orc, raw, capacity=5000)[1:]
    C = np.cumsum(flat.leaves()[:5000].astype(np.float64))
    assert flat.total() == C[-1]
    for _ in range(4):
        out = flat.sample(777, 0.5, gather=False)
        want = np.minimum(np.searchsorted(C, out["mass"], side="right"), 4999)
        assert np.array_equal(out["idx"], want)
        below = np.where(want > 0, C[np.maximum(want - 1, 0)], 0.0)
        assert np.array_equal(out["rem"], out["mass"] - below)


def test_flat_matches_tree_away_from_boundaries(orc):
    # real leaves: the scan and the tree round differently, so only draws the oracle marks as
    # near a boundary may differ
    g = wl.rng(33)
    raw = g.lognormal(0, 1, 1 << 14).astype(np.float32)
    tree, flat = _twins(orc, raw, seed=9)
    diff = near = 0
    for _ in range(20):
        a, b = tree.sample(1024, 0.4, gather=False), flat.sample(1024, 0.4, gather=False)
        d = a["idx"] != b["idx"]
        assert np.all(b["near"][d] | a["near"][d])
        diff += int(d.sum())
        near += int(b["near"].sum())
    assert diff <= 2   # 20480 draws


def test_flat_chi_square_and_updates(orc):
    w = wl.WORKLOADS["tiny"]
    g = wl.rng(34)
    raw = wl.raw_priorities(g, w.capacity, "uniform")
    tree, flat = _twins(orc, raw, alpha=w.alpha)
    idx = g.integers(0, w.capacity, 300)
    idx[:50] = idx[50:100]
    td = wl.td_errors(g, 300)
    td[5] = np.nan
    assert tree.update(idx, td) == flat.update(idx, td) == 0
    assert np.array_equal(tree.leaves(), flat.leaves()) and tree.max_raw == flat.max_raw
    L = flat.leaves()[: w.capacity].astype(np.float64)
    counts = np.zeros(w.capacity)
    for _ in range(500):
        counts += np.bincount(flat.sample(1024, w.beta, gather=False)["idx"], minlength=w.capacity)
    N = counts.sum()
    assert stats.chisquare(counts, N * L / L.sum()).pvalue > 1e-4
    q = L ** (0.5 / w.alpha)
    assert stats.chisquare(counts, N * q / q.sum()).pvalue < 1e-10
    out = flat.sample(2048, 0.7, gather=False)
    want = (L[out["idx"]] / L.min()) ** -0.7
    harness.assert_weights_close(out["w"], want)


def test_flat_search_every_boundary(orc):
    # integer leaves: the prefix sums are exact, so a mass equal to C[i] goes to leaf i + 1 (the
    # strict ">"), one ulp below it stays on leaf i, and the leftover is exact
    g = wl.rng(35)
    raw = g.integers(1, 9, 200).astype(np.float32)
    tree, flat = _twins(orc, raw, capacity=256, alpha=1.0)
    C = np.cumsum(raw.astype(np.float64))
    for i in range(len(raw) - 1):
        for m, want in ((C[i], i + 1), (np.nextafter(C[i], -np.inf), i), (np.nextafter(C[i], np.inf), i + 1)):
            leaf, rem = flat.descend(m)
            assert leaf == want and rem == m - (C[want - 1] if want else 0.0)
            assert tree.descend(m) == (leaf, rem)
    assert flat.descend(C[-1])[0] == len(raw)      # past the end: the sampler clamps it (R7)
