"""GPU parity: libgbper (through the C ABI) against the oracle, element by element, on the
same seeded inputs.  Indices bit-exact except oracle-marked boundary draws (< 0.01%), sums
within 1e-6 relative (built to be bit-identical), IS weights within 1e-5 relative, gathered
fields byte-exact."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines skip this module
    pytest.skip("no CUDA device", allow_module_level=True)

from rl_infra_gb300 import capi  # noqa: E402
from rl_infra_gb300 import workloads as wl  # noqa: E402
from tests import harness  # noqa: E402
from tests.gpu_helpers import Pair, dev, prefill  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rl_infra_gb300 import build
    build.build()
    capi.load()


# the update's three paths, each forced through per_config: climb from the changed leaves,
# scatter + rebuild every level, or propagate entry by entry
CLIMB = dict(rebuild_batch=capi.REBUILD_NEVER, element_batch=capi.ELEMENT_NEVER)
REBUILD = dict(rebuild_batch=1, element_batch=capi.ELEMENT_NEVER)
ELEMENT = dict(rebuild_batch=capi.REBUILD_NEVER, element_batch=capi.ELEMENT_ALWAYS)
DEFAULT = dict()
PATH_IDS = ["climb", "rebuild", "element"]


def _small(name, **kw):
    w = wl.WORKLOADS[name]
    return wl.Workload(**{**w.__dict__, **kw})


# -- the small workload, end to end --------------------------------------------------------

def test_tiny_workload_rounds():
    w = wl.WORKLOADS["tiny"]
    g = wl.rng(0)
    p = Pair(w.capacity, w.state_dim, w.row_stride, w.alpha, w.eps, w.mode, seed=0)
    prefill(p, w, g)
    p.check_tree()
    p.check_counters()
    for _ in range(w.rounds):
        _, want = p.sample(w.batch, w.beta)
        p.update(want["idx"], wl.td_errors(g, w.batch))
        p.check_tree()
        p.check_counters()
    assert p.gpu.status_device() == 0
    p.close()


@pytest.mark.parametrize("capacity,count", [(1, 1), (2, 2), (3, 3), (1000, 700), (4096, 4096),
                                            (5000, 3000), (1 << 14, 1 << 14)])
def test_partial_and_ragged_fills(capacity, count):
    w = _small("tiny", capacity=capacity)
    g = wl.rng(1, capacity)
    p = Pair(capacity, 8, 8, 0.6, 1e-6, 0, seed=3)
    prefill(p, w, g, count=count, chunk=max(1, count // 3))
    p.check_tree()
    p.check_counters()
    for B in (1, 7, 32, 2 * count + 5):
        _, want = p.sample(B, 0.4)
        assert np.all(want["idx"] < count)
        p.update(want["idx"], wl.td_errors(g, B))
        p.check_tree()
    p.check_counters()
    p.close()


def test_ring_wrap_and_oversized_insert():
    cap = 3000
    w = _small("tiny", capacity=cap, state_dim=5, row_stride=7)
    g = wl.rng(2)
    p = Pair(cap, 5, 7, 0.6, 1e-6, 0, seed=4)
    for count, with_prio in ((1000, True), (1500, False), (1200, True), (7001, True), (1, False),
                             (2999, False), (3000, True), (250, True)):
        rows = wl.transitions(g, count, w)
        prio = wl.raw_priorities(g, count, "lognormal") if with_prio else None
        p.add(rows, prio)
        p.check_tree()
        p.check_counters()
        _, want = p.sample(64, 0.5)
        p.update(want["idx"], wl.td_errors(g, 64))
    assert np.array_equal(p.gpu.read_state(capi.PER_STATE_STATES).reshape(cap, 5),
                          p.orc.ring_states())
    p.close()


@pytest.mark.parametrize("d,dp", [(0, 0), (0, 1), (0, 4), (1, 1), (3, 8), (8, 8), (48, 64), (64, 64), (63, 65)])
def test_gather_row_shapes(d, dp):
    cap = 4096
    w = _small("tiny", capacity=cap, state_dim=d, row_stride=dp)
    g = wl.rng(3, d * 100 + dp)
    p = Pair(cap, d, dp, 0.6, 1e-6, 0, seed=5)
    prefill(p, w, g)
    for B in (1, 33, 1000):
        _, want = p.sample(B, 0.4)
        p.update(want["idx"], wl.td_errors(g, B))
    p.check_tree()
    p.close()


@pytest.mark.parametrize("rb", [CLIMB, REBUILD, ELEMENT], ids=PATH_IDS)
def test_update_duplicates_nan_inf_and_bad_indices(rb):
    cap = 1 << 12
    w = _small("tiny", capacity=cap)
    g = wl.rng(4)
    p = Pair(cap, 8, 8, 0.7, 1e-6, 0, seed=6, **rb)
    prefill(p, w, g, count=cap - 100)
    for rnd in range(6):
        _, want = p.sample(512, 0.5)
        idx = wl.duplicate_positions(g, want["idx"], 0.25)
        td = wl.td_errors(g, 512)
        if rnd == 2:
            td[:5] = [np.nan, np.inf, -np.inf, 0.0, -0.0]
            td[7] = 1e30
        if rnd == 3:
            idx[10] = -5
            idx[11] = cap - 50          # an unfilled slot: skipped
            idx[12] = 1 << 40
        p.update(idx, td)
        p.check_tree()
        p.check_counters()
        flags = p.gpu.status_device()
        assert flags == (capi.PER_DEVFLAG_BAD_INDEX if rnd == 3 else 0)
    p.close()


@pytest.mark.parametrize("rb", [CLIMB, REBUILD], ids=PATH_IDS[:2])
def test_update_all_in_one_subtree_overflow_path(rb):
    """More entries than one CTA sorts at once land in one subtree: the chunked path (or, with
    the rebuild path, thousands of entries racing for a few hundred winner words)."""
    cap = 1 << 16
    w = _small("tiny", capacity=cap)
    g = wl.rng(5)
    p = Pair(cap, 8, 8, 0.6, 1e-6, 0, seed=7, **rb)
    prefill(p, w, g)
    for B in (4096, 20000):
        idx = g.integers(0, 300, size=B).astype(np.int64)   # all inside the first subtree
        p.update(idx, wl.td_errors(g, B))
        p.check_tree()
        p.check_counters()
    _, want = p.sample(1024, 0.4)
    p.close()


@pytest.mark.parametrize("mode", [0, 1])
def test_large_batch_climb(mode):
    """Batches of 4096 entries and more on the climb path (CTAs of 16 warps, lists of 128):
    duplicates, bad indices, NaN/Inf, and one subtree holding more entries than its list."""
    cap = 1 << 17
    w = _small("tiny", capacity=cap, state_dim=4, row_stride=4, mode=mode)
    g = wl.rng(13, mode)
    p = Pair(cap, 4, 4, 0.6, 1e-6, mode, seed=3, **CLIMB)
    prefill(p, w, g)
    for rnd in range(4):
        B = (4096, 8192, 20000, 5000)[rnd]
        idx = g.integers(0, cap, B).astype(np.int64)
        idx = wl.duplicate_positions(g, idx, 0.25)
        td = wl.td_errors(g, B)
        if rnd == 1:
            idx[:3] = [-1, cap + 7, 1 << 40]
            td[5:8] = [np.nan, np.inf, -np.inf]
        if rnd == 2:
            idx[:3000] = g.integers(0, 200, 3000)   # one subtree: more than its list holds
        p.update(idx, td)
        p.check_tree()
        p.check_counters()
        assert p.gpu.status_device() == (capi.PER_DEVFLAG_BAD_INDEX if rnd == 1 else 0)
        _, want = p.sample(1024, 0.4, check_rows=False)
    p.close()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("size", [1 << 16, 5000, 3])
def test_climb_crowded_and_partly_filled(mode, size):
    """The climb path on a full ring and on rings holding 5000 or 3 of 2^16 slots (the subtrees
    then split only the filled part; the spine above it is rebuilt), with batches that give one
    subtree (2^0, 2^3, 2^6, 2^9 and 2^10 of them) 33 to 600 entries, more than one warp's group
    of 32 and more than its list, packed into 256 or 1024 slots (also spanning a whole aligned
    block of 1024) or spread over 8192."""
    cap = 1 << 16
    w = _small("tiny", capacity=cap, state_dim=4, row_stride=4, mode=mode)
    g = wl.rng(21, 10 * mode + (size % 7))
    p = Pair(cap, 4, 4, 0.6, 1e-6, mode, seed=5, **CLIMB)
    prefill(p, w, g, count=size)
    for B in (5, 40, 300, 600, 2100, 5000):
        for crowd in ("none", "dense", "spread", "ends"):
            idx = g.integers(0, size, B).astype(np.int64)
            width = {"none": 0, "dense": 256, "spread": 8192, "ends": 1024}[crowd]
            if width:
                # most entries in one stretch of `width` slots
                width = min(width, size)
                lo = int(g.integers(0, size - width + 1))
                k = (9 * B) // 10
                idx[:k] = lo + g.integers(0, width, k)
                if crowd == "ends" and B - k >= 2:
                    blk = (lo // width) * width   # both ends of an aligned block
                    idx[k:k + 2] = [blk, min(blk + width, size) - 1]
            idx = wl.duplicate_positions(g, idx, 0.2) if B > 4 else idx
            p.update(idx, wl.td_errors(g, B))
            p.check_tree()
            p.check_counters()
            assert p.gpu.status_device() == 0
        p.sample(int(min(B, 512)), 0.4, check_rows=False)
        if mode == 1:
            _assert_rank_order(p)
    p.close()


def test_update_dispatch_follows_lasting_crowding():
    """With the default dispatch, updates whose entries keep crowding a few slots first climb
    over finer and finer subtree splits (2^6 up to 2^10 subtrees), then switch to the level
    rebuild when even the finest split is crowded, and return to the climb (and to coarser
    splits) once the draws spread; the trees match the oracle after every round, whatever the
    path.  Crowding: every slot prefilled at priority 1e-6, each round inserts 64 rows at the
    running maximum (they hold nearly all the mass), samples 512 and updates them with TD errors
    of order 1e-3.  Spread: one large update gives every slot a priority of order 1, then rounds
    insert rows at such priorities."""
    cap = 1 << 16                     # 2^16 leaves: the finest split has 64-leaf subtrees
    w = _small("tiny", capacity=cap, state_dim=4, row_stride=4)
    g = wl.rng(31, 1)
    p = Pair(cap, 4, 4, 0.6, 1e-6, 0, seed=8)
    rows = wl.transitions(g, cap, w)
    p.add(rows, np.full(cap, 1e-6, np.float32))
    rebuild_at = 32 * 2
    reports = []
    for rnd in range(12):
        p.add(wl.transitions(g, 64, w), None)
        _, want = p.sample(512, 0.4, check_rows=False)
        p.update(want["idx"], (wl.td_errors(g, 512) * 1e-3).astype(np.float32))
        p.check_tree()
        c = p.counters()["crowd"]
        reports.append((c >> 28, c & 0xFFFFF))
    assert any(P == 6 and n > 32 for P, n in reports), reports          # crowded at the size split
    assert any(P == 10 and n >= rebuild_at for P, n in reports), reports  # still crowded at the finest
    idx = np.arange(cap, dtype=np.int64)
    p.update(idx, np.abs(wl.td_errors(g, cap)) + 0.5)   # a size-chosen rebuild: every slot near 1
    p.check_tree()
    for rnd in range(12):
        p.add(wl.transitions(g, 512, w), (np.abs(wl.td_errors(g, 512)) + 0.5).astype(np.float32))
        _, want = p.sample(512, 0.4, check_rows=False)
        p.update(want["idx"], np.abs(wl.td_errors(g, 512)) + 0.5)
        p.check_tree()
        c = p.counters()["crowd"]
        reports.append((c >> 28, c & 0xFFFFF))
    assert reports[-1][1] <= 32 and reports[-1][0] < 10, reports          # spread: climbing, coarser
    p.check_counters()
    assert p.gpu.status_device() == 0
    p.close()


def test_equal_priorities_and_beta_zero():
    cap = 1 << 12
    w = _small("tiny", capacity=cap)
    g = wl.rng(6)
    p = Pair(cap, 8, 8, 1.0, 1e-6, 0, seed=8)
    rows = wl.transitions(g, cap, w)
    p.add(rows, np.full(cap, 0.5, np.float32))
    got, want = p.sample(cap, 0.0)
    assert np.all(got["w"].cpu().numpy() == 1.0)
    got, want = p.sample(cap, 0.7)
    gi = got["idx"].cpu().numpy()
    assert np.array_equal(np.sort(gi), np.arange(cap))  # one draw per leaf
    p.close()


@pytest.mark.parametrize("rb", [DEFAULT, CLIMB, REBUILD, ELEMENT], ids=["default"] + PATH_IDS)
def test_many_sizes_of_batch_and_tree(rb):
    for D in (0, 1, 4, 5, 6, 9, 10, 11, 15, 16, 17):
        cap = 1 << D
        w = _small("tiny", capacity=cap, state_dim=4, row_stride=4)
        g = wl.rng(7, D)
        p = Pair(cap, 4, 4, 0.6, 1e-6, 0, seed=D, **rb)
        prefill(p, w, g)
        for B in (1, 31, 32, 33, 257, 2049):
            _, want = p.sample(B, 0.4)
            p.update(want["idx"], wl.td_errors(g, B))
        p.check_tree()
        p.check_counters()
        p.close()


@pytest.mark.parametrize("D,cap", [(0, 1), (3, 5), (6, 64), (10, 1000), (12, 1 << 12), (13, 5000),
                                   (15, 20000), (16, 40000), (18, 1 << 18)])
def test_large_batches_two_draws_per_warp(D, cap):
    """Batches of 4096 draws or more walk on 16-lane halves (8-lane quarters from 8192) of a warp
    in rounds of up to 6 levels (for trees whose round count that keeps), below a top of 8 levels
    walked in shared memory on trees deeper than 12; odd batch sizes leave sub-warps without a
    draw."""
    w = _small("tiny", capacity=cap, state_dim=64, row_stride=64)
    g = wl.rng(17, D)
    p = Pair(cap, 64, 64, 0.7, 1e-6, 0, seed=D)
    prefill(p, w, g)
    for B in (4096, 5001, 8192, 8195):
        _, want = p.sample(B, 0.5)
        idx = wl.duplicate_positions(g, want["idx"], 0.25)
        p.update(idx, wl.td_errors(g, B))
    p.check_tree()
    p.check_counters()
    p.close()


@pytest.mark.parametrize("D,cap", [(22, 1 << 22), (23, (1 << 22) + 5)])
def test_large_batches_top_levels_in_shared_memory(D, cap):
    """Batches of 4096 draws or more (16-lane halves or 8-lane quarters of a warp) on trees of
    2^22 leaves and up: the top 8 levels are walked from a copy in shared memory, the middle
    rounds from left children and the last round from its leaves alone, the nodes above them
    rebuilt by pairwise sums; the second tree is barely half filled, so its right half holds
    empty subtrees."""
    w = _small("tiny", capacity=cap, state_dim=4, row_stride=4)
    g = wl.rng(19, D)
    p = Pair(cap, 4, 4, 0.7, 1e-6, 0, seed=D)
    prefill(p, w, g, chunk=1 << 18)
    for B in (8192, 6000, 8195, 12000):
        _, want = p.sample(B, 0.5)
        idx = wl.duplicate_positions(g, want["idx"], 0.25)
        p.update(idx, wl.td_errors(g, B))
    p.check_tree()
    p.check_counters()
    p.close()


@pytest.mark.parametrize("alpha", [0.6, 0.5, 1.5, 0.123456789])
def test_leaf_values_over_a_wide_range(alpha):
    """Leaves p^alpha for priorities spread over 2^-30 .. 2^30 (and exact powers of two),
    through the insert path and the update path, bit-identical to the oracle's."""
    cap = 1 << 20
    g = wl.rng(14, int(alpha * 1000))
    p = Pair(cap, 0, 0, alpha, 1e-9, 0, seed=1, with_ring=True)
    raw = np.exp2(g.uniform(-30, 30, cap)).astype(np.float32)
    raw[::97] = np.float32(2.0) ** g.integers(-20, 20, len(raw[::97])).astype(np.float32)
    z = np.zeros(cap, np.uint32)
    rows = {"states": np.zeros((cap, 0), np.float32), "next_states": np.zeros((cap, 0), np.float32),
            "actions": z, "rewards": z.view(np.float32), "dones": z.astype(np.uint8)}
    for lo in range(0, cap, 1 << 18):
        p.add({k: v[lo: lo + (1 << 18)] for k, v in rows.items()}, raw[lo: lo + (1 << 18)])
    p.check_tree()
    idx = g.integers(0, cap, 8192).astype(np.int64)
    td = (np.exp2(g.uniform(-20, 20, 8192)) * g.choice([-1, 1], 8192)).astype(np.float32)
    p.update(idx, td)
    p.check_tree()
    p.close()


# -- rank-based variant ---------------------------------------------------------------------

@pytest.mark.parametrize("rb", [CLIMB, REBUILD], ids=PATH_IDS[:2])
@pytest.mark.parametrize("cap,fill", [(1, 1), (100, 37), (4095, 4095), (4096, 4096), (4097, 4097),
                                      (100000, 65536)])
def test_rank_small(cap, fill, rb):
    w = _small("rank", capacity=cap, state_dim=6, row_stride=8)
    g = wl.rng(8, cap)
    p = Pair(cap, 6, 8, 0.7, 1e-6, 1, seed=9, **rb)
    prefill(p, w, g, count=fill, chunk=max(1, fill // 2))
    cdf = p.gpu.read_state(capi.PER_STATE_CDF)
    harness.assert_sums_close(cdf[1:], p.orc.cdf()[1:], what="rank CDF")
    for rnd in range(3):
        _, want = p.sample(min(1024, 4 * fill + 1), 0.5)
        idx = want["idx"].copy()
        td = wl.td_errors(g, len(idx))
        if rnd == 1:
            idx[: len(idx) // 4] = idx[len(idx) // 4: 2 * (len(idx) // 4)]
        p.update(idx, td)
        p.check_tree()
        p.check_counters()
    p.close()


def _assert_rank_order(p):
    got = p.gpu.read_state(capi.PER_STATE_RANK_ORDER)
    want = p.orc.rank_order()
    assert got.shape == want.shape
    assert np.array_equal(got, want), f"rank order differs at {np.flatnonzero(got != want)[:8]}"


@pytest.mark.parametrize("alpha", [0.0, 1.0, 1.5])
def test_rank_guide_across_alphas(alpha):
    """The rank sampler's guide buckets at other exponents: at alpha 0 every bucket spans two
    ranks' mass; at 1.5 the bucket count is capped, so the sparse end's buckets hold more than
    three candidate ranks and the sampler searches them.  Draws, weights and rows match the
    oracle, partly filled and full."""
    cap = 50000
    w = _small("rank", capacity=cap, state_dim=4, row_stride=4)
    g = wl.rng(31, int(alpha * 10))
    p = Pair(cap, 4, 4, alpha, 1e-6, 1, seed=13)
    prefill(p, w, g, count=30000, chunk=30000)
    for rnd in range(4):
        if rnd == 2:
            prefill(p, w, g, count=cap - 30000, chunk=cap - 30000)
        _, want = p.sample(1024, 0.5)
        p.update(want["idx"], wl.td_errors(g, 1024))
        p.check_tree()
    p.check_counters()
    p.close()


@pytest.mark.parametrize("cap,fill,flags", [(50000, 50000, 0), (30000, 20000, 0),
                                            (30000, 20000, capi.PER_FLAG_RANK_RESORT)])
def test_rank_order_kept_between_samples(cap, fill, flags):
    """The slot order after each sample equals the oracle's full sort, whether it was merged
    from the previous order (a few written slots) or sorted again (many): updates with repeated
    indices and equal priorities, ring inserts that overwrite slots or grow the filled range,
    and one large update that forces a full sort."""
    w = _small("rank", capacity=cap, state_dim=2, row_stride=4)
    g = wl.rng(21, cap)
    p = Pair(cap, 2, 4, 0.7, 1e-6, 1, seed=12, flags=flags)
    prefill(p, w, g, count=fill, chunk=fill)
    p.sample(512, 0.5)
    _assert_rank_order(p)
    for rnd in range(10):
        size = int(p.orc.size)
        idx = g.integers(0, size, 600)
        idx[:150] = idx[150:300]                      # repeated indices: the last writer wins
        td = wl.td_errors(g, len(idx))
        td[300:340] = 0.25                            # equal priorities: ties by slot
        if rnd == 6:
            idx = g.integers(0, size, size // 4)      # more than an eighth: sorted again
            td = wl.td_errors(g, len(idx))
        p.update(idx, td)
        if rnd % 3 == 1:
            rows = wl.transitions(g, 300, w)
            p.add(rows, wl.raw_priorities(g, 300, w.prio))
        p.sample(512, 0.5)
        _assert_rank_order(p)
    p.check_counters()
    assert p.gpu.status_device() == 0
    p.close()


def test_rank_refresh_then_sample():
    """per_rank_refresh brings the order up to date on its own (merge after few writes, sort
    after many); the sample that follows uses it as it is, and both match the oracle."""
    cap = 40000
    w = _small("rank", capacity=cap, state_dim=2, row_stride=4)
    g = wl.rng(23, cap)
    p = Pair(cap, 2, 4, 0.7, 1e-6, 1, seed=5)
    prefill(p, w, g, count=cap, chunk=cap)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for rnd in range(6):
        n_upd = 700 if rnd != 3 else cap // 4
        idx = g.integers(0, cap, n_upd)
        p.update(idx, wl.td_errors(g, n_upd))
        assert capi.per_rank_refresh(p.gpu._h, st) == capi.PER_OK
        torch.cuda.synchronize()
        got = p.gpu.read_state(capi.PER_STATE_RANK_ORDER).astype(np.int64)
        assert np.array_equal(got, p.orc.rank_order().astype(np.int64)), rnd
        assert capi.per_rank_refresh(p.gpu._h, st) == capi.PER_OK   # nothing written since: no change
        p.sample(1024, 0.5)
        _assert_rank_order(p)
    assert p.gpu.status_device() == 0
    p.close()
    q = capi.ReplayBuffer(64, 2)
    assert capi.per_rank_refresh(q._h, st) == capi.PER_ERR_INVALID_ARG   # proportional mode
    q.close()


@pytest.mark.parametrize("seed", [3, 17, 31])
def test_rank_order_random_operations(seed):
    """Seeded random rank-mode histories (inserts of every size, some wrapping or larger than the
    ring, updates with repeats, NaN/Inf and equal priorities): after every sample the kept order
    is the oracle's full order."""
    g = wl.rng(seed, 5)
    cap = int(g.integers(2000, 30000))
    w = _small("rank", capacity=cap, state_dim=2, row_stride=2)
    p = Pair(cap, 2, 2, 0.7, 1e-6, 1, seed=seed)
    prefill(p, w, g, count=int(g.integers(1, cap)), chunk=cap)
    for rnd in range(12):
        op = g.random()
        if op < 0.4:
            count = int(g.integers(1, 3000)) if g.random() < 0.8 else int(g.integers(cap, 2 * cap))
            p.add(wl.transitions(g, count, w), wl.raw_priorities(g, count, w.prio) if g.random() < 0.7 else None)
        else:
            size = int(p.orc.size)
            B = int(g.integers(1, 3000))
            idx = g.integers(0, size, B)
            if B > 4:
                idx = wl.duplicate_positions(g, idx, 0.3)
            td = wl.td_errors(g, B)
            if B > 10:
                td[:3] = [np.nan, np.inf, 0.0]
                td[3:8] = 0.5
            p.update(idx, td)
        p.sample(int(g.integers(1, 1025)), 0.5, check_rows=False)
        _assert_rank_order(p)
    p.check_counters()
    assert p.gpu.status_device() == 0
    p.close()


@pytest.mark.slow
def test_rank_more_than_a_million_slots():
    """3M slots: more than 256 sort tiles, so the look-back reads group totals in rounds."""
    cap = 3_000_000
    w = _small("rank", capacity=cap, state_dim=2, row_stride=4)
    g = wl.rng(15)
    p = Pair(cap, 2, 4, 0.7, 1e-6, 1, seed=11)
    prefill(p, w, g, chunk=1 << 20)
    for _ in range(2):
        _, want = p.sample(2048, 0.5)
        p.update(want["idx"], wl.td_errors(g, 2048))
    p.check_tree()
    p.check_counters()
    p.close()


def test_rank_ties_keep_slot_order():
    cap = 9000
    w = _small("rank", capacity=cap, state_dim=4, row_stride=4)
    g = wl.rng(9)
    p = Pair(cap, 4, 4, 0.7, 1e-6, 1, seed=10)
    rows = wl.transitions(g, cap, w)
    prio = np.repeat(np.array([0.5, 2.0, 1.0], np.float32), cap // 3)
    p.add(rows, prio)
    for _ in range(3):
        p.sample(1024, 0.5)
    p.close()


# -- CUDA graphs: a captured round replays with the device-resident counters -------------------

# -- uniform mode and float dones -------------------------------------------------------------

@pytest.mark.parametrize("cap,fill", [(1, 1), (3, 2), (1000, 999), (4096, 4096), (5000, 3001),
                                      (1 << 16, 1 << 16)])
def test_uniform_mode(cap, fill):
    w = _small("tiny", capacity=cap, state_dim=6, row_stride=8, mode=capi.PER_MODE_UNIFORM)
    g = wl.rng(21, cap)
    p = Pair(cap, 6, 8, 0.6, 1e-6, capi.PER_MODE_UNIFORM, seed=9)
    prefill(p, w, g, count=fill, chunk=max(1, fill // 2))
    p.check_tree()
    p.check_counters()
    for B in (1, 5, 64, 100, 1024, fill, 3 * fill + 1):
        _, want = p.sample(B, 0.4)
        assert np.all(want["idx"] < fill)
        assert p.update(want["idx"], wl.td_errors(g, B)) == 0
        p.check_counters()
    assert p.stats["mismatch"] == 0, p.stats          # the division has no boundary slack
    assert p.gpu.status_device() == 0
    p.close()


def test_uniform_mode_wrap_and_update_no_op():
    cap = 2000
    w = _small("tiny", capacity=cap, state_dim=4, row_stride=4, mode=capi.PER_MODE_UNIFORM)
    g = wl.rng(22)
    p = Pair(cap, 4, 4, 0.6, 1e-6, capi.PER_MODE_UNIFORM, seed=2)
    for count in (700, 1800, 5003, 1):
        p.add(wl.transitions(g, count, w), wl.raw_priorities(g, count, "lognormal"))
        p.check_counters()
        _, want = p.sample(256, 0.4)
        p.update(want["idx"], wl.td_errors(g, 256))
    # updates with out-of-range indices change nothing and raise no device flag in this mode
    p.update(np.array([-1, cap + 5, 3], np.int64), np.ones(3, np.float32))
    assert p.gpu.status_device() == 0
    assert np.array_equal(p.gpu.read_state(capi.PER_STATE_STATES).reshape(cap, 4), p.orc.ring_states())
    with pytest.raises(capi.PerError):
        p.gpu.min()
    p.close()


# -- flat mode: the pages' own cumulative array + search ----------------------------------------

FLAT = capi.PER_MODE_FLAT


@pytest.mark.parametrize("cap,fill", [(1, 1), (3, 2), (2047, 2047), (2048, 2048), (2049, 2049),
                                      (5000, 3001), (1 << 16, 1 << 16), (100000, 70001)])
def test_flat_mode(cap, fill):
    w = _small("tiny", capacity=cap, state_dim=6, row_stride=8, mode=FLAT)
    g = wl.rng(24, cap)
    p = Pair(cap, 6, 8, 0.6, 1e-6, FLAT, seed=11)
    prefill(p, w, g, count=fill, chunk=max(1, fill // 3))
    p.check_tree()
    p.check_counters()
    for B in (1, 7, 512, 3 * fill + 1):
        _, want = p.sample(B, 0.4)
        idx = wl.duplicate_positions(g, want["idx"], 0.25) if B > 4 else want["idx"]
        td = wl.td_errors(g, B)
        td[:1] = np.nan
        p.update(idx, td)
        p.check_tree()
        p.check_counters()
    assert p.stats["mismatch"] <= max(1, p.stats["draws"] // 10000), p.stats
    assert p.gpu.status_device() == 0
    p.close()


def test_flat_mode_wrap_bad_indices_and_gather():
    cap = 3000
    w = _small("tiny", capacity=cap, state_dim=5, row_stride=7, mode=FLAT)
    g = wl.rng(25)
    p = Pair(cap, 5, 7, 0.6, 1e-6, FLAT, seed=4)
    for count, with_prio in ((1000, True), (1500, False), (7001, True), (1, False), (3000, True)):
        rows = wl.transitions(g, count, w)
        p.add(rows, wl.raw_priorities(g, count, "lognormal") if with_prio else None)
        p.check_tree()
        p.check_counters()
        _, want = p.sample(256, 0.5)
        p.update(want["idx"], wl.td_errors(g, 256))
    p.update(np.array([-1, cap + 5, 3], np.int64), np.ones(3, np.float32))
    assert p.gpu.status_device() == capi.PER_DEVFLAG_BAD_INDEX
    p.check_tree()
    p.close()


def test_flat_mode_wide_range_and_equal_leaves():
    """Leaves over 2^-30 .. 2^30 (the fixed-point sums must stay as close to the exact prefix as
    binary64 summation) and a run of equal leaves (exact sums: every boundary is exact)."""
    cap = 1 << 15
    g = wl.rng(27)
    p = Pair(cap, 0, 0, 1.0, 1e-30, FLAT, seed=2, with_ring=False)
    raw = np.exp2(g.uniform(-30, 30, cap)).astype(np.float32)
    p.gpu.add(None, None, dev(np.zeros(cap, np.uint32)), dev(np.zeros(cap, np.float32)),
              dev(np.zeros(cap, np.uint8)), dev(raw))
    p.orc.add(raw_prio=raw, count=cap)
    p.check_tree()
    for _ in range(4):
        p.sample(4096, 0.4, check_rows=False)
    assert p.stats["mismatch"] <= max(1, p.stats["draws"] // 10000), p.stats
    p.close()
    q = Pair(4096, 0, 0, 1.0, 1e-6, FLAT, seed=3, with_ring=False)
    ones = np.full(4096, 0.75, np.float32)
    q.gpu.add(None, None, dev(np.zeros(4096, np.uint32)), dev(np.zeros(4096, np.float32)),
              dev(np.zeros(4096, np.uint8)), dev(ones))
    q.orc.add(raw_prio=ones, count=4096)
    assert np.array_equal(q.gpu.read_state(capi.PER_STATE_CUMULATIVE) if q.gpu.total() else None,
                          np.arange(1, 4097) * 0.75)
    for B in (4096, 1000):
        got, want = q.sample(B, 0.4, check_rows=False)
        assert q.stats["mismatch"] == 0
    q.close()


def test_flat_mode_over_a_thousand_tiles():
    """More than 1024 tiles of 2048 leaves, a ragged last tile, and the reduce pass's last CTA
    scanning more than 4 tile sums per thread."""
    cap = (1 << 21) + 4099
    g = wl.rng(28)
    p = Pair(cap, 0, 0, 0.6, 1e-6, FLAT, seed=5, with_ring=False)
    raw = wl.raw_priorities(g, cap, "lognormal")
    p.gpu.add(None, None, dev(np.zeros(cap, np.uint32)), dev(np.zeros(cap, np.float32)),
              dev(np.zeros(cap, np.uint8)), dev(raw))
    p.orc.add(raw_prio=raw, count=cap)
    for _ in range(3):
        _, want = p.sample(2048, 0.4, check_rows=False)
        p.update(want["idx"], wl.td_errors(g, 2048))
    p.check_tree()
    assert p.stats["mismatch"] <= max(1, p.stats["draws"] // 10000), p.stats
    p.close()


@pytest.mark.slow
def test_flat_apex_size_rounds():
    """2^21 slots, B = 512, ingest 4096 per round, the apex shapes, in flat mode."""
    w = _small("apex", mode=FLAT)
    g = wl.rng(26)
    p = Pair(w.capacity, w.state_dim, w.row_stride, w.alpha, w.eps, FLAT, seed=0, with_ring=True)
    prefill(p, w, g, chunk=1 << 18)
    for rnd in range(4):
        rows = wl.transitions(g, w.ingest, w)
        p.add(rows, None)
        _, want = p.sample(w.batch, w.beta, check_rows=(rnd == 3))
        p.update(want["idx"], wl.td_errors(g, w.batch))
    p.check_tree()
    p.check_counters()
    assert p.stats["mismatch"] <= max(1, p.stats["draws"] // 10000), p.stats
    p.close()


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_float_dones(mode):
    cap = 3000
    w = _small("tiny", capacity=cap, state_dim=8, row_stride=8, mode=mode)
    g = wl.rng(23, mode)
    p = Pair(cap, 8, 8, 0.6, 1e-6, mode, seed=4, flags=capi.PER_FLAG_DONES_F32)
    prefill(p, w, g, count=cap, chunk=cap)
    for B in (1, 77, 512):
        got, want = p.sample(B, 0.4)
        assert got["dones"].dtype == torch.float32
        d = got["dones"].cpu().numpy()
        assert set(np.unique(d)) <= {0.0, 1.0}
        assert d.sum() > 0 or B < 512
        p.update(want["idx"], wl.td_errors(g, B))
    p.close()


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_graph_replayed_rounds(mode):
    """Insert + sample + update captured once per staging offset as CUDA graphs and replayed:
    every replay inserts at the device cursor, draws a fresh batch (device call counter) and, in
    rank mode, merges into whichever buffer holds the order -- each replay's batch and the final
    state equal the oracle stepping the same rounds."""
    cap, d, dp, B, I, NO = 4096, 8, 8, 64, 256, 3
    w = _small("tiny", capacity=cap, state_dim=d, row_stride=dp, mode=mode)
    g = wl.rng(31, mode)
    p = Pair(cap, d, dp, 0.6, 1e-6, mode, seed=5)
    prefill(p, w, g, count=cap, chunk=cap)
    _, want = p.sample(B, 0.5)                       # rank mode: the first order, sorted eagerly
    p.update(want["idx"], wl.td_errors(g, B))
    L, h = capi.load(), p.gpu._h
    rows = [wl.transitions(g, I, w) for _ in range(NO)]
    dev_rows = [{k: dev(v) for k, v in r.items()} for r in rows]
    idx_sets = [g.integers(0, cap, B).astype(np.int64) for _ in range(NO)]
    td_sets = [wl.td_errors(g, B) for _ in range(NO)]
    d_idx = [dev(x) for x in idx_sets]
    d_td = [dev(x) for x in td_sets]
    out = p.gpu.alloc_batch(B)
    optr = [out[k].data_ptr() for k in ("idx", "w", "states", "next_states", "actions", "rewards", "dones")]
    graphs = []
    for o in range(NO):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            r = dev_rows[o]
            assert L.per_add(h, I, r["states"].data_ptr(), r["next_states"].data_ptr(), r["actions"].data_ptr(),
                             r["rewards"].data_ptr(), r["dones"].data_ptr(), None, cs) == 0
            assert L.per_sample(h, B, ctypes.c_float(0.5), *optr, cs) == 0
            assert L.per_update_priorities(h, B, d_idx[o].data_ptr(), d_td[o].data_ptr(), cs) == 0
        graphs.append(gr)
    for rnd in range(4 * NO):
        o = rnd % NO
        graphs[o].replay()
        torch.cuda.synchronize()
        r = rows[o]
        p.orc.add(r["states"], r["next_states"], r["actions"], r["rewards"], r["dones"], None, count=I)
        want = p.orc.sample(B, 0.5, gather=True)
        gi = out["idx"].cpu().numpy()
        harness.assert_indices(gi, want["idx"], want["near"])
        same = gi == want["idx"]
        harness.assert_weights_close(out["w"].cpu().numpy(), want["w"], mask=same)
        for k in ("states", "next_states", "rewards", "dones"):
            assert np.array_equal(out[k].cpu().numpy()[same].view(np.uint8), want[k][same].view(np.uint8)), k
        if mode == 1:
            _assert_rank_order(p)                    # the order this replay's sample used
        p.orc.update(idx_sets[o], td_sets[o])
    torch.cuda.synchronize()
    if mode in (0, 3):
        p.check_tree()
    p.check_counters()
    assert p.gpu.status_device() == 0
    p.close()


@pytest.mark.parametrize("mode", [0, 2, 3])
def test_graph_replayed_while_filling(mode):
    """Rounds captured while the ring is still filling: every replay inserts at the device cursor
    and the filled size grows on the device, which the samplers (and the flat scan) read there."""
    cap, d, B, I, NO = 4096, 4, 64, 300, 2
    w = _small("tiny", capacity=cap, state_dim=d, row_stride=d, mode=mode)
    g = wl.rng(34, mode)
    p = Pair(cap, d, d, 0.6, 1e-6, mode, seed=6)
    prefill(p, w, g, count=500, chunk=500)
    L, h = capi.load(), p.gpu._h
    rows = [wl.transitions(g, I, w) for _ in range(NO)]
    dev_rows = [{k: dev(v) for k, v in r.items()} for r in rows]
    td = [wl.td_errors(g, B) for _ in range(NO)]
    d_td = [dev(x) for x in td]
    out = p.gpu.alloc_batch(B)
    optr = [out[k].data_ptr() for k in ("idx", "w", "states", "next_states", "actions", "rewards", "dones")]
    graphs = []
    for o in range(NO):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            r = dev_rows[o]
            assert L.per_add(h, I, r["states"].data_ptr(), r["next_states"].data_ptr(), r["actions"].data_ptr(),
                             r["rewards"].data_ptr(), r["dones"].data_ptr(), None, cs) == 0
            assert L.per_sample(h, B, ctypes.c_float(0.5), *optr, cs) == 0
            assert L.per_update_priorities(h, B, out["idx"].data_ptr(), d_td[o].data_ptr(), cs) == 0
        graphs.append(gr)
    for rnd in range(16):                      # 500 + 16 * 300 > 4096: the ring fills and wraps
        o = rnd % NO
        graphs[o].replay()
        torch.cuda.synchronize()
        r = rows[o]
        p.orc.add(r["states"], r["next_states"], r["actions"], r["rewards"], r["dones"], None, count=I)
        want = p.orc.sample(B, 0.5, gather=True)
        gi = out["idx"].cpu().numpy()
        harness.assert_indices(gi, want["idx"], want["near"])
        same = gi == want["idx"]
        assert np.array_equal(out["states"].cpu().numpy()[same], want["states"][same])
        p.orc.update(want["idx"], td[o])
    c = p.counters()                           # the device's counters (the host counted no replay)
    assert (c["calls"], c["cursor"], c["size"]) == (p.orc.sample_calls, p.orc.cursor, p.orc.size)
    assert c["max_raw"] == np.float32(p.orc.max_raw)
    if mode != 2:
        p.check_tree()
    assert p.gpu.status_device() == 0
    p.close()


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")   # the refused call launches nothing
def test_rank_mode_refuses_capture_before_full():
    """A rank-mode sample captured while the ring is filling would keep sorting the captured
    number of slots on every replay; the call is refused during capture until the ring is full."""
    cap, d = 4096, 4
    w = _small("rank", capacity=cap, state_dim=d, row_stride=d)
    g = wl.rng(33)
    p = Pair(cap, d, d, 0.7, 1e-6, 1, seed=3)
    prefill(p, w, g, count=1000, chunk=1000)
    L, h = capi.load(), p.gpu._h
    out = p.gpu.alloc_batch(64)
    optr = [out[k].data_ptr() for k in ("idx", "w", "states", "next_states", "actions", "rewards", "dones")]
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert L.per_sample(h, 64, ctypes.c_float(0.5), *optr, cs) == capi.PER_ERR_INVALID_ARG
    del gr
    p.sample(64, 0.5)                      # outside capture the call runs as usual
    prefill(p, w, g, count=cap - 1000, chunk=cap - 1000)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert L.per_sample(h, 64, ctypes.c_float(0.5), *optr, cs) == 0
    gr.replay()
    torch.cuda.synchronize()
    want = p.orc.sample(64, 0.5, gather=False)
    harness.assert_indices(out["idx"].cpu().numpy(), want["idx"], want["near"])
    p.close()


@pytest.mark.parametrize("seed", [99, 7, 2024])
def test_random_configurations(seed):
    """Seeded random mixes of mode, capacity, row shape, insert sizes (wrapping), batch sizes,
    float dones and update path, every call checked against the oracle."""
    g = wl.rng(seed)
    modes = [0, 1, 2, 3]
    paths = [DEFAULT, CLIMB, REBUILD, ELEMENT]
    for case in range(24):
        mode = modes[case % 4]
        cap = int(g.integers(1, 6000)) if case % 3 else int(g.integers(1, 40000))
        d = int(g.choice([0, 1, 3, 4, 8, 17]))
        dp = d + int(g.choice([0, 0, 1, 4]))
        path = paths[int(g.integers(0, 4))] if mode == 0 else (DEFAULT if mode != 1 else paths[int(g.integers(0, 3))])
        alpha = float(g.choice([0.0, 0.5, 0.6, 1.0]))
        w = _small("tiny", capacity=cap, state_dim=d, row_stride=dp, mode=mode)
        flags = capi.PER_FLAG_DONES_F32 if g.random() < 0.3 else 0
        p = Pair(cap, d, dp, alpha, 1e-6, mode, seed=case, flags=flags, **path)
        for rnd in range(4):
            count = int(g.integers(1, 2 * cap + 2))
            rows = wl.transitions(g, count, w)
            prio = wl.raw_priorities(g, count, "lognormal") if g.random() < 0.7 else None
            p.add(rows, prio)
            p.check_counters()
            B = int(g.integers(1, 2000))
            _, want = p.sample(B, float(g.uniform(0, 1)))
            idx = want["idx"].copy()
            if B > 3 and g.random() < 0.5:
                idx = wl.duplicate_positions(g, idx, 0.3)
            p.update(idx, wl.td_errors(g, B))
            p.check_tree()
        assert p.gpu.status_device() == 0, (case, mode, cap)
        p.close()


# -- the full-size workloads (sampled checks) -------------------------------------------------

@pytest.mark.slow
def test_apex_full_size_rounds():
    w = wl.WORKLOADS["apex"]
    g = wl.rng(10)
    p = Pair(w.capacity, w.state_dim, w.row_stride, w.alpha, w.eps, w.mode, seed=0)
    prefill(p, w, g)
    p.check_tree()
    staging = wl.transitions(wl.rng(10, 1), w.staging, w)
    for r in range(12):
        lo = (r * w.ingest) % w.staging
        rows = {k: v[lo: lo + w.ingest] for k, v in staging.items()}
        p.add(rows, None)
        _, want = p.sample(w.batch, w.beta)
        p.update(want["idx"], wl.td_errors(g, w.batch))
        if r % 4 == 3:
            p.check_tree()
            p.check_counters()
    p.check_tree()
    p.check_counters()
    assert p.stats["mismatch"] <= harness.IDX_MISMATCH_CAP * p.stats["draws"]
    p.close()


@pytest.mark.slow
def test_dqn_full_size_steps():
    w = wl.WORKLOADS["dqn"]
    g = wl.rng(11)
    p = Pair(w.capacity, w.state_dim, w.row_stride, w.alpha, w.eps, w.mode, seed=0)
    prefill(p, w, g)  # prio 'max': every row at the running maximum
    for t in (0, 1, 2, 170, 339, 340):
        _, want = p.sample(w.batch, w.beta_at(t))
        p.update(want["idx"], wl.td_errors(g, w.batch))
    p.check_tree()
    p.check_counters()
    p.close()


@pytest.mark.slow
def test_stress_full_size_sampled():
    """2^24 slots x 256 floats: rows drawn on the device (32 GiB), priorities on the host; the
    oracle keeps the priority trees only and rows are checked by re-drawing their chunk."""
    w = wl.WORKLOADS["stress"]
    g = wl.rng(12)
    p = Pair(w.capacity, w.state_dim, w.row_stride, w.alpha, w.eps, w.mode, seed=0,
             with_ring=False)
    chunk = 1 << 18
    for c in range(w.capacity // chunk):
        s, n = wl.device_rows(torch, 12, c, chunk, w.state_dim)
        a, r, d = wl.device_scalars(torch, 12, c, chunk, w)
        prio = wl.raw_priorities(g, chunk, w.prio)
        p.gpu.add(s, n, a, r, d, dev(prio))
        p.orc.add(raw_prio=prio, count=chunk)
        del s, n
    p.check_tree()
    for rnd in range(3):
        got, want = p.sample(w.batch, w.beta, check_rows=False)
        idx = wl.duplicate_positions(g, want["idx"], w.dup_frac)
        p.update(idx, wl.td_errors(g, w.batch))
        # rows of a sample of draws against their re-drawn source chunk
        gi = got["idx"].cpu().numpy()
        for j in np.linspace(0, w.batch - 1, 16).astype(int):
            slot = int(gi[j])
            s, n = wl.device_rows(torch, 12, slot // chunk, chunk, w.state_dim)
            assert torch.equal(got["states"][j], s[slot % chunk])
            assert torch.equal(got["next_states"][j], n[slot % chunk])
            a, r, d = wl.device_scalars(torch, 12, slot // chunk, chunk, w)
            assert int(got["actions"][j]) == int(a[slot % chunk])
            assert float(got["rewards"][j]) == float(r[slot % chunk])
            assert int(got["dones"][j]) == int(d[slot % chunk])
    p.check_tree()
    p.check_counters()
    p.close()


@pytest.mark.slow
def test_rank_full_size_steps():
    w = wl.WORKLOADS["rank"]
    g = wl.rng(13)
    p = Pair(w.capacity, w.state_dim, w.row_stride, w.alpha, w.eps, w.mode, seed=0)
    prefill(p, w, g)
    for _ in range(4):
        _, want = p.sample(w.batch, w.beta)
        p.update(want["idx"], wl.td_errors(g, w.batch))
        p.check_tree()
    p.check_counters()
    p.close()


# -- error paths (host-side rejection, no launch) ---------------------------------------------

def test_invalid_arguments_rejected():
    b = capi.ReplayBuffer(64, 4)
    h = b._h
    s = capi.per_sample(h, 8, 0.4, None, None, None, None, None, None, None, None)
    assert s == capi.PER_ERR_INVALID_ARG
    idx = torch.empty(8, dtype=torch.int64, device="cuda")
    s = capi.per_sample(h, 8, 0.4, idx.data_ptr(), None, None, None, None, None, None, None)
    assert s == capi.PER_ERR_EMPTY
    s = capi.per_sample(h, 0, 0.4, idx.data_ptr(), None, None, None, None, None, None, None)
    assert s == capi.PER_ERR_INVALID_ARG
    s, _ = capi.per_min(h, None)
    assert s == capi.PER_ERR_EMPTY
    with pytest.raises(capi.PerError):
        capi.ReplayBuffer(0, 4)
    with pytest.raises(capi.PerError):
        capi.ReplayBuffer(16, 8, row_stride_out=4)
    with pytest.raises(capi.PerError):
        capi.ReplayBuffer(16, 8, eps=0.0)
    with pytest.raises(capi.PerError):      # unknown mode
        capi.ReplayBuffer(16, 8, mode=7)
    with pytest.raises(capi.PerError):      # unknown flag bit
        capi.ReplayBuffer(16, 8, flags=1 << 9)
    with pytest.raises(capi.PerError):      # flat mode needs every leaf finite: alpha <= 1
        capi.ReplayBuffer(16, 8, alpha=1.5, mode=capi.PER_MODE_FLAT)
    with pytest.raises(capi.PerError):      # eps^alpha below the smallest normal binary32
        capi.ReplayBuffer(16, 8, alpha=4.0, eps=1e-12)
    cfg = capi.per_config(0.6, 1e-6, 0, 8, 0, 0, 0, 0, 1)   # reserved must be 0
    with pytest.raises(capi.PerError):
        capi.per_create(16, 8, cfg)
    # min is proportional/flat only; uniform updates are checked but change nothing
    u = capi.ReplayBuffer(64, 0, mode=capi.PER_MODE_UNIFORM)
    s, _ = capi.per_min(u._h, None)
    assert s == capi.PER_ERR_INVALID_ARG
    assert capi.per_update_priorities(u._h, 4, None, None, None) == capi.PER_ERR_INVALID_ARG
    u.close()
    # float dones need a 4-byte aligned destination
    f = capi.ReplayBuffer(64, 0, flags=capi.PER_FLAG_DONES_F32)
    z = torch.zeros(64, dtype=torch.float32, device="cuda")
    f.add(None, None, torch.zeros(64, dtype=torch.int32, device="cuda"), z,
          torch.zeros(64, dtype=torch.uint8, device="cuda"))
    dst = torch.zeros(40, dtype=torch.uint8, device="cuda")
    s = capi.per_sample(f._h, 8, 0.4, idx.data_ptr(), None, None, None, None, None, dst.data_ptr() + 1, None)
    assert s == capi.PER_ERR_INVALID_ARG
    f.close()
    b.close()
