"""Drives the CUDA library and the oracle in lockstep on identical seeded inputs.

Inputs flow one way: workloads -> both sides, and the oracle's own sampled indices -> both
updates.  Nothing the CUDA path returns is ever fed to the oracle.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from rl_infra_gb300 import capi
from rl_infra_gb300 import workloads as wl
from tests import harness


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


# Boundary-draw counts of every sampled batch compared in this process, by configuration: the
# parity bar counts index mismatches (each must be a draw the oracle flags as near a boundary)
# and near-boundary draws, and reports both; tests/conftest.py prints them at the end of the run.
BOUNDARY_COUNTS: dict = {}

_FULL_SIZE = {"test_tiny_workload_rounds": "tiny (2^10, B=32)",
              "test_apex_full_size_rounds": "apex (2^21, B=512)",
              "test_dqn_full_size_steps": "dqn (2^20, B=1024)",
              "test_stress_full_size_sampled": "stress (2^24, B=8192)",
              "test_rank_full_size_steps": "rank (2^20, B=1024)",
              "test_flat_apex_size_rounds": "flat (2^21, B=512)"}
_MODE_NAMES = {0: "proportional", 1: "rank", 2: "uniform", 3: "flat"}


def _config_label(mode: int) -> str:
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0].split("::")[-1].split("[")[0]
    return _FULL_SIZE.get(test, f"{_MODE_NAMES.get(mode, mode)}, other cases")


def record_boundary(mode: int, r: dict):
    c = BOUNDARY_COUNTS.setdefault(_config_label(mode), {"draws": 0, "mismatch": 0, "near": 0})
    for k in c:
        c[k] += int(r[k])


class Pair:
    def __init__(self, capacity, d, dp=None, alpha=0.6, eps=1e-6, mode=0, seed=0,
                 with_ring=True, flags=0, rebuild_batch=0, element_batch=0):
        dp = d if dp is None else dp
        self.d, self.dp, self.mode = d, dp, mode
        self.gpu = capi.ReplayBuffer(capacity, d, alpha, eps, mode, dp, seed, flags=flags,
                                     rebuild_batch=rebuild_batch, element_batch=element_batch)
        self.orc = oracle.Oracle(capacity, d, dp, alpha, eps, mode, seed, with_ring)
        self.stats = {"draws": 0, "mismatch": 0, "near": 0, "leaf_ulp": 0}

    def close(self):
        self.gpu.close()
        self.orc.close()

    def add(self, rows: dict, prio=None):
        count = len(rows["actions"])
        self.gpu.add(dev(rows["states"]) if self.d else None,
                     dev(rows["next_states"]) if self.d else None, dev(rows["actions"]),
                     dev(rows["rewards"]), dev(rows["dones"]),
                     None if prio is None else dev(prio))
        self.orc.add(rows["states"], rows["next_states"], rows["actions"], rows["rewards"],
                     rows["dones"], prio, count=count)

    def sample(self, B, beta, check_rows=True):
        got = self.gpu.sample(B, beta, gather=True)
        want = self.orc.sample(B, beta, gather=check_rows)
        gi = got["idx"].cpu().numpy()
        r = harness.assert_indices(gi, want["idx"], want["near"])
        record_boundary(self.mode, r)
        for k in ("draws", "mismatch", "near"):
            self.stats[k] += r[k]
        same = gi == want["idx"]
        harness.assert_weights_close(got["w"].cpu().numpy(), want["w"], mask=same)
        if check_rows:
            for k in ("states", "next_states", "rewards", "dones"):
                g = got[k].cpu().numpy()
                wv = want[k]
                if k == "dones" and g.dtype == np.float32:   # PER_FLAG_DONES_F32
                    wv = (wv != 0).astype(np.float32)
                assert np.array_equal(g[same].view(np.uint8), wv[same].view(np.uint8)), k
            ga = got["actions"].cpu().numpy().view(np.uint32)
            assert np.array_equal(ga[same], want["actions"][same])
        return got, want

    def update(self, idx, td):
        self.gpu.update_priorities(dev(np.asarray(idx, np.int64)), dev(np.asarray(td, np.float32)))
        return self.orc.update(idx, td)

    def check_tree(self, full=True):
        if self.mode == capi.PER_MODE_UNIFORM:
            assert self.gpu.total() == self.orc.total() == self.orc.size
            return
        if self.mode == capi.PER_MODE_RANK:
            assert np.array_equal(self.gpu.read_state(capi.PER_STATE_RAW), self.orc.raw())
            return
        if self.mode == capi.PER_MODE_FLAT:
            gl = self.gpu.read_state(capi.PER_STATE_LEAVES)
            ol = self.orc.leaves()
            ulp = harness.f32_ulp_diff(gl, ol)
            assert ulp.max() <= 1, f"leaves differ by {ulp.max()} ulp"
            self.stats["leaf_ulp"] = int((ulp > 0).sum())
            n = int(self.orc.size)
            if n == 0:
                return
            # the scan's rounding order differs from the oracle's left-to-right sum: both are
            # within n * 2^-53 * T of the exact sums (relative 1e-9 covers 2^31 slots)
            T = self.gpu.total()
            assert abs(T - self.orc.total()) <= 1e-9 * self.orc.total()
            C = self.gpu.read_state(capi.PER_STATE_CUMULATIVE)
            want = np.cumsum(gl[:n].astype(np.float64))
            assert C.shape == want.shape and np.all(np.abs(C - want) <= 1e-9 * T)
            assert C[-1] == T
            assert self.gpu.min() == gl[:n].min()
            return
        gl = self.gpu.read_state(capi.PER_STATE_LEAVES)
        ol = self.orc.leaves()
        ulp = harness.f32_ulp_diff(gl, ol)
        assert ulp.max() <= 1, f"leaves differ by {ulp.max()} ulp"
        self.stats["leaf_ulp"] = int((ulp > 0).sum())
        assert self.stats["leaf_ulp"] <= max(1, len(gl) // 1_000_000), self.stats
        if full and len(gl) > 1:
            gs = self.gpu.read_state(capi.PER_STATE_SUMS)
            os_ = self.orc.sums()
            harness.assert_sums_close(gs[1:], os_[1:])
            gm = self.gpu.read_state(capi.PER_STATE_MINS)
            if self.stats["leaf_ulp"] == 0:
                assert np.array_equal(gs[1:], os_[1:]), "sums not bit-identical"
                assert np.array_equal(gm[1:], self.orc.mins()[1:]), "mins differ"
            assert harness.tree_identity_violations(gl, gs, gm) == {"sum": 0, "min": 0}
        assert self.gpu.total() == self.orc.total() or self.stats["leaf_ulp"] > 0
        if self.orc.size:
            assert self.gpu.min() == np.float32(self.orc.min()) or self.stats["leaf_ulp"] > 0

    def counters(self):
        c = self.gpu.read_state(capi.PER_STATE_COUNTERS)
        return {"calls": int(c[0]), "cursor": int(c[1]), "size": int(c[2]),
                "max_raw": float(np.array([c[3]], np.uint32).view(np.float32)[0]), "crowd": int(c[4])}

    def check_counters(self):
        c = self.counters()
        assert c["calls"] == self.orc.sample_calls
        assert c["cursor"] == self.orc.cursor
        assert c["size"] == self.orc.size
        assert c["max_raw"] == np.float32(self.orc.max_raw)
        assert self.gpu.size == self.orc.size


def prefill(pair: Pair, w: wl.Workload, g, count=None, chunk=1 << 16):
    count = w.capacity if count is None else count
    done = 0
    while done < count:
        c = min(chunk, count - done)
        rows = wl.transitions(g, c, w)
        prio = wl.raw_priorities(g, c, w.prio)
        pair.add(rows, prio)
        done += c
