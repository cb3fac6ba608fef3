"""CPU-side checks of the C ABI: the library builds, loads and exports every function that
include/gbper.h declares (no compute call is made without a GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

from rl_infra_gb300 import build, capi, workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:per_status|const char\s*\*)\s*(\w+)\s*\(", src, re.M)))


def test_library_builds_and_exports_every_declared_symbol():
    path = build.build()
    lib = ctypes.CDLL(path)
    names = _declared("gbper.h")
    assert "per_create" in names and "per_sample" in names and len(names) >= 12
    for name in names:
        assert hasattr(lib, name), f"{name} declared in gbper.h but not exported"
    assert sorted(capi.EXPORTS) == names


def test_binding_loads_without_a_device():
    L = capi.load()
    assert L.per_last_error(None) == b""
    out = ctypes.c_uint64(7)
    assert L.per_size(None, ctypes.byref(out)) == capi.PER_ERR_INVALID_ARG


def test_oracle_exports_its_header():
    import oracle
    lib = oracle.lib()
    src = open(os.path.join(ROOT, "oracle", "per_oracle.h")).read()
    names = set(re.findall(r"\b(orc_\w+)\s*\(", src))
    for name in names:
        assert hasattr(lib, name), name


def test_duplicate_positions_properties():
    g = wl.rng(0)
    idx = np.arange(8192, dtype=np.int64) * 3
    out = wl.duplicate_positions(g, idx, 0.25)
    changed = out != idx
    assert changed.sum() == 2048
    # every replaced position now repeats an index that an untouched position holds
    untouched = set(out[~changed].tolist())
    assert all(v in untouched for v in out[changed].tolist())


def test_workload_table_matches_the_configs():
    W = wl.WORKLOADS
    assert (W["tiny"].capacity, W["tiny"].state_dim, W["tiny"].batch) == (1 << 10, 8, 32)
    assert (W["apex"].capacity, W["apex"].state_dim, W["apex"].batch, W["apex"].ingest) == (
        1 << 21, 64, 512, 4096)
    assert (W["dqn"].capacity, W["dqn"].state_dim, W["dqn"].row_stride, W["dqn"].batch) == (
        1 << 20, 48, 64, 1024)
    assert W["dqn"].beta_at(0) == 0.4 and abs(W["dqn"].beta_at(341) - 1.0) < 1e-12
    assert (W["stress"].capacity, W["stress"].state_dim, W["stress"].batch) == (1 << 24, 256, 8192)
    assert (W["rank"].capacity, W["rank"].mode, W["rank"].alpha, W["rank"].beta) == (
        1 << 20, wl.RANK, 0.7, 0.5)
    assert (W["uniform"].capacity, W["uniform"].state_dim, W["uniform"].batch, W["uniform"].mode) == (
        1 << 21, 64, 512, wl.UNIFORM)
    p = wl.raw_priorities(wl.rng(1), 100000, "pareto")
    assert p.min() >= 1.0 and abs(np.median(p) - 2 ** (1 / 1.5)) < 0.03


def test_binding_constants_match_the_header():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hdr = open(os.path.join(root, "include", "gbper.h")).read()
    consts = {m.group(1): int(m.group(2)) for m in
              re.finditer(r"\b(PER_(?:MODE|FLAG|STATE|DEVFLAG|ERR)_[A-Z0-9_]+)\s*=\s*(\d+)u?\b", hdr)}
    assert {"PER_MODE_UNIFORM", "PER_FLAG_DONES_F32", "PER_STATE_RANK_ORDER"} <= consts.keys()
    for name, v in consts.items():
        assert getattr(capi, name) == v, name
    import oracle
    assert (oracle.PROPORTIONAL, oracle.RANK, oracle.UNIFORM) == (
        capi.PER_MODE_PROPORTIONAL, capi.PER_MODE_RANK, capi.PER_MODE_UNIFORM)
    assert (wl.PROPORTIONAL, wl.RANK, wl.UNIFORM) == (
        capi.PER_MODE_PROPORTIONAL, capi.PER_MODE_RANK, capi.PER_MODE_UNIFORM)
