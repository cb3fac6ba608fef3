"""The library's environment knobs choose other launch shapes (no cluster for the update, no
programmatic dependent launch, other update and sampler splits, the driver's carveout).  They are
read once per process, so each setting runs in a child process through the same oracle parity
checks as the default shapes."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines skip this module
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, ROOT)
import numpy as np
from rl_infra_gb300 import capi
from rl_infra_gb300 import workloads as wl
from tests.gpu_helpers import Pair, prefill

CLIMB = dict(rebuild_batch=capi.REBUILD_NEVER, element_batch=capi.ELEMENT_NEVER)
for mode in (0, 1, 3):
    for forced in (dict(), CLIMB):
        if mode == 3 and forced:
            continue   # flat mode always scatters
        cap = 1 << 15
        w = wl.Workload(**{**wl.WORKLOADS["tiny"].__dict__, "capacity": cap, "state_dim": 8,
                           "row_stride": 8, "mode": mode})
        g = wl.rng(7, 10 * mode + len(forced))
        p = Pair(cap, 8, 8, 0.6, 1e-6, mode, seed=4, **forced)
        prefill(p, w, g, count=cap - 1000)
        for B in (2, 64, 512, 3000, 20000):
            p.add(wl.transitions(g, 700, w), None)
            _, want = p.sample(min(B, 4096), 0.4, check_rows=True)
            idx = g.integers(0, int(p.orc.size), B)
            idx = wl.duplicate_positions(g, idx, 0.2) if B > 4 else idx
            p.update(idx, wl.td_errors(g, B))
            p.check_tree()
            p.check_counters()
        assert p.gpu.status_device() == 0
        p.close()
print("parity ok")
"""


@pytest.mark.parametrize("env", [
    {"GBPER_UPD_CLUSTER": "0"},
    {"GBPER_PDL": "0"},
    {"GBPER_UPD_SUBS": "1", "GBPER_UPD_PER": "2"},
    {"GBPER_CARVEOUT": "-1", "GBPER_SAMPLE_WARPS": "8", "GBPER_ADD_COPY_PER": "2",
     "GBPER_SAMPLE_CTAS_PER_SM": "4"},
], ids=["no-cluster", "no-pdl", "update-split", "driver-carveout-sampler-copy"])
def test_knob_settings_match_the_oracle(env):
    r = subprocess.run([sys.executable, "-c", CHILD.replace("ROOT", repr(ROOT))], cwd=ROOT,
                       env={**os.environ, **env}, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("parity ok"), (
        r.stdout[-3000:] + r.stderr[-3000:])
