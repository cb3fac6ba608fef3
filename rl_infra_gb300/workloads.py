"""Seeded synthetic inputs for the replay-buffer workloads.

This module only draws random inputs with the shapes and distributions of the five workloads;
it holds none of the replay method's arithmetic (no priority transform, tree, descent, weight
or gather).  The same bytes feed the CUDA library and the oracle.  Host arrays come from numpy's
PCG64; the large ring contents of the 2^24-slot workload are drawn on the device by torch's
seeded CUDA generator and re-drawn chunk by chunk when a test needs a row back.

Workloads (capacity, state_dim -> gathered row stride, batch, alpha, beta, eps):
  tiny    2^10,  8 -> 8,     B=32,   0.6, 0.4, 1e-6; raw ~ U(0.01, 1); 10 rounds
  apex    2^21,  64 -> 64,   B=512,  0.6, 0.4, 1e-6; raw ~ lognormal(0, 1); 4096-row ingest
          per round from a staging pool of 2^16 rows; 1000 rounds
  dqn     2^20,  48 -> 64,   B=1024, 0.6, beta 0.4 -> 1.0 over 341 steps; prefill at the
          running maximum priority; actions in [0, 3), rewards N(0, 0.1), dones Bernoulli(0.01)
  stress  2^24,  256 -> 256, B=8192, 0.7, 0.5, 1e-6; raw ~ Pareto-I(shape 1.5, x_m 1); 25% of
          the update positions duplicate another position's index; 200 rounds
  rank    2^20,  64 -> 64,   B=1024, 0.7, 0.5, 1e-6; raw ~ |N(0,1)| + 1e-6; rank-based
TD errors are N(0, 1) (the method takes their magnitude).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PROPORTIONAL = 0
RANK = 1
UNIFORM = 2
FLAT = 3


@dataclass(frozen=True)
class Workload:
    name: str
    capacity: int
    state_dim: int
    row_stride: int
    batch: int
    alpha: float
    beta: float
    eps: float
    rounds: int
    mode: int = PROPORTIONAL
    prio: str = "uniform"          # how the prefill's raw priorities are drawn
    ingest: int = 0                # rows inserted at the cursor each round
    staging: int = 0               # rows in the device staging pool the ingest cycles through
    n_actions: int = 4
    reward_sigma: float = 1.0
    done_p: float = 0.05
    dup_frac: float = 0.0          # share of update positions that repeat another index
    beta_end: float | None = None  # annealed beta: beta -> beta_end over `rounds` steps
    extra: dict = field(default_factory=dict)

    def beta_at(self, t: int) -> float:
        if self.beta_end is None:
            return self.beta
        frac = min(t / float(self.rounds), 1.0)
        return self.beta + (self.beta_end - self.beta) * frac


WORKLOADS = {
    "tiny": Workload("tiny", 1 << 10, 8, 8, 32, 0.6, 0.4, 1e-6, 10, prio="uniform"),
    "apex": Workload("apex", 1 << 21, 64, 64, 512, 0.6, 0.4, 1e-6, 1000, prio="lognormal",
                     ingest=4096, staging=1 << 16),
    "dqn": Workload("dqn", 1 << 20, 48, 64, 1024, 0.6, 0.4, 1e-6, 341, prio="max",
                    n_actions=3, reward_sigma=0.1, done_p=0.01, beta_end=1.0),
    "stress": Workload("stress", 1 << 24, 256, 256, 8192, 0.7, 0.5, 1e-6, 200, prio="pareto",
                       dup_frac=0.25),
    "rank": Workload("rank", 1 << 20, 64, 64, 1024, 0.7, 0.5, 1e-6, 100, mode=RANK,
                     prio="absnormal"),
    # the apex shapes drawn uniformly: the plain replay that prioritized replay replaces
    "uniform": Workload("uniform", 1 << 21, 64, 64, 512, 0.6, 0.4, 1e-6, 1000, mode=UNIFORM,
                        prio="lognormal"),
}


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """An independent PCG64 stream per (seed, stream)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def transitions(g: np.random.Generator, count: int, wl: Workload) -> dict:
    """count rows: states, next_states ~ N(0,1) f32 [count, state_dim]; actions u32 uniform in
    [0, n_actions); rewards f32 N(0, reward_sigma); dones u8 Bernoulli(done_p)."""
    d = wl.state_dim
    return {
        "states": g.standard_normal((count, d), dtype=np.float32),
        "next_states": g.standard_normal((count, d), dtype=np.float32),
        "actions": g.integers(0, wl.n_actions, size=count, dtype=np.uint32),
        "rewards": (g.standard_normal(count) * wl.reward_sigma).astype(np.float32),
        "dones": (g.random(count) < wl.done_p).astype(np.uint8),
    }


def raw_priorities(g: np.random.Generator, count: int, kind: str) -> np.ndarray | None:
    """Prefill raw priorities, f32.  'max' returns None (rows take the running maximum)."""
    if kind == "uniform":
        return g.uniform(0.01, 1.0, size=count).astype(np.float32)
    if kind == "lognormal":
        return g.lognormal(0.0, 1.0, size=count).astype(np.float32)
    if kind == "pareto":
        # Pareto type I with x_m = 1 and shape 1.5 by inversion of U in [0, 1)
        u = g.random(count)
        return ((1.0 - u) ** (-1.0 / 1.5)).astype(np.float32)
    if kind == "absnormal":
        return (np.abs(g.standard_normal(count)) + 1e-6).astype(np.float32)
    if kind == "max":
        return None
    raise ValueError(kind)


def td_errors(g: np.random.Generator, count: int) -> np.ndarray:
    return g.standard_normal(count).astype(np.float32)


def duplicate_positions(g: np.random.Generator, idx: np.ndarray, frac: float) -> np.ndarray:
    """Replace round(frac * B) positions, chosen without replacement, by the index held at a
    donor position drawn from the positions left untouched."""
    idx = np.array(idx, dtype=np.int64, copy=True)
    B = len(idx)
    k = int(round(frac * B))
    if k == 0 or B < 2:
        return idx
    k = min(k, B - 1)
    perm = g.permutation(B)
    replaced, keep = perm[:k], perm[k:]
    donors = keep[g.integers(0, len(keep), size=k)]
    idx[replaced] = idx[donors]
    return idx


# -- device-side ring contents for the largest workloads (torch, seeded CUDA generator) ------

def device_rows(torch, seed: int, chunk: int, rows: int, d: int, device="cuda"):
    """states and next_states for one chunk of `rows` rows, drawn on the device; the same
    (seed, chunk) always yields the same bytes."""
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1_000_003 + chunk) & 0x7FFFFFFFFFFFFFFF)
    s = torch.randn((rows, d), generator=gen, device=device, dtype=torch.float32)
    n = torch.randn((rows, d), generator=gen, device=device, dtype=torch.float32)
    return s, n


def device_scalars(torch, seed: int, chunk: int, rows: int, wl: Workload, device="cuda"):
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1_000_033 + chunk + 7) & 0x7FFFFFFFFFFFFFFF)
    actions = torch.randint(0, wl.n_actions, (rows,), generator=gen, device=device,
                            dtype=torch.int32)
    rewards = torch.randn((rows,), generator=gen, device=device) * wl.reward_sigma
    dones = (torch.rand((rows,), generator=gen, device=device) < wl.done_p).to(torch.uint8)
    return actions, rewards.float(), dones
