"""The allocation-free rank-order entry point, against the oracle and the existing entry point.

per_rank_order_noalloc serves callers that may not allocate device memory (work enqueued
while a CUDA graph is being captured, allocation-free real-time loops, device memory owned by
another framework's pool); its scratch is a fixed array compiled into the library.  This file
is collected last so that a failure here leaves every other test already run.

Two references, each compared slot for slot (the order is integer work, so the bar is exact):
  * the oracle's rank order (a plain sort over (priority descending, slot ascending)) and
    numpy's stable lexsort of the same keys;
  * per_sample's rank order: a rank-mode buffer with alpha = 0 gives every rank the same
    probability, so with B equal to the filled size the stratified draw j falls on rank j + 1
    exactly and per_sample's indices are the whole rank order.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
from rl_infra_gb300 import build, capi  # noqa: E402
from rl_infra_gb300 import workloads as wl  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    capi.load()


def _rank_order_via_sample(raw: np.ndarray, seed: int) -> torch.Tensor:
    n = len(raw)
    buf = capi.ReplayBuffer(n, 0, alpha=0.0, eps=1e-6, mode=capi.PER_MODE_RANK, seed=seed)
    z = torch.zeros(n, dtype=torch.int32, device="cuda")
    buf.add(None, None, z, z.float(), z.to(torch.uint8), torch.from_numpy(raw).cuda())
    out = buf.sample(n, 0.5, gather=False)
    torch.cuda.synchronize()
    order = out["idx"].clone()
    buf.close()
    return order


def _rank_order_via_oracle(raw: np.ndarray) -> np.ndarray:
    n = len(raw)
    o = oracle.Oracle(n, 0, 0, 0.6, 1e-6, oracle.RANK, 0, with_ring=False)
    o.add(raw_prio=raw, count=n)
    order = o.rank_order().astype(np.int64)
    o.close()
    return order


@pytest.mark.parametrize("n", [1, 4095, 50000, 1 << 18])
def test_noalloc_rank_order_matches_oracle_and_existing_entry_point(n):
    g = wl.rng(99, n)
    raw = wl.raw_priorities(g, n, "absnormal")
    raw[n // 3: n // 3 + n // 10] = raw[n // 2]          # a run of ties
    want = _rank_order_via_oracle(raw)
    assert np.array_equal(want, np.lexsort((np.arange(n), -raw.astype(np.float64))))
    via_sample = _rank_order_via_sample(raw, seed=n).to(torch.int64).cpu().numpy()
    assert np.array_equal(via_sample, want)
    d_raw = torch.from_numpy(raw).cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):                                  # two calls in a row share the scratch
        d_order = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        d_status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        s = capi.per_rank_order_noalloc(d_raw.data_ptr(), n, d_order.data_ptr(), d_status.data_ptr(),
                                        stream)
        assert s == capi.PER_OK
        torch.cuda.synchronize()
        assert int(d_status.item()) == 0, f"call {call}: device flags {int(d_status.item()):#x}"
        got = (d_order.to(torch.int64) & 0xFFFFFFFF).cpu().numpy()
        assert np.array_equal(got, want), f"call {call}: {(got != want).sum()} slots differ"


def test_noalloc_without_status_word():
    n = 3000
    raw = wl.raw_priorities(wl.rng(5, n), n, "absnormal")
    d_raw = torch.from_numpy(raw).cuda()
    d_order = torch.empty(n, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert capi.per_rank_order_noalloc(d_raw.data_ptr(), n, d_order.data_ptr(), None, stream) == capi.PER_OK
    torch.cuda.synchronize()
    assert np.array_equal(d_order.cpu().numpy().astype(np.int64), _rank_order_via_oracle(raw))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    d_raw = torch.ones(16, dtype=torch.float32, device="cuda")
    d_order = torch.empty(16, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert capi.per_rank_order_noalloc(d_raw.data_ptr(), (1 << 18) + 1, d_order.data_ptr(), None,
                                       stream) == capi.PER_ERR_INVALID_ARG
    assert capi.per_rank_order_noalloc(d_raw.data_ptr(), 0, d_order.data_ptr(), None,
                                       stream) == capi.PER_ERR_INVALID_ARG
    assert capi.per_rank_order_noalloc(None, 16, d_order.data_ptr(), None,
                                       stream) == capi.PER_ERR_INVALID_ARG
    assert capi.per_rank_order_noalloc(d_raw.data_ptr(), 16, d_order.data_ptr(), d_order.data_ptr() + 2,
                                       stream) == capi.PER_ERR_INVALID_ARG
