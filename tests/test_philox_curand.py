"""The oracle's Philox4x32-10 against cuRAND's device implementation of the same generator
(Salmon, Moraes, Dror, Shaw, SC'11), word for word, at counters and keys spread over their
ranges: the generator the sampling draws from is pinned to an implementation other than the
oracle's own."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _build_ref():
    src = os.path.join(HERE, "curand_ref", "philox_curand.cu")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libphilox_curand.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.check_call(["nvcc", "-shared", "-Xcompiler", "-fPIC", "-O2",
                               "-gencode", "arch=compute_103a,code=sm_103a", src, "-o", so])
    return ctypes.CDLL(so)


@pytest.mark.gpu
def test_oracle_philox_matches_curand():
    import torch
    lib = _build_ref()
    lib.philox_curand.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    g = np.random.default_rng(2024)
    n = 4096
    ctr = g.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = g.integers(0, 2 ** 32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    ctr[:8] = 0                                      # the zero counter and key, and the sampling's
    key[:4] = 0                                      # own layout (draw j, call, tag 0 / 1)
    ctr[8:16, 0] = np.arange(8)
    ctr[8:16, 1:3] = [[7, 0]] * 8
    ctr[8:16, 3] = [0, 1] * 4
    ctr[16:20] = 0xFFFFFFFF
    key[16:20] = 0xFFFFFFFF
    d_ctr = torch.from_numpy(ctr.reshape(-1).view(np.int32)).cuda()
    d_key = torch.from_numpy(key.reshape(-1).view(np.int32)).cuda()
    d_out = torch.zeros(4 * n, dtype=torch.int32, device="cuda")
    assert lib.philox_curand(d_ctr.data_ptr(), d_key.data_ptr(), d_out.data_ptr(), n) == 0
    got = d_out.cpu().numpy().view(np.uint32).reshape(n, 4)
    want = np.stack([oracle.philox4x32_10(ctr[i], key[i]) for i in range(n)])
    bad = np.flatnonzero(np.any(got != want, axis=1))
    assert bad.size == 0, f"{bad.size} of {n} counters differ, first at {bad[:4]}"
