"""The binary32 power used for leaves (rl_infra_gb300/csrc/leaf_pow.cuh), built for the host:
its results equal fl32(pow(x, alpha)) in binary64 bit for bit, its double-float value stays
within 2^-44 of x^alpha (extended-precision reference), and its fallback to the binary64 pow
is rare."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "leafpow_host.cpp")
HDR = os.path.join(ROOT, "rl_infra_gb300", "csrc", "leaf_pow.cuh")
LIB = os.path.join(ROOT, "tests", "_build", "libleafpow_host.so")


@pytest.fixture(scope="module")
def lp():
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                               "-I", os.path.dirname(HDR), SRC, "-o", tmp])
        os.replace(tmp, LIB)
    L = ctypes.CDLL(LIB)
    vp = ctypes.c_void_p
    L.lp_eval.argtypes = [vp, ctypes.c_int, ctypes.c_double, vp, vp, vp, vp]

    def run(x, alpha):
        x = np.ascontiguousarray(x, dtype=np.float32)
        n = len(x)
        out, vhi, vlo = (np.zeros(n, np.float32) for _ in range(3))
        fast = np.zeros(n, np.uint8)
        L.lp_eval(x.ctypes.data_as(vp), n, float(alpha), out.ctypes.data_as(vp),
                  vhi.ctypes.data_as(vp), vlo.ctypes.data_as(vp), fast.ctypes.data_as(vp))
        return out, vhi.astype(np.longdouble) + vlo.astype(np.longdouble), fast.astype(bool)
    return run


def _inputs(seed, n):
    g = np.random.default_rng(seed)
    # log-uniform over 2^-40 .. 2^40, plus priorities in the ranges the workloads produce
    a = np.exp2(g.uniform(-40, 40, n)).astype(np.float32)
    b = (np.abs(g.standard_normal(n)) + 1e-6).astype(np.float32)
    c = g.lognormal(0, 1, n).astype(np.float32)
    d = np.float32(2.0) ** g.integers(-30, 30, n).astype(np.float32)       # exact powers of two
    e = np.nextafter(d, np.float32(np.inf))
    return np.concatenate([a, b, c, d, e])


@pytest.mark.parametrize("alpha", [0.6, 0.7, 0.5, 1.0 / 3.0, 0.9, 1.5, 0.123456789])
def test_leaf_power_exact_and_within_bound(lp, alpha):
    x = _inputs(int(alpha * 1e6), 200_000)
    out, v, fast = lp(x, alpha)
    want = np.power(x.astype(np.float64), alpha).astype(np.float32)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32)), (
        f"{(out != want).sum()} results differ from fl32(pow)")
    ref = np.power(x.astype(np.longdouble), np.longdouble(alpha))
    rel = np.abs((v[fast] - ref[fast]) / ref[fast])
    assert rel.max() < 2.0 ** -44, float(rel.max())
    # the first three groups are random; the last two (powers of two and their neighbours) hold
    # results on or next to a binary32 rounding midpoint for exponents like 1/2, which need the
    # binary64 pow by design
    assert fast[: 3 * 200_000].mean() > 0.9999, fast[: 3 * 200_000].mean()


def test_leaf_power_special_exponents(lp):
    x = _inputs(7, 10_000)
    out, _, fast = lp(x, 0.0)
    assert np.all(out == 1.0) and fast.all()
    out, _, fast = lp(x, 1.0)
    assert np.array_equal(out, x) and fast.all()


def test_leaf_power_falls_back_outside_the_normal_range(lp):
    x = np.array([1e-40, 3e38, 1e-30, 1e30], np.float32)
    out, _, fast = lp(x, 1.5)
    with np.errstate(over="ignore"):
        want = np.power(x.astype(np.float64), 1.5).astype(np.float32)
    assert np.array_equal(out, want)
    assert not fast[0]
