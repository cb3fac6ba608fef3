"""The oracle: a plain, sequential CPU implementation of prioritized experience replay.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
import this package.  The C source (``per_oracle.c``) is compiled with gcc into
``_build/libper_oracle.so`` and driven through ctypes; this module only marshals arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "per_oracle.c")
_HDR = os.path.join(_HERE, "per_oracle.h")
_LIB = os.path.join(_HERE, "_build", "libper_oracle.so")
_lock = threading.Lock()
_libs: dict = {}

PROPORTIONAL = 0
RANK = 1
UNIFORM = 2
FLAT = 3


def _lib_path(plant: int) -> str:
    return _LIB if plant == 0 else _LIB.replace(".so", f"_plant{plant}.so")


def build(force: bool = False, plant: int = 0) -> str:
    """Compile the oracle with gcc (binary64 as written: no contraction, no fast-math).
    `plant` > 0 builds a separate test copy with one known mistake planted in the
    near-boundary rule (ORC_PLANT in per_oracle.c), for the tests that show its pins catch it."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    out = _lib_path(plant)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(out) or os.path.getmtime(out) < newest:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            f"-DORC_PLANT={int(plant)}", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, out)
    return out


def lib(plant: int = 0) -> ctypes.CDLL:
    with _lock:
        if plant not in _libs:
            L = ctypes.CDLL(build(plant=plant))
            u32, u64, i64, f32, f64, vp = (ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64,
                                           ctypes.c_float, ctypes.c_double, ctypes.c_void_p)
            L.orc_philox4x32_10.argtypes = [vp, vp, vp]
            L.orc_philox4x32_10.restype = None
            L.orc_uniform53.argtypes = [u64, u32, u64, u32]
            L.orc_uniform53.restype = f64
            L.orc_create.argtypes = [u64, u32, u32, f64, f64, u32, u64, ctypes.c_int]
            L.orc_create.restype = vp
            L.orc_destroy.argtypes = [vp]
            L.orc_destroy.restype = None
            L.orc_add.argtypes = [vp, u64, vp, vp, vp, vp, vp, vp]
            L.orc_add.restype = ctypes.c_int
            L.orc_sample.argtypes = [vp, u32, f32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            L.orc_sample.restype = ctypes.c_int
            L.orc_update.argtypes = [vp, u32, vp, vp]
            L.orc_update.restype = ctypes.c_int
            L.orc_descend.argtypes = [vp, f64, vp]
            L.orc_descend.restype = i64
            L.orc_locate.argtypes = [vp, f64, vp, vp, vp]
            L.orc_locate.restype = ctypes.c_int
            L.orc_rank_order.argtypes = [vp, vp]
            L.orc_rank_order.restype = i64
            for name in ("orc_capacity", "orc_nleaves", "orc_size", "orc_cursor",
                         "orc_sample_calls"):
                getattr(L, name).argtypes = [vp]
                getattr(L, name).restype = u64
            L.orc_max_raw.argtypes = [vp]
            L.orc_max_raw.restype = f32
            L.orc_total.argtypes = [vp]
            L.orc_total.restype = f64
            L.orc_min.argtypes = [vp]
            L.orc_min.restype = f32
            for name in ("orc_leaves", "orc_sums", "orc_mins", "orc_raw", "orc_cdf",
                         "orc_ring_states", "orc_ring_next"):
                getattr(L, name).argtypes = [vp]
                getattr(L, name).restype = vp
            _libs[plant] = L
    return _libs[plant]


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniform53(seed: int, j: int, call: int, tag: int) -> float:
    return lib().orc_uniform53(seed, j, call, tag)


class OracleError(RuntimeError):
    pass


class Oracle:
    """One replay buffer held by the oracle (host memory only)."""

    def __init__(self, capacity, state_dim, row_stride_out=None, alpha=0.6, eps=1e-6,
                 mode=PROPORTIONAL, seed=0, with_ring=True, plant=0):
        self.capacity = int(capacity)
        self.d = int(state_dim)
        self.dp = int(row_stride_out if row_stride_out is not None else state_dim)
        self.mode = mode
        self.with_ring = bool(with_ring)
        self._L = lib(plant)
        self._h = self._L.orc_create(self.capacity, self.d, self.dp, float(alpha), float(eps),
                                   int(mode), int(seed), int(with_ring))
        if not self._h:
            raise OracleError("orc_create rejected its arguments or ran out of memory")
        self.n = int(self._L.orc_nleaves(self._h))

    def close(self):
        if self._h:
            self._L.orc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- operations -----------------------------------------------------------------------
    def add(self, states=None, next_states=None, actions=None, rewards=None, dones=None,
            raw_prio=None, count=None):
        if count is None:
            count = len(actions) if actions is not None else len(raw_prio)
        arrs = [None if a is None else np.ascontiguousarray(a, dtype=t)
                for a, t in ((states, np.float32), (next_states, np.float32),
                             (actions, np.uint32), (rewards, np.float32),
                             (dones, np.uint8), (raw_prio, np.float32))]
        rc = self._L.orc_add(self._h, int(count), *[_p(a) for a in arrs])
        if rc != 0:
            raise OracleError(f"orc_add -> {rc}")

    def sample(self, B, beta, gather=True):
        B = int(B)
        out = {
            "idx": np.zeros(B, np.int64), "w": np.zeros(B, np.float32),
            "near": np.zeros(B, np.uint8), "rem": np.zeros(B, np.float64),
            "mass": np.zeros(B, np.float64),
        }
        g = gather and self.with_ring
        if g:
            out["states"] = np.zeros((B, self.dp), np.float32)
            out["next_states"] = np.zeros((B, self.dp), np.float32)
            out["actions"] = np.zeros(B, np.uint32)
            out["rewards"] = np.zeros(B, np.float32)
            out["dones"] = np.zeros(B, np.uint8)
        rc = self._L.orc_sample(
            self._h, B, float(beta), _p(out["idx"]), _p(out["w"]),
            _p(out.get("states")), _p(out.get("next_states")), _p(out.get("actions")),
            _p(out.get("rewards")), _p(out.get("dones")), _p(out["near"]), _p(out["rem"]),
            _p(out["mass"]))
        if rc != 0:
            raise OracleError(f"orc_sample -> {rc}")
        out["near"] = out["near"].astype(bool)
        return out

    def update(self, idx, td) -> int:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        td = np.ascontiguousarray(td, dtype=np.float32)
        rc = self._L.orc_update(self._h, len(idx), _p(idx), _p(td))
        if rc < 0:
            raise OracleError(f"orc_update -> {rc}")
        return rc

    def descend(self, mass):
        rem = ctypes.c_double(0.0)
        leaf = self._L.orc_descend(self._h, float(mass), ctypes.byref(rem))
        return int(leaf), rem.value

    def locate(self, mass):
        """(slot, mass above the slot's extent start, near-boundary flag) of one mass, by the
        same step sample() takes for each draw."""
        slot = ctypes.c_int64(0)
        rem = ctypes.c_double(0.0)
        near = ctypes.c_uint8(0)
        rc = self._L.orc_locate(self._h, float(mass), ctypes.byref(slot), ctypes.byref(rem),
                                ctypes.byref(near))
        if rc != 0:
            raise OracleError(f"orc_locate -> {rc}")
        return int(slot.value), rem.value, bool(near.value)

    def rank_order(self) -> np.ndarray:
        out = np.zeros(max(self.size, 1), np.uint32)
        s = self._L.orc_rank_order(self._h, _p(out))
        if s < 0:
            raise OracleError(f"orc_rank_order -> {s}")
        return out[:s]

    # -- state ----------------------------------------------------------------------------
    @property
    def size(self):
        return int(self._L.orc_size(self._h))

    @property
    def cursor(self):
        return int(self._L.orc_cursor(self._h))

    @property
    def sample_calls(self):
        return int(self._L.orc_sample_calls(self._h))

    @property
    def max_raw(self):
        return float(self._L.orc_max_raw(self._h))

    def total(self):
        return float(self._L.orc_total(self._h))

    def min(self):
        return float(self._L.orc_min(self._h))

    def _view(self, fn, dtype, count):
        ptr = getattr(self._L, fn)(self._h)
        if not ptr:
            return None
        buf = (ctypes.c_char * (count * np.dtype(dtype).itemsize)).from_address(ptr)
        return np.frombuffer(buf, dtype=dtype, count=count).copy()

    def leaves(self):
        return self._view("orc_leaves", np.float32, self.n)

    def sums(self):
        return self._view("orc_sums", np.float64, self.n)

    def mins(self):
        return self._view("orc_mins", np.float32, self.n)

    def raw(self):
        return self._view("orc_raw", np.float32, self.capacity)

    def cdf(self):
        return self._view("orc_cdf", np.float64, self.capacity + 1)

    def ring_states(self):
        return self._view("orc_ring_states", np.float32, self.capacity * self.d).reshape(
            self.capacity, self.d)
