"""Thin ctypes binding of libgbper: the C functions under their own names, plus a small
``ReplayBuffer`` class that marshals torch tensors (device pointer, current CUDA stream).

Nothing here computes: every step of sampling, weighting, gathering and updating runs in the
CUDA kernels of libgbper.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

PER_OK = 0
PER_ERR_INVALID_ARG = 1
PER_ERR_OOM = 2
PER_ERR_CUDA = 3
PER_ERR_EMPTY = 4
PER_ERR_DEVICE_FLAG = 5
PER_ERR_TIMEOUT = 6

PER_MODE_PROPORTIONAL = 0
PER_MODE_RANK = 1
PER_MODE_UNIFORM = 2
PER_MODE_FLAT = 3

PER_DEVFLAG_BAD_INDEX = 1
PER_DEVFLAG_TIMEOUT = 2
PER_DEVFLAG_RANK_STALE = 4
PER_FLAG_RANK_RESORT = 1
PER_FLAG_DONES_F32 = 2
REBUILD_NEVER = 0xFFFFFFFF      # per_config.rebuild_batch: never scatter + rebuild
ELEMENT_NEVER = 1               # per_config.element_batch: never propagate entry by entry
ELEMENT_ALWAYS = 0xFFFFFFFF     # per_config.element_batch: always propagate entry by entry

PER_STATE_LEAVES, PER_STATE_SUMS, PER_STATE_MINS, PER_STATE_RAW, PER_STATE_CDF = 0, 1, 2, 3, 4
PER_STATE_STATES, PER_STATE_NEXT, PER_STATE_ACTIONS, PER_STATE_REWARDS = 5, 6, 7, 8
PER_STATE_DONES, PER_STATE_COUNTERS, PER_STATE_RANK_ORDER, PER_STATE_CUMULATIVE = 9, 10, 11, 12

_STATE_DTYPE = {
    PER_STATE_LEAVES: np.float32, PER_STATE_SUMS: np.float64, PER_STATE_MINS: np.float32,
    PER_STATE_RAW: np.float32, PER_STATE_CDF: np.float64, PER_STATE_STATES: np.float32,
    PER_STATE_NEXT: np.float32, PER_STATE_ACTIONS: np.uint32, PER_STATE_REWARDS: np.float32,
    PER_STATE_DONES: np.uint8, PER_STATE_COUNTERS: np.uint64, PER_STATE_RANK_ORDER: np.uint32,
    PER_STATE_CUMULATIVE: np.float64,
}

# every symbol include/gbper.h declares
EXPORTS = ("per_create", "per_destroy", "per_add", "per_sample", "per_update_priorities",
           "per_total", "per_min", "per_size", "per_status_device", "per_last_error",
           "per_read_state", "per_nleaves", "per_rank_order_noalloc", "per_rank_refresh")


class per_config(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_double), ("eps", ctypes.c_double), ("mode", ctypes.c_uint32),
                ("row_stride_out", ctypes.c_uint32), ("seed", ctypes.c_uint64),
                ("flags", ctypes.c_uint32), ("rebuild_batch", ctypes.c_uint32),
                ("element_batch", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class PerError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libgbper.so; raises if it is missing (there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise ImportError(f"libgbper is not built ({path}); run rl_infra_gb300.build.build()")
            _build.build()
        L = ctypes.CDLL(path)
        vp, u32, u64, f32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float
        st = ctypes.c_int
        L.per_create.argtypes = [u64, u32, ctypes.POINTER(per_config), ctypes.POINTER(vp)]
        L.per_create.restype = st
        L.per_destroy.argtypes = [vp]
        L.per_destroy.restype = st
        L.per_add.argtypes = [vp, u64, vp, vp, vp, vp, vp, vp, vp]
        L.per_add.restype = st
        L.per_sample.argtypes = [vp, u32, f32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.per_sample.restype = st
        L.per_update_priorities.argtypes = [vp, u32, vp, vp, vp]
        L.per_update_priorities.restype = st
        L.per_total.argtypes = [vp, ctypes.POINTER(ctypes.c_double), vp]
        L.per_total.restype = st
        L.per_min.argtypes = [vp, ctypes.POINTER(ctypes.c_float), vp]
        L.per_min.restype = st
        L.per_size.argtypes = [vp, ctypes.POINTER(u64)]
        L.per_size.restype = st
        L.per_nleaves.argtypes = [vp, ctypes.POINTER(u64)]
        L.per_nleaves.restype = st
        L.per_status_device.argtypes = [vp, ctypes.POINTER(u32), vp]
        L.per_status_device.restype = st
        L.per_last_error.argtypes = [vp]
        L.per_last_error.restype = ctypes.c_char_p
        L.per_read_state.argtypes = [vp, u32, u64, u64, vp, vp]
        L.per_read_state.restype = st
        L.per_rank_order_noalloc.argtypes = [vp, u32, vp, vp, vp]
        L.per_rank_refresh.argtypes = [vp, vp]
        L.per_rank_refresh.restype = st
        L.per_rank_order_noalloc.restype = st
        _lib = L
        return L


# -- the C functions under their own names (pointers and sizes in, status out) ---------------

def per_create(capacity, state_dim, cfg: per_config | None):
    L = load()
    h = ctypes.c_void_p()
    s = L.per_create(capacity, state_dim, ctypes.byref(cfg) if cfg is not None else None,
                     ctypes.byref(h))
    if s != PER_OK:
        raise PerError(s, "per_create: " + L.per_last_error(None).decode())
    return h


def per_destroy(h):
    return load().per_destroy(h)


def per_add(h, count, d_states, d_next, d_actions, d_rewards, d_dones, d_raw_prio, stream):
    return load().per_add(h, count, d_states, d_next, d_actions, d_rewards, d_dones, d_raw_prio,
                          stream)


def per_sample(h, B, beta, d_idx, d_w, d_states, d_next, d_actions, d_rewards, d_dones, stream):
    return load().per_sample(h, B, beta, d_idx, d_w, d_states, d_next, d_actions, d_rewards,
                             d_dones, stream)


def per_update_priorities(h, B, d_idx, d_td, stream):
    return load().per_update_priorities(h, B, d_idx, d_td, stream)


def per_total(h, stream):
    v = ctypes.c_double()
    s = load().per_total(h, ctypes.byref(v), stream)
    return s, v.value


def per_min(h, stream):
    v = ctypes.c_float()
    s = load().per_min(h, ctypes.byref(v), stream)
    return s, v.value


def per_size(h):
    v = ctypes.c_uint64()
    s = load().per_size(h, ctypes.byref(v))
    return s, v.value


def per_nleaves(h):
    v = ctypes.c_uint64()
    s = load().per_nleaves(h, ctypes.byref(v))
    return s, v.value


def per_status_device(h, stream):
    v = ctypes.c_uint32()
    s = load().per_status_device(h, ctypes.byref(v), stream)
    return s, v.value


def per_last_error(h):
    return load().per_last_error(h).decode()


def per_read_state(h, which, first, count, host_dst, stream):
    return load().per_read_state(h, which, first, count, host_dst, stream)


def per_rank_refresh(h, stream):
    """Rank mode: bring the slot order up to date (the step per_sample takes first)."""
    return load().per_rank_refresh(h, stream)


def per_rank_order_noalloc(d_raw, n, d_order, d_status, stream):
    """Slot order by raw priority, descending, without any device allocation (n <= 2^18);
    d_status (a device uint32, or None) receives the device's PER_DEVFLAG_* bits."""
    return load().per_rank_order_noalloc(d_raw, n, d_order, d_status, stream)


# -- torch-facing convenience ---------------------------------------------------------------

def _ptr(t, dtype, what, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{what} is required")
    import torch
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class ReplayBuffer:
    """One GPU-resident prioritized replay buffer (device memory owned by libgbper)."""

    def __init__(self, capacity, state_dim, alpha=0.6, eps=1e-6, mode=PER_MODE_PROPORTIONAL,
                 row_stride_out=None, seed=0, flags=0, rebuild_batch=0, element_batch=0):
        import torch
        self.capacity = int(capacity)
        self.state_dim = int(state_dim)
        self.row_stride = int(row_stride_out if row_stride_out is not None else state_dim)
        self.mode = mode
        self.dones_dtype = None  # set below, once torch is imported
        self.device = torch.device("cuda", torch.cuda.current_device())
        self.dones_dtype = torch.float32 if int(flags) & PER_FLAG_DONES_F32 else torch.uint8
        cfg = per_config(float(alpha), float(eps), int(mode), self.row_stride, int(seed), int(flags),
                         int(rebuild_batch), int(element_batch), 0)
        self._h = per_create(self.capacity, self.state_dim, cfg)
        self.nleaves = per_nleaves(self._h)[1]

    def close(self):
        if getattr(self, "_h", None):
            per_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, s, what):
        if s != PER_OK:
            raise PerError(s, f"{what}: {per_last_error(self._h)}")

    def add(self, states, next_states, actions, rewards, dones, raw_prio=None, stream=None):
        import torch
        count = int(actions.numel())
        s = per_add(self._h, count, _ptr(states, torch.float32, "states", self.state_dim == 0),
                    _ptr(next_states, torch.float32, "next_states", self.state_dim == 0),
                    _ptr(actions, torch.int32, "actions") if actions.dtype == torch.int32
                    else _ptr(actions, torch.uint32, "actions"),
                    _ptr(rewards, torch.float32, "rewards"), _ptr(dones, torch.uint8, "dones"),
                    _ptr(raw_prio, torch.float32, "raw_prio", True), _stream(stream))
        self._check(s, "per_add")

    def alloc_batch(self, B, gather=True):
        import torch
        dev = self.device
        out = {"idx": torch.empty(B, dtype=torch.int64, device=dev),
               "w": torch.empty(B, dtype=torch.float32, device=dev)}
        if gather:
            out["states"] = torch.empty((B, self.row_stride), dtype=torch.float32, device=dev)
            out["next_states"] = torch.empty((B, self.row_stride), dtype=torch.float32, device=dev)
            out["actions"] = torch.empty(B, dtype=torch.int32, device=dev)
            out["rewards"] = torch.empty(B, dtype=torch.float32, device=dev)
            out["dones"] = torch.empty(B, dtype=self.dones_dtype, device=dev)
        return out

    def sample(self, B, beta, out=None, gather=True, stream=None):
        import torch
        if out is None:
            out = self.alloc_batch(B, gather)
        g = lambda k, dt: _ptr(out.get(k), dt, k, True)
        s = per_sample(self._h, int(B), float(beta), _ptr(out["idx"], torch.int64, "idx"),
                       g("w", torch.float32), g("states", torch.float32),
                       g("next_states", torch.float32), g("actions", torch.int32),
                       g("rewards", torch.float32), g("dones", self.dones_dtype), _stream(stream))
        self._check(s, "per_sample")
        return out

    def update_priorities(self, idx, td, stream=None):
        import torch
        s = per_update_priorities(self._h, int(idx.numel()), _ptr(idx, torch.int64, "idx"),
                                  _ptr(td, torch.float32, "td"), _stream(stream))
        self._check(s, "per_update_priorities")

    def total(self, stream=None):
        s, v = per_total(self._h, _stream(stream))
        self._check(s, "per_total")
        return v

    def min(self, stream=None):
        s, v = per_min(self._h, _stream(stream))
        self._check(s, "per_min")
        return v

    @property
    def size(self):
        return per_size(self._h)[1]

    def status_device(self, stream=None):
        s, flags = per_status_device(self._h, _stream(stream))
        if s not in (PER_OK, PER_ERR_DEVICE_FLAG):
            self._check(s, "per_status_device")
        return flags

    def read_state(self, which, first=0, count=None, stream=None):
        dtype = _STATE_DTYPE[which]
        if count is None and which == PER_STATE_CUMULATIVE:   # the device's filled size
            count = int(self.read_state(PER_STATE_COUNTERS, 2, 1)[0]) - first
        if count is None:
            count = {PER_STATE_LEAVES: self.nleaves, PER_STATE_SUMS: self.nleaves,
                     PER_STATE_MINS: self.nleaves, PER_STATE_RAW: self.capacity,
                     PER_STATE_CDF: self.capacity + 1,
                     PER_STATE_STATES: self.capacity * self.state_dim,
                     PER_STATE_NEXT: self.capacity * self.state_dim,
                     PER_STATE_ACTIONS: self.capacity, PER_STATE_REWARDS: self.capacity,
                     PER_STATE_DONES: self.capacity, PER_STATE_COUNTERS: 5,
                     PER_STATE_RANK_ORDER: self.size}[which] - first
        buf = np.empty(max(count, 1), dtype=dtype)
        s = per_read_state(self._h, which, first, count, buf.ctypes.data_as(ctypes.c_void_p),
                           _stream(stream))
        self._check(s, "per_read_state")
        return buf[:count]
