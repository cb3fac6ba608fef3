"""Benchmark of the prioritized-replay hot path: PER steps/s on the 2^21-leaf, B=512 workload.

One step = ingest 4096 rows at the ring cursor (priority = running maximum), draw a stratified
batch of 512 (Philox + descent + IS weights + row gather), update the 512 priorities from TD
errors.  Inputs (staging rows, TD errors) are resident in device memory before timing; L2 is
flushed (a 512 MiB device write) between timed steps, outside the per-step CUDA events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica on its
own GPU (the path has no cross-GPU exchange); the reported time is the maximum over ranks.
--impl reference times the CPU oracle (test infrastructure, single thread) on the same
workload, a bounded number of steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PER steps/s at 2^21 leaves, B=512 (sample+IS+gather+update); HBM GB/s"
UNIT = "steps/s"
WORKLOAD = "apex"
APEX_WORKLOAD = "apex: 2^21 leaves, state_dim 64, B=512, ingest 4096/step, alpha 0.6, beta 0.4"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# -- algorithmic bytes (the byte model) -------------------------------------------------------

def distinct_ancestors(leaves: np.ndarray, D: int, levels: range) -> int:
    """Number of distinct nodes over the given heights above the given leaves."""
    u = np.unique(np.asarray(leaves, dtype=np.int64))
    return int(sum(len(np.unique(u >> h)) for h in levels))


def bytes_ingest(count, d, D, cursor, C):
    slots = (cursor + np.arange(count, dtype=np.int64)) % C
    nodes = distinct_ancestors(slots, D, range(1, D + 1))
    rows = count * 2 * (4 * d) * 2           # states + next: read source, write ring
    scalars = count * (4 + 4 + 1) * 2        # actions, rewards, dones: read + write
    return rows + scalars + 4 * count + 36 * nodes


def bytes_sample(idx, d, dp, D):
    # left child read at every visited internal node: distinct path nodes at depths 0..D-1
    path_nodes = distinct_ancestors(idx, D, range(1, D + 1))
    B = len(idx)
    descent = 8 * path_nodes + 4 * B
    weights = 8 * B
    gather = B * (2 * (4 * d + 4 * dp) + (4 + 4 + 1) * 2 + 8)
    return descent + weights + gather


def bytes_update(idx, D):
    B = len(idx)
    nodes = distinct_ancestors(idx, D, range(1, D + 1))
    return 12 * B + 4 * len(np.unique(idx)) + 36 * nodes


def strip_c_comments(src: str) -> str:
    """C/CUDA source with its comments removed and every run of whitespace made one space, so
    that an edit of comments or layout alone leaves the result unchanged (string and character
    literals are kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(name):
    """First 16 hex digits of the sha256 of a kernel source file, comments and layout aside."""
    p = os.path.join(ROOT, "rl_infra_gb300", "csrc", name)
    code = strip_c_comments(open(p, encoding="utf-8").read())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def traffic_from_profiles(kernel, kernel_file, workload="apex"):
    """Per-launch DRAM bytes (read + write) of a kernel on a workload, from the committed ncu
    summary profiles/traffic.txt (lines of key=value: kernel, file, src_sha,
    dram_bytes_per_launch, workload), if the kernel's source file is unchanged since the capture
    (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash(kernel_file)
    for line in open(p):
        parts = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if (parts.get("kernel") == kernel and parts.get("file") == kernel_file and parts.get("src_sha") == want
                and parts.get("workload") == workload):
            try:
                return float(parts["dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


# -- clocks during the timed region -------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# -- raw CUDA runtime calls for the timed loop (a few microseconds of host time per step, so the
#    host stays ahead of the device and the events time device work only) -------------------------

class Cudart:
    def __init__(self):
        import ctypes
        self.ct = ctypes
        lib = None
        for name in ("libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so.13", "libcudart.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("libcudart not found")
        vp = ctypes.c_void_p
        lib.cudaEventCreate.argtypes = [ctypes.POINTER(vp)]
        lib.cudaEventRecord.argtypes = [vp, vp]
        lib.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), vp, vp]
        lib.cudaEventDestroy.argtypes = [vp]
        lib.cudaMemsetAsync.argtypes = [vp, ctypes.c_int, ctypes.c_size_t, vp]
        self.lib = lib

    def events(self, n):
        out = []
        for _ in range(n):
            e = self.ct.c_void_p()
            if self.lib.cudaEventCreate(self.ct.byref(e)) != 0:
                raise RuntimeError("cudaEventCreate failed")
            out.append(e)
        return out

    def elapsed_ms(self, a, b):
        v = self.ct.c_float()
        if self.lib.cudaEventElapsedTime(self.ct.byref(v), a, b) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return v.value

    def destroy(self, evs):
        for e in evs:
            self.lib.cudaEventDestroy(e)


# -- the GPU arm ---------------------------------------------------------------------------------

def setup_gpu(torch, w, seed=0):
    from rl_infra_gb300 import capi
    from rl_infra_gb300 import workloads as wl
    buf = capi.ReplayBuffer(w.capacity, w.state_dim, w.alpha, w.eps, w.mode, w.row_stride, seed)
    g = wl.rng(seed, 77)
    chunk = 1 << 18
    for c in range(w.capacity // chunk):
        s, n = wl.device_rows(torch, seed, c, chunk, w.state_dim)
        a, r, d = wl.device_scalars(torch, seed, c, chunk, w)
        prio = torch.from_numpy(wl.raw_priorities(g, chunk, w.prio)).cuda()
        buf.add(s, n, a, r, d, prio)
    s, n = wl.device_rows(torch, seed + 1, 0, w.staging, w.state_dim)
    a, r, d = wl.device_scalars(torch, seed + 1, 0, w.staging, w)
    staging = {"states": s, "next_states": n, "actions": a, "rewards": r, "dones": d}
    torch.cuda.synchronize()
    return buf, staging, g


def _check(L, h, status, what):
    if status != 0:
        raise RuntimeError(f"{what}: status {status}: {L.per_last_error(h).decode()}")


def _ring_ptrs(t: dict, lo: int):
    """Device addresses of row `lo` of each staging array (states, next, actions, rewards, dones)."""
    out = []
    for k in ("states", "next_states", "actions", "rewards", "dones"):
        v = t[k]
        row = v.element_size() * (v.shape[1] if v.dim() > 1 else 1)
        out.append(v.data_ptr() + lo * row)
    return out


def _out_ptrs(out: dict):
    return [out[k].data_ptr() for k in ("idx", "w", "states", "next_states", "actions", "rewards",
                                         "dones")]


# -- replicas: one process per GPU, each running the whole step on its own buffer --------------

def max_over_ranks(value: float, dist=None) -> float:
    """The slowest replica's time: MAX all-reduce of one float over every rank (a no-op on one
    process).  NCCL reduces a CUDA tensor, gloo a CPU tensor."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(world: int, steps: int, max_secs: float) -> float:
    """Whole-job steps/s: every rank ran `steps` steps; the job took the slowest rank's time."""
    if max_secs <= 0:
        raise ValueError("timed region must be positive")
    return world * steps / max_secs


def run_gpu(args, rank, world):
    import ctypes
    import torch
    from rl_infra_gb300 import capi
    from rl_infra_gb300 import workloads as wl
    w = wl.WORKLOADS[WORKLOAD]
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", dev))
    buf, staging, g = setup_gpu(torch, w)
    L, h = capi.load(), buf._h
    K, W = args.steps, args.warmup
    B, I = w.batch, w.ingest
    TD_SLOTS = 4096
    td = torch.from_numpy(wl.td_errors(g, TD_SLOTS * B)).cuda()
    out = buf.alloc_batch(B)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    evict = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    evict_out = torch.empty((), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    st = ctypes.c_void_p(stream.cuda_stream)
    beta = ctypes.c_float(w.beta)
    # every pointer of the step, computed once: the timed loop only issues the three C calls
    add_args = [(h, I, *_ring_ptrs(staging, o * I), None, st) for o in range(w.staging // I)]
    sample_args = (h, B, beta, *_out_ptrs(out), st)
    idx_ptr, td0 = out["idx"].data_ptr(), td.data_ptr()
    n_ofs = len(add_args)

    flush_l2 = args.l2 == "flush"
    cr = Cudart()
    rec, memset = cr.lib.cudaEventRecord, cr.lib.cudaMemsetAsync
    flush_ptr, flush_n = flush.data_ptr(), flush.numel()

    def step(t, ev=None, flush=True):
        if ev is not None:
            rec(ev[0], st)
        _check(L, h, L.per_add(*add_args[t % n_ofs]), "per_add")
        if ev is not None and ev[1] is not None:
            rec(ev[1], st)
        _check(L, h, L.per_sample(*sample_args), "per_sample")
        if ev is not None and ev[2] is not None:
            rec(ev[2], st)
        _check(L, h, L.per_update_priorities(h, B, idx_ptr, td0 + 4 * B * (t % TD_SLOTS), st),
               "per_update")
        if ev is not None:
            rec(ev[3], st)
        if flush_l2 and flush:
            # evict L2 between steps, outside the step's events: write 512 MiB, then read 256 MiB
            # so the next step starts on clean, unrelated lines rather than a write-back backlog
            memset(flush_ptr, 0, flush_n, st)
            torch.sum(evict, 0, out=evict_out)

    # the clock sampler starts before the warm-up, so the timed steps follow the warm-up directly
    clocks = ClockSampler(dev) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    for t in range(W):
        step(t)
    torch.cuda.synchronize()
    cursor0 = int(buf.read_state(capi.PER_STATE_COUNTERS, 1, 1)[0])  # device cursor before timing

    # timed region: K steps, each bracketed by two events on the launching stream (no events
    # between the three calls, so each kernel's launch overlaps its predecessor's tail)
    sev = cr.events(2 * K)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for t in range(K):
        step(W + t, (sev[2 * t], None, None, sev[2 * t + 1]))
    host_s = time.perf_counter() - t0
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist:
        dist.barrier()
    step_ms = np.array([cr.elapsed_ms(sev[2 * t], sev[2 * t + 1]) for t in range(K)])
    cr.destroy(sev)

    # continuous: the same K steps back to back between one pair of events (the canonical form:
    # K steps bracketed by synchronisation; no flush, the 1 GiB ring exceeds L2)
    ca, cb = cr.events(2)
    torch.cuda.synchronize()
    rec(ca, st)
    t1 = time.perf_counter()
    for t in range(K):
        _check(L, h, L.per_add(*add_args[(W + t) % n_ofs]), "per_add")
        _check(L, h, L.per_sample(*sample_args), "per_sample")
        _check(L, h, L.per_update_priorities(h, B, idx_ptr, td0 + 4 * B * ((W + t) % TD_SLOTS), st),
               "per_update")
    cont_host_s = time.perf_counter() - t1
    rec(cb, st)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None   # the sampler spans both timed loops
    cont_s = cr.elapsed_ms(ca, cb) / 1e3
    cr.destroy([ca, cb])
    cont_s = max_over_ranks(cont_s, dist)

    # per-kernel breakdown (for the roofline): a second pass with an event between the calls and,
    # like the timed region, no flush between steps.  Each event pair also carries a launch
    # without the programmatic overlap, so these durations are upper bounds.
    Kop = min(K, 4000)
    flat = cr.events(4 * Kop)
    for t in range(Kop):
        step(W + K + t, flat[4 * t: 4 * t + 4], flush=False)
    torch.cuda.synchronize()
    per = np.array([[cr.elapsed_ms(flat[4 * t + i], flat[4 * t + i + 1]) for i in range(3)]
                    for t in range(Kop)])
    cr.destroy(flat)

    # the same rounds captured as one CUDA graph (one round per staging offset, each an
    # insertion + sample + update) and replayed back to back: the kernels advance their own
    # device counters, so every replayed round inserts at the cursor and draws a fresh batch
    graph_res = None
    if not args.no_graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for o in range(n_ofs):
                _check(L, h, L.per_add(*(add_args[o][:-1] + (cs,))), "per_add")
                _check(L, h, L.per_sample(*(sample_args[:-1] + (cs,))), "per_sample")
                _check(L, h, L.per_update_priorities(h, B, idx_ptr, td0 + 4 * B * o, cs), "per_update")
        torch.cuda.synchronize()
        reps = max(1, K // n_ofs)
        for _ in range(max(1, W // n_ofs)):
            gr.replay()
        torch.cuda.synchronize()
        ga, gb = cr.events(2)
        rec(ga, st)
        for _ in range(reps):
            gr.replay()
        rec(gb, st)
        torch.cuda.synchronize()
        g_s = max_over_ranks(cr.elapsed_ms(ga, gb) / 1e3, dist)
        cr.destroy([ga, gb])
        if buf.status_device() != 0:
            raise RuntimeError("device error flag raised during the graph replays")
        graph_res = {"value": round(aggregate_throughput(world, reps * n_ofs, g_s), 2), "unit": UNIT,
                     "ms_per_step": round(g_s * 1e3 / (reps * n_ofs), 5), "steps": reps * n_ofs,
                     "note": (f"{n_ofs} rounds (insertion + sample + update each) captured as one CUDA graph, "
                              "replayed back to back between two events")}
        del gr
    total_s = float(step_ms.sum()) / 1e3
    total_s = max_over_ranks(total_s, dist)
    value_flushed = aggregate_throughput(world, K, total_s)
    if buf.status_device() != 0:
        raise RuntimeError("device error flag raised during the benchmark")

    # byte model from this run's actual indices and ring range
    idx = out["idx"].cpu().numpy()
    D = int(np.log2(buf.nleaves))
    b_add = bytes_ingest(I, w.state_dim, D, cursor0, w.capacity)
    b_sam = bytes_sample(idx, w.state_dim, w.row_stride, D)
    b_upd = bytes_update(idx, D)
    ops = {
        "k_add": (float(np.median(per[:, 0])), b_add, "k_tree.cu"),
        "k_sample_prop": (float(np.median(per[:, 1])), b_sam, "k_sample.cu"),
        "k_update": (float(np.median(per[:, 2])), b_upd, "k_tree.cu"),
    }
    peak, peak_src = load_peaks()
    dom = max(ops, key=lambda k: ops[k][0])
    ms, byt, src = ops[dom]
    achieved = byt / (ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 2), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 5),
                "traffic": traffic_from_profiles(dom, src), "peak_source": peak_src,
                "algorithmic_bytes_per_launch": int(byt), "median_launch_us": round(ms * 1e3, 3)}
    step_bytes = b_add + b_sam + b_upd

    res = {
        "metric": METRIC, "value": round(aggregate_throughput(world, K, cont_s), 2), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(cont_s * 1e3 / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; rows N(0,1) drawn on the device, lognormal(0,1) priorities)",
        "config": {"workload": APEX_WORKLOAD,
                   "l2": ("value: not flushed, inputs larger than L2 (1 GiB ring + 48 MiB trees + "
                          "32 MiB staging vs 129 MB L2; each step ingests new rows and gathers random "
                          "ones); per_step_l2_flushed: 512 MiB write + 256 MiB read between steps"),
                   "timing": ("value: K steps back to back on one stream between two CUDA events, "
                              "synchronised on both sides; per-kernel figures from a separate pass "
                              "with an event between the calls and no flush (as the timed region)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "wall_s_timed_loop": round(wall, 4), "host_enqueue_s": round(host_s, 4),
                   "host_enqueue_us_per_step": round(cont_host_s * 1e6 / K, 3)},
        "hbm_gbs_algorithmic": round(step_bytes / (cont_s / K) / 1e9 / world, 2),
        "bytes_per_step": {"k_add": int(b_add), "k_sample_prop": int(b_sam), "k_update": int(b_upd)},
        "ops_median_us": {k: round(v[0] * 1e3, 3) for k, v in ops.items()},
        "ops_p99_us": {k: round(float(np.percentile(per[:, i], 99)) * 1e3, 3)
                       for i, k in enumerate(ops)},
        "ops_max_us": {k: round(float(per[:, i].max()) * 1e3, 3) for i, k in enumerate(ops)},
        "roofline": roofline,
        "gpu_launches": 3 * K,
        "per_step_l2_flushed": {"value": round(value_flushed, 2), "unit": UNIT,
                                "us_per_step_median": round(float(np.median(step_ms)) * 1e3, 3),
                                "us_per_step_p99": round(float(np.percentile(step_ms, 99)) * 1e3, 3),
                                "timing": "two events per step, L2 flushed between steps"
                                          if flush_l2 else "two events per step, no flush"},
    }
    if clk:
        res["clocks"] = clk
    if graph_res:
        res["graph"] = graph_res

    # steady state: right after the prefill every new row enters at the running maximum, so the
    # draws crowd the last rows written until the ring has turned over once (2^21 / 4096 = 512
    # steps); the same step timed back to back once that pass is complete
    done = int(buf.read_state(capi.PER_STATE_COUNTERS, 0, 1)[0])    # sample calls = steps so far
    ring_pass = w.capacity // I
    t_next = W + K + Kop + K
    for t in range(max(0, ring_pass + 64 - done)):
        _check(L, h, L.per_add(*add_args[(t_next + t) % n_ofs]), "per_add")
        _check(L, h, L.per_sample(*sample_args), "per_sample")
        _check(L, h, L.per_update_priorities(h, B, idx_ptr, td0 + 4 * B * ((t_next + t) % TD_SLOTS), st),
               "per_update")
    torch.cuda.synchronize()
    after = int(buf.read_state(capi.PER_STATE_COUNTERS, 0, 1)[0])
    Ks = max(K, 2000)
    sa, sb = cr.events(2)
    rec(sa, st)
    for t in range(Ks):
        _check(L, h, L.per_add(*add_args[(t_next + t) % n_ofs]), "per_add")
        _check(L, h, L.per_sample(*sample_args), "per_sample")
        _check(L, h, L.per_update_priorities(h, B, idx_ptr, td0 + 4 * B * ((t_next + t) % TD_SLOTS), st),
               "per_update")
    rec(sb, st)
    torch.cuda.synchronize()
    ss_s = max_over_ranks(cr.elapsed_ms(sa, sb) / 1e3, dist)
    cr.destroy([sa, sb])
    if buf.status_device() != 0:
        raise RuntimeError("device error flag raised during the steady-state steps")
    crowd = int(buf.read_state(capi.PER_STATE_COUNTERS, 4, 1)[0])
    res["steady_state"] = {"value": round(aggregate_throughput(world, Ks, ss_s), 2), "unit": UNIT,
                           "last_update_report": {"subtrees_log2": crowd >> 28, "most_entries": crowd & 0xFFFFF},
                           "ms_per_step": round(ss_s * 1e3 / Ks, 5), "steps": Ks, "after_steps": after,
                           "note": ("the same step, back to back between two events, once the ring has "
                                    "turned over (every slot rewritten since the prefill); `value` times "
                                    "the K steps right after the warm-up, while new rows entered at the "
                                    "running maximum still crowd the draws")}
    res["e2e"] = run_e2e(torch, buf, w, staging, g, min(K, 4000), dist)
    buf.close()
    if dist:
        dist.destroy_process_group()
    return res


def run_flat_design(args):
    """The apex step with the pages' own flat sampler (PER_MODE_FLAT: the leaves summed into a
    cumulative array at each sample, one search per draw, no tree; updates only scatter leaves)
    timed like the headline: K steps back to back between two events, then a pass with an event
    between the calls for the per-call medians."""
    import ctypes
    import dataclasses
    import torch
    from rl_infra_gb300 import capi
    from rl_infra_gb300 import workloads as wl
    w = dataclasses.replace(wl.WORKLOADS[WORKLOAD], mode=wl.FLAT)
    buf, staging, g = setup_gpu(torch, w)
    L, h = capi.load(), buf._h
    K, W, B, I = args.steps, args.warmup, w.batch, w.ingest
    TD_SLOTS = 4096
    td = torch.from_numpy(wl.td_errors(g, TD_SLOTS * B)).cuda()
    out = buf.alloc_batch(B)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    beta = ctypes.c_float(w.beta)
    add_args = [(h, I, *_ring_ptrs(staging, o * I), None, st) for o in range(w.staging // I)]
    sample_args = (h, B, beta, *_out_ptrs(out), st)
    idx_ptr, td0 = out["idx"].data_ptr(), td.data_ptr()
    cr = Cudart()
    rec = cr.lib.cudaEventRecord

    def calls(t, ev=None):
        if ev is not None:
            rec(ev[0], st)
        _check(L, h, L.per_add(*add_args[t % len(add_args)]), "per_add")
        if ev is not None:
            rec(ev[1], st)
        _check(L, h, L.per_sample(*sample_args), "per_sample")
        if ev is not None:
            rec(ev[2], st)
        _check(L, h, L.per_update_priorities(h, B, idx_ptr, td0 + 4 * B * (t % TD_SLOTS), st), "per_update")
        if ev is not None:
            rec(ev[3], st)

    for t in range(W):
        calls(t)
    torch.cuda.synchronize()
    ca, cb = cr.events(2)
    rec(ca, st)
    for t in range(K):
        calls(W + t)
    rec(cb, st)
    torch.cuda.synchronize()
    cont_s = cr.elapsed_ms(ca, cb) / 1e3
    cr.destroy([ca, cb])
    Kop = min(K, 2000)
    ev = cr.events(4 * Kop)
    for t in range(Kop):
        calls(W + K + t, ev[4 * t: 4 * t + 4])
    torch.cuda.synchronize()
    per = np.array([[cr.elapsed_ms(ev[4 * t + i], ev[4 * t + i + 1]) for i in range(3)] for t in range(Kop)])
    cr.destroy(ev)
    if buf.status_device() != 0:
        raise RuntimeError("device error flag raised during the flat-design run")
    n = w.capacity
    # the scan reads every leaf and writes C (4 + 8 bytes per slot); the search reads about 5
    # rounds of 32 probes per draw
    res = {"value": round(K / cont_s, 2), "unit": UNIT, "ms_per_step": round(cont_s * 1e3 / K, 5),
           "steps": K, "scan_bytes": 12 * n,
           "ops_median_us": {"per_add (k_add, leaves only)": round(float(np.median(per[:, 0])) * 1e3, 3),
                             "per_sample (k_flat_reduce + k_flat_scan + k_sample_flat)": round(float(np.median(per[:, 1])) * 1e3, 3),
                             "per_update (k_upd_scatter + k_upd_apply + k_upd_finish)":
                                 round(float(np.median(per[:, 2])) * 1e3, 3)},
           "gpu_launches_per_step": 7,
           "note": ("the apex step in PER_MODE_FLAT (the pages' cumulative array + search, no tree), "
                    "K steps back to back between two events; per-call medians from a pass with events "
                    "between the calls (2.048 us event resolution)")}
    buf.close()
    return res


def run_crowded(args):
    """Lasting crowding on the apex shape: every slot prefilled at raw priority 1e-6, each step
    inserts 512 rows at the running maximum (they keep nearly all the mass, so the draws crowd
    the newest rows), samples 512 and updates them with TD errors of order 1e-3.  Steps/s with
    the default update dispatch (which follows the crowding) and with each update path forced,
    K steps back to back between two events after W + 64 untimed steps."""
    import ctypes
    import torch
    from rl_infra_gb300 import capi
    from rl_infra_gb300 import workloads as wl
    w = wl.WORKLOADS[WORKLOAD]
    K, W, B, I = args.steps, args.warmup, w.batch, 512
    res = {"note": ("apex shape (2^21 slots, state_dim 64, B=512) with every slot prefilled at raw "
                    "priority 1e-6, 512 rows a step inserted at the running maximum, TD errors N(0,1) x 1e-3; "
                    "K steps back to back between two events")}
    for label, rb in (("default", 0), ("climb", capi.REBUILD_NEVER), ("rebuild", 1)):
        buf = capi.ReplayBuffer(w.capacity, w.state_dim, w.alpha, w.eps, w.mode, w.row_stride, 0,
                                rebuild_batch=rb)
        chunk = 1 << 18
        for c in range(w.capacity // chunk):
            sd, nd = wl.device_rows(torch, 0, c, chunk, w.state_dim)
            a, r, d = wl.device_scalars(torch, 0, c, chunk, w)
            buf.add(sd, nd, a, r, d, torch.full((chunk,), 1e-6, dtype=torch.float32, device="cuda"))
        sd, nd = wl.device_rows(torch, 1, 0, 1 << 14, w.state_dim)
        a, r, d = wl.device_scalars(torch, 1, 0, 1 << 14, w)
        staging = {"states": sd, "next_states": nd, "actions": a, "rewards": r, "dones": d}
        g = wl.rng(0, 88)
        td = torch.from_numpy(wl.td_errors(g, 64 * B) * np.float32(1e-3)).cuda()
        out = buf.alloc_batch(B)
        L, h = capi.load(), buf._h
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        add_args = [(h, I, *_ring_ptrs(staging, o * I), None, st) for o in range((1 << 14) // I)]
        sample_args = (h, B, ctypes.c_float(w.beta), *_out_ptrs(out), st)
        idx_ptr, td0 = out["idx"].data_ptr(), td.data_ptr()

        def one(t):
            _check(L, h, L.per_add(*add_args[t % len(add_args)]), "per_add")
            _check(L, h, L.per_sample(*sample_args), "per_sample")
            _check(L, h, L.per_update_priorities(h, B, idx_ptr, td0 + 4 * B * (t % 64), st), "per_update")

        for t in range(W + 64):
            one(t)
            if t % 8 == 7:
                torch.cuda.synchronize()   # let the crowding count reach the host
        torch.cuda.synchronize()
        cr = Cudart()
        e0, e1 = cr.events(2)
        cr.lib.cudaEventRecord(e0, st)
        for t in range(K):
            one(W + 64 + t)
        cr.lib.cudaEventRecord(e1, st)
        torch.cuda.synchronize()
        secs = cr.elapsed_ms(e0, e1) / 1e3
        cr.destroy([e0, e1])
        crowd = int(buf.read_state(capi.PER_STATE_COUNTERS, 4, 1)[0])
        if buf.status_device() != 0:
            raise RuntimeError("device error flag raised during the crowded run")
        res[label] = {"value": round(K / secs, 2), "unit": UNIT, "us_per_step": round(secs * 1e6 / K, 3),
                      "steps": K, "last_report": {"subtrees_log2": crowd >> 28, "most_entries": crowd & 0xFFFFF}}
        buf.close()
        del staging, td, out
        torch.cuda.empty_cache()
    return res


def run_e2e(torch, buf, w, staging, g, K, dist):
    """Steps/s through the public C calls with the inputs in pinned host memory: each step copies
    its ingest rows and TD errors host->device (one packed copy) and the sampled batch
    device->host (one packed copy), inside the timing."""
    import ctypes
    from rl_infra_gb300 import capi
    from rl_infra_gb300 import workloads as wl
    L, h = capi.load(), buf._h
    B, I, d = w.batch, w.ingest, w.state_dim
    n_ofs = w.staging // I
    # packed host arena per step: states | next | actions | rewards | dones | pad | td
    sizes = [("states", I * d * 4), ("next_states", I * d * 4), ("actions", I * 4),
             ("rewards", I * 4), ("dones", I), ("td", B * 4)]
    offs, o = {}, 0
    for k, n in sizes:
        offs[k] = o
        o = (o + n + 255) // 256 * 256
    arena = o
    host_in = torch.empty((n_ofs, arena), dtype=torch.uint8).pin_memory()
    td_all = wl.td_errors(g, n_ofs * B).reshape(n_ofs, B)
    for s_ in range(n_ofs):
        lo = s_ * I
        for k, n in sizes[:-1]:
            v = staging[k][lo:lo + I].contiguous().view(torch.uint8).reshape(-1).cpu()
            host_in[s_, offs[k]:offs[k] + n] = v
        host_in[s_, offs["td"]:offs["td"] + B * 4] = torch.from_numpy(td_all[s_].view(np.uint8))
    # packed device output arena: idx | w | states | next | actions | rewards | dones
    osz = [("idx", B * 8), ("w", B * 4), ("states", B * w.row_stride * 4),
           ("next_states", B * w.row_stride * 4), ("actions", B * 4), ("rewards", B * 4),
           ("dones", B)]
    ooffs, o = {}, 0
    for k, n in osz:
        ooffs[k] = o
        o = (o + n + 255) // 256 * 256
    out_bytes = o
    # G-step groups over 2G device arenas each way: group g+1's inputs go up on one copy stream
    # while group g computes, and group g-1's batches come down on another.  The compute stream
    # waits on the copy streams once per group, so the kernels of a group keep their
    # programmatic overlap; every step still has its own H2D copy and its own D2H copy.  A short
    # run is set by the pipeline's fill (the first step starts after its group's copies), a long
    # one by the group boundaries: measured on GB300, groups of one step for 20 steps (35.0-35.3K
    # steps/s against 33.6K with groups of 4), of 4 for 20,000 (36.3K against 34.5K for 1).
    G = 1 if K <= 64 else 4
    NA = 2 * G
    dev_in = [torch.empty(arena, dtype=torch.uint8, device="cuda") for _ in range(NA)]
    dev_out = [torch.empty(out_bytes, dtype=torch.uint8, device="cuda") for _ in range(NA)]
    host_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(NA)]
    cr = Cudart()
    lib, vp = cr.lib, ctypes.c_void_p
    lib.cudaStreamCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
    lib.cudaStreamDestroy.argtypes = [vp]
    lib.cudaMemcpyAsync.argtypes = [vp, vp, ctypes.c_size_t, ctypes.c_int, vp]
    lib.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
    lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
    s_in, s_out = vp(), vp()
    if lib.cudaStreamCreateWithFlags(ctypes.byref(s_in), 1) or lib.cudaStreamCreateWithFlags(ctypes.byref(s_out), 1):
        raise RuntimeError("cudaStreamCreateWithFlags failed")

    def sync_events(n):
        evs = []
        for _ in range(n):
            e = vp()
            if lib.cudaEventCreateWithFlags(ctypes.byref(e), 2):   # cudaEventDisableTiming
                raise RuntimeError("cudaEventCreateWithFlags failed")
            evs.append(e)
        return evs

    ev_in, ev_comp, ev_out = sync_events(2), sync_events(2), sync_events(2)   # by group parity
    stream = torch.cuda.current_stream()
    st = ctypes.c_void_p(stream.cuda_stream)
    host_base = host_in.data_ptr()
    args = []
    for b in range(NA):
        bi, bo = dev_in[b].data_ptr(), dev_out[b].data_ptr()
        args.append(((h, I, bi + offs["states"], bi + offs["next_states"], bi + offs["actions"],
                      bi + offs["rewards"], bi + offs["dones"], None, st),
                     (h, B, ctypes.c_float(w.beta), *[bo + ooffs[k] for k, _ in osz], st),
                     (h, B, bo + ooffs["idx"], bi + offs["td"], st)))
    rec, wait, cpy = lib.cudaEventRecord, lib.cudaStreamWaitEvent, lib.cudaMemcpyAsync

    def upload(grp):
        """H2D copies of group grp's steps into its arenas, once group grp-2 no longer uses them."""
        p_ = grp & 1
        if grp >= 2:
            wait(s_in, ev_comp[p_], 0)
        for t in range(grp * G, grp * G + G):
            b = t % NA
            cpy(dev_in[b].data_ptr(), host_base + (t % n_ofs) * arena, arena, 1, s_in)
        rec(ev_in[p_], s_in)

    def group(grp):
        """Group grp's steps on the compute stream, then the D2H copy of each step's batch."""
        p_ = grp & 1
        wait(st, ev_in[p_], 0)
        if grp >= 2:
            wait(st, ev_out[p_], 0)         # group grp-2's batches have left these arenas
        for t in range(grp * G, grp * G + G):
            a_add, a_sam, a_upd = args[t % NA]
            _check(L, h, L.per_add(*a_add), "per_add")
            _check(L, h, L.per_sample(*a_sam), "per_sample")
            _check(L, h, L.per_update_priorities(*a_upd), "per_update")
        rec(ev_comp[p_], st)
        wait(s_out, ev_comp[p_], 0)
        for t in range(grp * G, grp * G + G):
            b = t % NA
            cpy(host_out[b].data_ptr(), dev_out[b].data_ptr(), out_bytes, 2, s_out)
        rec(ev_out[p_], s_out)

    def run_groups(g0, ng):
        upload(g0)
        for grp in range(g0, g0 + ng):
            if grp + 1 < g0 + ng:
                upload(grp + 1)
            group(grp)

    run_groups(0, 2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = cr.events(2)
    torch.cuda.synchronize()
    ngroups = max(1, K // G)
    K = ngroups * G
    rec(e0, s_in)
    run_groups(2, ngroups)
    rec(e1, s_out)
    torch.cuda.synchronize()
    secs = cr.elapsed_ms(e0, e1) / 1e3
    cr.destroy([e0, e1] + ev_in + ev_comp + ev_out)
    lib.cudaStreamDestroy(s_in)
    lib.cudaStreamDestroy(s_out)
    secs = max_over_ranks(secs, dist)
    world = dist.get_world_size() if dist else 1
    return {"value": round(aggregate_throughput(world, K, secs), 2), "unit": UNIT,
            "h2d_bytes_per_step": int(sum(n for _, n in sizes)),
            "d2h_bytes_per_step": int(sum(n for _, n in osz)), "steps": K,
            "note": ("pinned host rows + TD errors in, sampled batch out, one copy each way for every step, "
                     f"inside the timing; the copies run on two copy streams in groups of {G} step(s) over {2 * G} "
                     "device arenas each way, overlapping the neighbouring groups' kernels")}


# -- the other workloads (sample + update steps; rank adds the sort) -------------------------------

KERNEL_FILES = {"k_sample_prop": "k_sample.cu", "k_update": "k_tree.cu", "k_sample_uniform": "k_sample.cu",
                "k_rank_merge": "k_rank.cu", "k_sample_rank": "k_sample.cu"}

OTHER = {
    "tiny": "tiny: 2^10 leaves, state_dim 8, B=32, alpha 0.6, beta 0.4",
    "dqn": "dqn: 2^20 leaves, state_dim 48 gathered into 64-float rows, B=1024, beta 0.4->1.0 over 341 steps",
    "stress": "stress: 2^24 leaves, state_dim 256, B=8192, 25% duplicate update indices, alpha 0.7, beta 0.5",
    "rank": "rank-based: 2^20 slots, state_dim 64, B=1024, order brought up to date (merge, or radix sort when rebuilt) + rank sample + update, alpha 0.7, beta 0.5",
    "uniform": "uniform: 2^21 slots, state_dim 64, B=512, uniform stratified draws + gather, dones as f32 (the update is a no-op)",
}


def run_other(args, name, resort=False, steps=None, warmup=None, op_steps=None):
    """Steps/s of one sample (+IS +gather) and one update per step on another workload; the rank
    workload's sample call brings the slot order up to date (merging the slots written since
    the previous sample, or with `resort` sorting every slot again).  Same timing rules as the
    apex step: `steps` steps (default --steps) after `warmup` untimed ones, two events around
    each step and L2 flushed between steps; per-call medians from `op_steps` further steps."""
    import ctypes
    import torch
    from rl_infra_gb300 import capi
    from rl_infra_gb300 import workloads as wl
    import dataclasses
    w = wl.WORKLOADS[name]
    if getattr(args, "state_dim", None) is not None:   # the same tree and batch with other rows
        w = dataclasses.replace(w, state_dim=args.state_dim, row_stride=max(args.state_dim, 0))
    torch.cuda.set_device(0)
    flags = (capi.PER_FLAG_RANK_RESORT if resort else 0) | (capi.PER_FLAG_DONES_F32 if w.mode == wl.UNIFORM else 0)
    buf = capi.ReplayBuffer(w.capacity, w.state_dim, w.alpha, w.eps, w.mode, w.row_stride, 0, flags=flags)
    g = wl.rng(0, 55)
    chunk = min(w.capacity, 1 << 18)
    for c in range(w.capacity // chunk):
        sd, nd = wl.device_rows(torch, 0, c, chunk, w.state_dim)
        a, r, d = wl.device_scalars(torch, 0, c, chunk, w)
        prio = wl.raw_priorities(g, chunk, w.prio)
        buf.add(sd, nd, a, r, d, None if prio is None else torch.from_numpy(prio).cuda())
        del sd, nd
    torch.cuda.synchronize()
    L, h = capi.load(), buf._h
    K = args.steps if steps is None else steps
    W = args.warmup if warmup is None else warmup
    B = w.batch
    out = buf.alloc_batch(B)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # update batches: the sampled indices, or (stress) a copy with 25% duplicated positions
    NS = 64
    idx_sets = torch.empty((NS, B), dtype=torch.int64, device="cuda")
    td = torch.from_numpy(wl.td_errors(g, NS * B)).cuda().view(NS, B)
    for k in range(NS):
        buf.sample(B, w.beta_at(0), out=out)
        ix = out["idx"].cpu().numpy()
        if w.dup_frac:
            ix = wl.duplicate_positions(g, ix, w.dup_frac)
        idx_sets[k] = torch.from_numpy(ix).cuda()
    torch.cuda.synchronize()
    ptrs = [out[k].data_ptr() for k in ("idx", "w", "states", "next_states", "actions", "rewards", "dones")]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    evict = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    evict_out = torch.empty((), dtype=torch.float32, device="cuda")
    cr = Cudart()
    rec, memset = cr.lib.cudaEventRecord, cr.lib.cudaMemsetAsync
    flush_l2 = args.l2 == "flush"

    rank = w.mode == wl.RANK

    def calls(t):
        """The step's C calls: (rank) the order brought up to date, the sample, the update."""
        beta = ctypes.c_float(w.beta_at(t % max(w.rounds, 1)))
        k = t % NS
        out_ = []
        if rank:
            out_.append(lambda: _check(L, h, L.per_rank_refresh(h, st), "per_rank_refresh"))
        out_.append(lambda: _check(L, h, L.per_sample(h, B, beta, *ptrs, st), "per_sample"))
        out_.append(lambda: _check(L, h, L.per_update_priorities(h, B, idx_sets[k].data_ptr(), td[k].data_ptr(), st),
                                   "per_update"))
        return out_

    NC = len(calls(0))

    def step(t, ev):
        """One step; ev holds NC + 1 events (None: no event at that point)."""
        for i, c in enumerate(calls(t)):
            if ev[i] is not None:
                rec(ev[i], st)
            c()
        rec(ev[NC], st)
        if flush_l2:
            memset(flush.data_ptr(), 0, flush.numel(), st)
            torch.sum(evict, 0, out=evict_out)

    warm = cr.events(NC + 1)
    for t in range(W):
        step(t, warm)
    torch.cuda.synchronize()
    sev = cr.events(2 * K)
    t0 = time.perf_counter()
    for t in range(K):
        step(W + t, [sev[2 * t]] + [None] * (NC - 1) + [sev[2 * t + 1]])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    step_ms = np.array([cr.elapsed_ms(sev[2 * t], sev[2 * t + 1]) for t in range(K)])
    cr.destroy(sev)
    Kop = min(K, 1000) if op_steps is None else op_steps
    fl = cr.events((NC + 1) * Kop)
    for t in range(Kop):
        step(W + K + t, fl[(NC + 1) * t: (NC + 1) * (t + 1)])
    torch.cuda.synchronize()
    per = np.array([[cr.elapsed_ms(fl[(NC + 1) * t + i], fl[(NC + 1) * t + i + 1]) for i in range(NC)]
                    for t in range(Kop)])
    cr.destroy(fl + warm)
    if buf.status_device() != 0:
        raise RuntimeError("device error flag raised during the benchmark")
    idx = out["idx"].cpu().numpy()
    D = int(np.log2(buf.nleaves))
    upd_idx = idx_sets[(W + K + Kop - 1) % NS].cpu().numpy()
    if rank:
        n = w.capacity
        d = len(np.unique(upd_idx))
        # order merge: previous keys + slots in, new keys + slots out (16 B per slot), and the
        # listed slots' entries (slot, old key, raw: 12 B) once; the full sort: the histogram pass
        # reads 4 B per key, passes 0-2 read and write 8 B per key, pass 3 reads 8 and writes 4 B
        b_ord = (16 * n + 12 * d) if not resort else (4 * n + 3 * 16 * n + 12 * n)
        # the sampler: CDF guide and probes (about 2 x 8 B), the order entry (4 B), weight and
        # index (12 B), rows read and written, action, reward, done in and out
        b_sam = B * (16 + 4 + 12 + 2 * (4 * w.state_dim + 4 * w.row_stride) + 18)
        b_upd = 12 * B + 8 * d
        names = ("sort (k_rs_hist4 + 4 k_rs_onesweep)" if resort else "k_rank_merge", "k_sample_rank",
                 "k_upd_block")
        byts = (b_ord, b_sam, b_upd)
    elif w.mode == wl.UNIFORM:
        # idx + weight out; rows read and written; action, reward in and out; done 1 B in, 4 B out
        b_sam = B * (8 + 4 + 2 * (4 * w.state_dim + 4 * w.row_stride) + 8 + 8 + 5)
        names = ("k_sample_uniform", "update (no kernel in this mode)")
        byts = (b_sam, 0)
    else:
        b_sam = bytes_sample(idx, w.state_dim, w.row_stride, D)
        b_upd = bytes_update(upd_idx, D)
        names = ("k_sample_prop", "k_update")
        byts = (b_sam, b_upd)
    ops = {nm: (float(np.median(per[:, i])), byts[i]) for i, nm in enumerate(names)}
    if w.mode == wl.UNIFORM:
        del ops[names[1]]
    b_step = sum(byts)
    peak, peak_src = load_peaks()
    dom = max(ops, key=lambda k: ops[k][0])
    ms, byt = ops[dom]
    achieved = byt / (ms * 1e-3) / 1e9
    total_s = float(step_ms.sum()) / 1e3
    res = {
        "metric": f"PER steps/s ({OTHER[name].split(':')[0]} workload)", "value": round(K / total_s, 2),
        "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": round(total_s * 1e3 / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": OTHER[name] + (f" (rows of {w.state_dim} floats)" if getattr(args, "state_dim", None)
                                              is not None else ""),
                   "l2": "flushed between steps" if flush_l2 else "not flushed",
                   "wall_s_timed_loop": round(wall, 4)},
        "step_us_median": round(float(np.median(step_ms)) * 1e3, 3),
        "ops_median_us": {k: round(v[0] * 1e3, 3) for k, v in ops.items()},
        "bytes_per_step": {k: int(v[1]) for k, v in ops.items()},
        "hbm_gbs_algorithmic": round(b_step / (total_s / K) / 1e9, 2),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 5),
                     "traffic": traffic_from_profiles(dom, KERNEL_FILES[dom], name) if dom in KERNEL_FILES else None,
                     "peak_source": peak_src, "algorithmic_bytes_per_launch": int(byt),
                     "median_launch_us": round(ms * 1e3, 3)},
        # rank: order (merge, or histogram + 4 sort passes) + sampler + the cluster update kernel
        "gpu_launches": ((7 if resort else 3) if w.mode == wl.RANK else 1 if w.mode == wl.UNIFORM else 2) * K,
    }
    if w.mode == wl.RANK:
        res["config"]["rank_order"] = ("every slot sorted again at each sample (4-pass radix sort)" if resort
                                       else "previous order merged with the slots written since")
    buf.close()
    return res


def run_workloads(args):
    """The larger configurations beside the headline (one GPU): dqn, stress and rank (the order
    kept between samples, and sorted again at each sample), each timed like run_other: the
    driver's --steps steps after --warmup, L2 flushed between steps, per-call medians from at
    least 200 further steps.  Each buffer is freed before the next is made (stress holds 32 GiB)."""
    import torch
    keep = ("value", "unit", "steps", "warmup", "ms_per_step", "step_us_median", "ops_median_us",
            "bytes_per_step", "hbm_gbs_algorithmic", "roofline", "gpu_launches", "config")
    out = {}
    for name in ("dqn", "stress", "rank"):
        r = run_other(args, name, op_steps=max(args.steps, 200))
        rec = {k: r[k] for k in keep if k in r}
        if name == "rank":
            full = run_other(args, "rank", resort=True, op_steps=max(args.steps, 200))
            rec["full_resort"] = {k: full[k] for k in keep if k in full}
        out[name] = rec
        torch.cuda.empty_cache()
    return out


# -- the update's two paths against the batch size ------------------------------------------------

def run_update_crossover(args):
    """Median time of one per_update_priorities call (L2 flushed before each) by batch size, on
    the path that climbs from each changed leaf and on the path that scatters and rebuilds every
    tree level, for the tree sizes of the workloads.  The library's default dispatch picks the
    rebuild from the batch size where it becomes the faster one."""
    import ctypes
    import torch
    from rl_infra_gb300 import capi
    from rl_infra_gb300 import workloads as wl
    torch.cuda.set_device(0)
    cr = Cudart()
    rec, memset = cr.lib.cudaEventRecord, cr.lib.cudaMemsetAsync
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    L = capi.load()
    g = wl.rng(0, 77)
    reps = max(5, min(args.steps, 40))
    rows = []
    configs = [("tiny tree", 1 << 10, wl.PROPORTIONAL), ("2^16 tree", 1 << 16, wl.PROPORTIONAL),
               ("dqn tree", 1 << 20, wl.PROPORTIONAL), ("apex tree", 1 << 21, wl.PROPORTIONAL),
               ("stress tree", 1 << 24, wl.PROPORTIONAL), ("rank slots", 1 << 20, wl.RANK)]
    if args.crossover_trees:
        keep = set(args.crossover_trees.split(","))
        configs = [c for c in configs if c[0].split()[0] in keep]
    for label, n, mode in configs:
        bufs = {}
        paths = [("climb", capi.REBUILD_NEVER, capi.ELEMENT_NEVER), ("rebuild", 1, capi.ELEMENT_NEVER)]
        if mode == wl.PROPORTIONAL:
            paths.append(("element", capi.REBUILD_NEVER, capi.ELEMENT_ALWAYS))
        for path, rb, eb in paths:
            buf = capi.ReplayBuffer(n, 0, 0.6, 1e-6, mode, 0, 0, rebuild_batch=rb, element_batch=eb)
            chunk = min(n, 1 << 20)
            a = torch.zeros(chunk, dtype=torch.int32, device="cuda")
            r = torch.zeros(chunk, dtype=torch.float32, device="cuda")
            d = torch.zeros(chunk, dtype=torch.uint8, device="cuda")
            for c in range(n // chunk):
                prio = torch.from_numpy(wl.raw_priorities(g, chunk, "lognormal")).cuda()
                buf.add(None, None, a, r, d, prio)
            bufs[path] = buf
        torch.cuda.synchronize()
        Bs = [b for b in (1, 4, 16, 64, 256, 1024, 4096, 8192, 16384, 32768, 65536, 131072, 262144, 1 << 20,
                          1 << 22) if b <= 4 * n]
        for B in Bs:
            idx = torch.from_numpy(g.integers(0, n, B).astype(np.int64)).cuda()
            td = torch.from_numpy(wl.td_errors(g, B)).cuda()
            row = {"tree": label, "n": n, "B": B}
            for path, buf in bufs.items():
                if path == "element" and B > 1024:
                    continue   # one entry after another: about 1.5 us each
                h = buf._h
                ev = cr.events(2 * reps)
                for t in range(3 + reps):
                    memset(flush.data_ptr(), 0, flush.numel(), st)
                    if t >= 3:
                        rec(ev[2 * (t - 3)], st)
                    _check(L, h, L.per_update_priorities(h, B, idx.data_ptr(), td.data_ptr(), st), "per_update")
                    if t >= 3:
                        rec(ev[2 * (t - 3) + 1], st)
                torch.cuda.synchronize()
                row[path + "_us"] = round(float(np.median([cr.elapsed_ms(ev[2 * k], ev[2 * k + 1])
                                                           for k in range(reps)])) * 1e3, 3)
                cr.destroy(ev)
            rows.append(row)
        for buf in bufs.values():
            if buf.status_device() != 0:
                raise RuntimeError("device error flag raised during the update sweep")
            buf.close()
    cross, elem = {}, {}
    for label, n, _ in configs:
        if not any(r["tree"] == label for r in rows):
            continue
        rs = [r for r in rows if r["tree"] == label]
        cross[label] = next((r["B"] for r in rs if r["rebuild_us"] < r["climb_us"]), None)
        if any("element_us" in r for r in rs):
            elem[label] = next((r["B"] for r in rs if "element_us" in r and r["element_us"] > r["climb_us"]), None)
    return {"metric": "per_update_priorities time by batch size, each path (us, L2 flushed)",
            "reps": reps, "rows": rows, "rebuild_faster_from_B": cross, "element_slower_from_B": elem}


# -- the oracle on the host cores ------------------------------------------------------------------

def oracle_steps_per_s(budget_s=12.0, max_steps=None, warmup=0):
    """The oracle's apex steps per second on one host core: `warmup` untimed steps after the
    prefill, then steps timed until `max_steps` or `budget_s` seconds, whichever comes first.
    The prefill priorities and the TD errors come from the same seeded stream, in the same
    order, as the GPU arm's (setup_gpu, run_gpu), so both arms run the same step on the same
    priorities; the rows (which the step only copies) come from a host stream of their own."""
    import oracle
    from rl_infra_gb300 import workloads as wl
    w = wl.WORKLOADS[WORKLOAD]
    g = wl.rng(0, 77)          # priorities, then TD errors: the GPU arm's stream
    rows_g = wl.rng(0, 99)
    o = oracle.Oracle(w.capacity, w.state_dim, w.row_stride, w.alpha, w.eps, w.mode, 0, True)
    chunk = 1 << 18
    for _ in range(w.capacity // chunk):
        rows = wl.transitions(rows_g, chunk, w)
        o.add(rows["states"], rows["next_states"], rows["actions"], rows["rewards"],
              rows["dones"], wl.raw_priorities(g, chunk, w.prio))
    staging = wl.transitions(rows_g, w.staging, w)
    TD_SLOTS = 4096
    td = wl.td_errors(g, TD_SLOTS * w.batch).reshape(TD_SLOTS, w.batch)

    def one(t):
        lo = (t * w.ingest) % w.staging
        o.add(*(staging[k][lo:lo + w.ingest] for k in
                ("states", "next_states", "actions", "rewards", "dones")), None)
        s = o.sample(w.batch, w.beta)
        o.update(s["idx"], td[t % TD_SLOTS])

    for t in range(warmup):
        one(t)
    t0 = time.perf_counter()
    steps = 0
    while True:
        one(warmup + steps)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and steps >= max_steps):
            break
    o.close()
    return steps / el, steps, el


def cpu_info():
    model = ""
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                model = ln.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    return model, os.cpu_count()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="apex",
                    choices=["apex", "tiny", "dqn", "stress", "rank", "uniform", "crowded"],
                    help="apex is the headline workload; the others are measured with --workload")
    ap.add_argument("--state-dim", type=int, default=None,
                    help="with --workload other than apex: rows of this many floats (the same tree and "
                         "batch; small rows keep a profiler capture of the tree kernels small)")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip timing the rounds captured as one CUDA graph")
    ap.add_argument("--l2", default="flush", choices=["flush", "warm"],
                    help="flush L2 between timed steps, or rely on inputs larger than L2")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-flat", action="store_true",
                    help="skip timing the apex step with the flat cumulative-array sampler")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the dqn, stress and rank records of the default run")
    ap.add_argument("--update-crossover", action="store_true",
                    help="time both update paths against the batch size and exit")
    ap.add_argument("--crossover-trees", default="",
                    help="comma-separated first words of the sweep's tree labels (tiny, 2^16, dqn, apex, "
                         "stress, rank); all when empty")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        if rank != 0:
            return
        # W untimed steps, then K timed ones, cut short (and said so in `sample`) only if they
        # would take more than the budget on the host
        budget = min(args.cpu_budget * max(1, args.steps // 1000), 120.0)
        sps, n, el = oracle_steps_per_s(budget_s=budget, max_steps=args.steps, warmup=args.warmup)
        model, cores = cpu_info()
        res = {"metric": METRIC, "value": round(sps, 3), "unit": UNIT, "n_gpus": world,
               "steps": n, "warmup": args.warmup, "ms_per_step": round(1e3 / sps, 4),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic (seeded)", "impl": "reference",
               "config": {"workload": APEX_WORKLOAD},
               "cpu_baseline": {"value": round(sps, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{n} apex steps in {el:.1f} s" + (
                                    f" (of {args.steps}: the {budget:.0f} s budget ran out)"
                                    if n < args.steps else ""),
                                "cpu": model, "host_cores": cores},
               "e2e": {"value": round(sps, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return

    if args.update_crossover:
        if rank == 0:
            print(json.dumps(run_update_crossover(args)))
        return
    if args.workload == "crowded":
        if rank == 0:
            print(json.dumps(run_crowded(args)))
        return
    if args.workload != "apex":
        if rank == 0:
            res = run_other(args, args.workload)
            if args.workload == "rank":
                full = run_other(args, "rank", resort=True)
                res["full_resort"] = {k: full[k] for k in ("value", "unit", "step_us_median", "ops_median_us",
                                                           "bytes_per_step", "roofline")}
            print(json.dumps(res))
        return
    res = run_gpu(args, rank, world)
    if rank == 0 and world == 1 and not args.no_flat:
        res["flat_design"] = run_flat_design(args)
    if rank == 0 and world == 1 and not args.no_workloads:
        res["workloads"] = run_workloads(args)
        res["workloads"]["apex_lasting_crowding"] = run_crowded(args)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            sps, n, el = oracle_steps_per_s(budget_s=args.cpu_budget)
            model, cores = cpu_info()
            res["cpu_baseline"] = {"value": round(sps, 3), "unit": UNIT, "cores": 1,
                                   "kind": "oracle", "sample": f"{n} apex steps in {el:.1f} s",
                                   "cpu": model, "host_cores": cores}
        print(json.dumps(res))


if __name__ == "__main__":
    main()
