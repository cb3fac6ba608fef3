"""The replicas-only multi-GPU path of bench.py, exercised on the CPU: two gloo ranks agree on the
slowest replica's time and on the whole-job throughput, and under torchrun the reference arm
prints exactly one JSON line, from rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, steps, out_q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        worst = bench.max_over_ranks(times[rank], dist)
        value = bench.aggregate_throughput(dist.get_world_size(), steps, worst)
        out_q.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times, steps, world = [0.5, 1.25], 1000, 2
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, steps, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, worst, value in got:
        assert worst == max(times)
        assert value == pytest.approx(world * steps / max(times))
    assert got[0][1:] == got[1][1:]


def test_single_process_is_identity():
    assert bench.max_over_ranks(0.25, None) == 0.25
    assert bench.aggregate_throughput(1, 400, 0.5) == 800.0
    with pytest.raises(ValueError):
        bench.aggregate_throughput(2, 10, 0.0)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "20", "--warmup", "3", "--cpu-budget", "0.5"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle" and res["e2e"]["h2d_bytes_per_step"] == 0
