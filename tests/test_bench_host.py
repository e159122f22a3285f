"""Host-side logic of bench.py's multi-GPU (replica) path, run on CPU.

The hot path does not shard: N GPUs run N independent replicas, the job
takes as long as the slowest one, and the reported value counts the work of
all of them.  Two gloo ranks stand in for two GPUs here.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 (r + 1) ms for its steps
        t = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
        v = bench.replica_throughput(8192, 4, world, t)
        out.put((rank, t, v))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    # every rank sees the slowest rank's time, and the same whole-job value
    assert [g[1] for g in got] == [20.0, 20.0]
    assert got[0][2] == got[1][2] == pytest.approx(8192 * 4 * 2 / 0.020)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.replica_throughput(100, 2, 1, 1000.0) == pytest.approx(200.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
