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


def test_traffic_records_are_gated_on_the_kernel_source(tmp_path, monkeypatch):
    """A DRAM-traffic record counts only while its kernel source is the one it
    was captured on: the same file gives its bytes, any edit gives None."""
    import hashlib
    csrc = tmp_path / "gated_delta_rule_kk_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("__global__ void k() {}\n")
    sha = hashlib.sha256((csrc / "k.cu").read_bytes()).hexdigest()[:12]
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment\n"
        f"row_a source=k.cu sha={sha} bytes_per_launch=1.5e+08\n"
        "row_b source=k.cu sha=000000000000 bytes_per_launch=2e+08\n"
        f"row_c source=missing.cu sha={sha} bytes_per_launch=3e+08\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("row_a") == 1.5e8
    assert bench.traffic_record("row_b") is None
    assert bench.traffic_record("row_c") is None
    assert bench.traffic_record("row_d") is None
    (csrc / "k.cu").write_text("__global__ void k() { }\n")
    assert bench.traffic_record("row_a") is None


def test_committed_traffic_records_are_well_formed():
    """Every record names an existing kernel source, a 12-digit hash and a
    positive byte count."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert rows
    for f in rows:
        kv = dict(x.split("=", 1) for x in f[1:])
        assert os.path.exists(os.path.join(ROOT, "gated_delta_rule_kk_gb300", "csrc", kv["source"]))
        assert len(kv["sha"]) == 12 and int(kv["sha"], 16) >= 0
        assert float(kv["bytes_per_launch"]) > 0
