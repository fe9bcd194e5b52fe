"""The bench's multi-rank paths on CPU (gloo, world size 2; no GPU needed).

Each rank of `bench.py --gpus N` runs an independent replica of the mixer
(there is no collective on the data path); the ranks only agree on the job's
time, the slowest rank's, and count every rank's tokens.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [100.0, 250.0][rank]
        total_ms, value = bench.replica_throughput(torch, local_ms, 2048, 10, world, dist, "cpu")
        out[rank] = (total_ms, value)
    finally:
        dist.destroy_process_group()


def test_replica_throughput_takes_the_slowest_rank_and_counts_every_rank():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        total_ms, value = res[rank]
        assert total_ms == 250.0
        assert value == pytest.approx(2 * 2048 * 10 / 0.25)


def test_replica_throughput_single_rank_needs_no_process_group():
    import bench

    assert bench.replica_throughput(torch, 50.0, 100, 4, 1) == (50.0, pytest.approx(100 * 4 / 0.05))


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` launched like the N-GPU bench: rank 0 times the
    oracle and prints one JSON line; the other rank exits 0 without output."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--ref-budget", "8"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
