"""bench.py's multi-process arithmetic with world_size 2 gloo ranks on CPU:
max-over-ranks timing, whole-job throughput of replicas, and the reference
arm doing its work on rank 0 only."""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [120.0, 150.0][rank]            # rank 1 is the slow one
    mx = bench.max_over_ranks(elapsed)
    value = bench.whole_job_steps_per_s(world, 300, mx)
    dist.barrier()
    q.put((rank, mx, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, value in res:
        assert mx == 150.0                    # every rank reports the slowest rank's time
        assert abs(value - 2 * 300 / 0.150) < 1e-9


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_steps_per_s(1, 100, 50.0) == 2000.0


def test_reference_arm_nonzero_rank_does_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.bench_reference(bench.parse_args(["--impl", "reference", "--steps", "1"]))
    assert capsys.readouterr().out == ""
