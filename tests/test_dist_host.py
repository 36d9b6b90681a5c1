"""The N > 1 path of bench.py on the CPU: two processes over gloo (the GPU
run uses NCCL with the same calls).  Each GPU runs an independent replica of
the round; the job time is the slowest rank's, the value counts every rank's
bytes, and only rank 0 prints."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [3.5, 4.25][rank]                    # rank 1 is the slower replica
        t_max = bench.reduce_max(per_rank_ms, world, "cpu")
        dist.barrier()
        # the reference arm: rank 0 alone runs and prints; other ranks return at once
        printed = ""
        if rank != 0:
            buf = io.StringIO()
            with redirect_stdout(buf):
                bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "gpus": world})())
            printed = buf.getvalue()
        out.put((rank, t_max, bench.dist_env(), printed))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_only_rank0_prints():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [4.25, 4.25]              # both ranks agree on the max
    assert [g[2] for g in got] == [(0, 2, 0), (1, 2, 1)]    # RANK / WORLD_SIZE / LOCAL_RANK read from the env
    assert got[1][3] == ""                                  # rank 1 printed nothing


def test_whole_job_value_counts_every_rank():
    import bench
    one = bench.whole_job_gbs(6.8e9, 10, 1, 10.0)
    two = bench.whole_job_gbs(6.8e9, 10, 2, 10.0)
    assert one == pytest.approx(6800.0)
    assert two == pytest.approx(2 * one)                    # weak scaling: per-rank work fixed
    assert bench.reduce_max(1.5, 1) == 1.5                  # one process: no collective
