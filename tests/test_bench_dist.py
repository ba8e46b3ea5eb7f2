"""Multi-rank bench logic on CPU (gloo, world size 2): the job's step time is
the slowest rank's and the value counts every rank's work."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 * (rank + 1)                       # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world, device="cpu")
    value = bench.whole_job_tflops(1e12, world, worst)
    q.put((rank, worst, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, value in res:
        assert worst == 20.0                      # slowest rank's time on every rank
        assert value == pytest.approx(2 * 1e12 / 0.020 / 1e12)  # both ranks' work


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)
