"""Multi-process host logic of bench.py on CPU: two gloo ranks (the GPU runs use one process per
GPU with the same functions over NCCL). Each rank is an independent replica, so the only
cross-rank step is taking the slowest rank's time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    mine = 10.0 + 5.0 * rank          # rank 1 is the slower one
    slowest = bench.max_over_ranks(mine, dist)
    rate = bench.whole_job_rate(16384 * 4, world, slowest / 1e3)
    out.put((rank, slowest, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
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
    for rank, slowest, rate in res:
        assert slowest == 15.0
        assert abs(rate - 2 * 16384 * 4 / 0.015) < 1e-6


def test_single_process_aggregation_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.whole_job_rate(100, 1, 0.5) == 200.0
