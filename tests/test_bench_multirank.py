"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks, max-over-ranks job time
and whole-job throughput (the path torch.distributed.run takes with --gpus 2)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.5, 4.0][rank]                     # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms, dist, "cpu")
    rate = bench.job_rate(100.0, world, ms_max * 1e-3)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms_max, rate, bench.dist_env()))


@pytest.mark.timeout(120)
def test_two_rank_max_and_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, ms_max, rate, env in res:
        assert ms_max == 4.0                  # the slowest rank's time
        assert rate == pytest.approx(2 * 100.0 / 4e-3)
        assert env == (2, rank, 0)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_rate(10.0, 1, 2.0) == 5.0
