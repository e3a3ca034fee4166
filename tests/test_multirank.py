"""The multi-rank bench path on CPU (gloo, world size 2): each rank runs its own copy of the workload (the
sequences are independent problems, so there is no data-path collective); the timed region is the maximum
over ranks and the reported value aggregates the tokens of every rank."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [12.5, 20.0][rank]
    total = bench.max_over_ranks(local, dist, "cpu")
    value = bench.whole_job_value(8192, 10, world, total)
    q.put((rank, total, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_takes_the_max_and_aggregates_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, total, value in res:
        assert total == 20.0
        assert value == pytest.approx(8192 * 10 * 2 / 0.020)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_value(100, 4, 1, 2.0) == pytest.approx(200000.0)
