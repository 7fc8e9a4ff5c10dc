"""The N>1 bench path on CPU: two gloo ranks, each its own replica; the job's rate uses the
slowest rank's time and every rank's work.  No GPU and no data-path collective."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    slow = bench.max_over_ranks(local_ms[rank], world, "cpu")
    rate = bench.whole_job_rate(1000, world, slow, 1.0)
    q.put((rank, slow, rate))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    local_ms = [2.0, 5.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, rate in got:
        assert slow == 5.0                      # max over ranks
        assert rate == pytest.approx(1000 * 2 / 5e-3)  # both ranks' work / slowest time


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(10, 1, 2.0, 1e-3) == pytest.approx(5.0)
