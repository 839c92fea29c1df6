"""The multi-rank host logic of bench.py on the CPU: two gloo ranks (one
process per rank, as the launcher starts them), each with its own replica
time; both see the slowest rank's time, and the whole-job rate counts every
rank's rows over that time."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 17.25][rank]
        got = bench.max_over_ranks(ms, world)
        q.put((rank, got, bench.whole_job_rate(4096, 10, world, got)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [17.25, 17.25]
    assert res[0][2] == pytest.approx(4096 * 10 * 2 / 17.25e-3)


def test_single_rank_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(4096, 4, 1, 2.0) == pytest.approx(4096 * 4 / 2e-3)
