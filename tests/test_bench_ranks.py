"""bench.py's multi-rank aggregation on CPU (two gloo ranks): every rank gets the
slowest rank's time, and the whole-job rate counts all ranks' work."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, rate = bench.whole_job(1.0 + rank, 1e6, dist)  # rank r takes 1 + r ms for 1e6 units
    q.put((rank, ms, rate))
    dist.destroy_process_group()


def test_two_ranks_take_the_max_time_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in out:
        assert ms == 2.0                       # the slower rank's time, on every rank
        assert rate == pytest.approx(2e6 / 2e-3)  # both ranks' units over that time


def test_single_process_is_its_own_job():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms, rate = bench.whole_job(4.0, 8e6, None)
    assert ms == 4.0 and rate == pytest.approx(8e6 / 4e-3)
