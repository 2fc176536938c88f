"""The multi-rank host logic of bench.py with two gloo ranks on the CPU: every
rank reports the slowest rank's times, and the whole-job rate counts the rows
of every rank in that time (one replica per GPU, no collective on the path)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms on the device and 10 - r s end to end
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist, device="cpu")
        q.put((rank, got, bench.job_rate(world, 4, 10, got[0] / 1e3)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [2.0, 10.0]           # max over ranks of each value
        assert rate == 2 * 4 * 10 / 2e-3   # both ranks' rows in the slowest rank's time


def test_one_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]
    assert bench.job_rate(1, 8, 16, 0.5) == 256.0
