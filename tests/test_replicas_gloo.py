"""The replica path of bench.py (N > 1, one process per GPU, no collective on the data path):
the timed region's times are reduced to their maximum over the ranks, so the reported rate is
the slowest replica's. Checked with two gloo ranks on the CPU."""
import multiprocessing as mp
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    q.put((rank, bench.max_over_ranks([10.0 + rank, 5.0 - rank, 7.0 * (rank + 1)], "cpu", world)))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_times_are_the_maximum_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [11.0, 5.0, 14.0]


def test_single_rank_keeps_its_values():
    import bench
    assert bench.max_over_ranks([1.5, 2.0], "cpu", 1) == [1.5, 2.0]
