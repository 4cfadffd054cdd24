"""The replica (N > 1) path of bench.py on CPU: two gloo ranks, max-over-ranks
interval and whole-job throughput."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_setup()[:2] == (world, rank)
    ms, value = bench.aggregate(10.0 + 5.0 * rank, 897.1e9 * 20, world, dist, "cpu")
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_max_interval():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    assert set(out.keys()) == {0, 1}
    for r in range(world):
        ms, value = out[r]
        assert ms == 15.0
        assert value == pytest.approx(897.1e9 * 20 * 2 / 15e-3 / 1e12)


def test_single_rank_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(5.0, 1e12, 1)
    assert ms == 5.0 and value == pytest.approx(200.0)
