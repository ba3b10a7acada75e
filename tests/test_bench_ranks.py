"""The benchmark's multi-rank accounting on CPU (gloo, two ranks): every rank times the same steps of its own
replica, the job's time is the slowest rank's, and the job's throughput counts every rank's units."""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    t_local = [12.0, 30.0][rank]  # ms: rank 1 is the slow one
    value, t_ms = bench.job_rate(units_per_rank=100, t_local_ms=t_local, world=world, device="cpu")
    out[rank] = (value, t_ms)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_every_rank_units():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        value, t_ms = res[rank]
        assert t_ms == 30.0
        assert value == pytest.approx(200 / 0.030)


def test_one_rank_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_rate(100, 25.0, 1, "cpu") == (100 / 0.025, 25.0)
