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


def test_traffic_summaries_match_their_kernel_sources():
    """Every committed ncu traffic summary that the benchmark reads names a kernel source whose current
    sha256 it was taken on (a stale summary would report no traffic), and the lookup is keyed by kernel,
    workload and batch: another workload or batch of the same kernel gets none."""
    sys.path.insert(0, ROOT)
    import bench

    src = os.path.join(ROOT, "expert_offload_moe_gb300", "csrc", "moe_decode_tc.cu")
    for (kernel, workload, M), fname in bench.TRAFFIC_SUMMARIES.items():
        got = bench.traffic_for(src, kernel, workload, M)
        assert got is not None and got > 0, fname
    assert bench.traffic_for(src, "ffn_tc_kernel", "gptoss20b_h2880_e32k4_resident_m1", 8) is None
    assert bench.traffic_for(src, "gateup_tc_kernel", "gptoss20b_h2880_e32k4_resident_m1", 1) is None
