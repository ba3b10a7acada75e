"""Expert-parallel sharding on CPU ranks (gloo): the partition of the experts over the ranks, and two ranks whose
rank-local results (the library's host expert FFN over each rank's own shard) summed by one all-reduce give the
whole layer within the 2e-3 metric of the oracle (xinfer docs "Options": each rank loads and offloads its own
expert shard; NCCL combines the rank-local MoE results).  No GPU: one GPU per rank is not available here."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    moe_build.build()
    moe.lib()


@pytest.mark.parametrize("E,world", [(16, 2), (32, 4), (512, 8), (7, 3), (5, 5), (1, 1)])
def test_partition_gives_every_expert_to_exactly_one_rank(E, world):
    owner = np.full(E, -1)
    counts = []
    for r in range(world):
        e2s, first, count = moe.ep_local_map(E, world, r)
        own = np.flatnonzero(e2s >= 0)
        assert np.array_equal(own, np.arange(first, first + count))  # contiguous
        assert np.array_equal(e2s[own], np.arange(count))  # slots 0..count-1 in ascending id order
        assert np.all(owner[own] == -1)
        owner[own] = r
        counts.append(count)
    assert np.all(owner >= 0) and max(counts) - min(counts) <= 1
    assert np.all(np.diff(owner) >= 0)  # rank r's range comes before rank r + 1's


def test_partition_rejects_bad_arguments():
    e2s = np.zeros(4, dtype=np.int32)
    for E, world, rank in [(0, 1, 0), (4, 0, 0), (4, 5, 0), (4, 2, 2), (4, 2, -1)]:
        assert moe.lib().moe_ep_local_map(E, world, rank, e2s.ctypes.data_as(moe._P), None, None) == moe.MOE_EINVAL


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    from expert_offload_moe_gb300 import synth

    H, I, E, k, M = 256, 128, 16, 2, 6
    Wr = synth.router_weights(4, 0, E, H)
    b = synth.router_bias(4, 0, E, 0.25)
    bank = synth.expert_records(4, 0, E, H, I)
    x = synth.activations(4, 0, 1, M, H)
    return H, I, E, k, M, Wr, b, bank, x


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from expert_offload_moe_gb300 import moe as m
    from expert_offload_moe_gb300 import stack

    H, I, E, k, M, Wr, b, bank, x = _case()
    # the replicated router: every rank routes every token the same way (the GPU route kernel on GPU ranks; the
    # oracle's routing stands in for it here, where the ranks have no GPU)
    ids, w = oracle.topk_softmax(oracle.router_logits(x, Wr, b), k)
    e2s, first, count = m.ep_local_map(E, world, rank)
    part = torch.from_numpy(stack.ep_host_partial(bank, e2s, ids, w, x, H, I))
    out[(rank, "own")] = sorted(set(ids[np.isin(ids, np.arange(first, first + count))].tolist()))
    dist.all_reduce(part)  # one sum all-reduce of out[M, H]
    out[(rank, "out")] = part.numpy().copy()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_shards_all_reduced_give_the_whole_layer(world):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from parity import compare_values

    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    H, I, E, k, M, Wr, b, bank, x = _case()
    o = oracle.moe_layer(x, Wr, b, bank, np.arange(E, dtype=np.int32), k, H, I)
    for r in range(world):
        assert np.array_equal(res[(r, "out")], res[(0, "out")])  # every rank holds the same combined output
    assert all(len(res[(r, "own")]) > 0 for r in range(world))  # each shard had routes of its own
    compare_values(res[(0, "out")], o["out_f32"], True)
