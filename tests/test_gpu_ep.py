"""Expert-parallel shards on one GPU: each rank's shard layer (its contiguous range of experts resident, the
router replicated) computes exactly the routes to its own experts and returns the others as its cold list, and
the ranks' fp32 outputs summed (what the one all-reduce does across GPUs) equal the whole layer within the
2e-3 metric of the oracle.  The ranks run one after another here; nothing waits across them."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import compare_routing, compare_values, route_arrays  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


@pytest.mark.parametrize("name,world,M", [("tiny_h256_i128_e16k2", 2, 4), ("gptoss20b_h2880_e32k4_resident_m1", 2, 1),
                                          ("gptoss20b_h2880_e32k4_resident_m1", 4, 8),
                                          ("e512k10_h2048_i512_s256_m1", 8, 1)])
def test_shards_sum_to_the_whole_layer(name, world, M):
    w = synth.WORKLOADS[name]
    li = stack.LayerInputs(w, 1, e2s=np.arange(w.experts, dtype=np.int32))
    x_bits = synth.activations(0, 1, 50, M, w.hidden)
    x = stack.bf16_tensor(x_bits)
    o = oracle.moe_layer(x_bits, li.Wr, li.bias, li.bank.numpy(), np.arange(w.experts, dtype=np.int32), w.top_k,
                         w.hidden, w.inter)
    total = torch.zeros((M, w.hidden), dtype=torch.float32, device="cuda")
    n_hot = 0
    for r in range(world):
        sh = stack.EPShard(li, world, r)
        try:
            out = torch.empty((M, w.hidden), dtype=torch.float32, device="cuda")
            res = sh.forward(x, M, out, reduce=False)
            g = route_arrays(res, w.experts, w.top_k)
            own = (np.arange(w.experts) >= sh.first) & (np.arange(w.experts) < sh.first + sh.count)
            assert np.all(own[g["hot_expert"]]) and not np.any(own[g["cold_expert"]])
            os_ = oracle.compact(o["ids"], o["w"], sh.e2s)  # the oracle's compaction under the shard's map
            os_.update(ids=o["ids"], w=o["w"])
            compare_routing(g, os_, o["logits"], w.top_k, sh.e2s)  # same routing as the whole layer
            n_hot += int(g["counts"][0])
            total += out
        finally:
            sh.close()
    torch.cuda.synchronize()
    assert n_hot == M * w.top_k  # every route is some rank's hot route
    compare_values(total.cpu().numpy(), o["out_f32"], True)
