"""Next-layer prefetch (tinyserve README "How it works" 4, FATE) on the GPU: the layer's routing of another
layer's input picks the experts to copy in, the map follows the oracle's prefetch step, the copied slots hold
the bank's records, and a route of that same input then finds its experts resident."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import NEAR_TIE, compare_routing, compare_values, dev_bytes, route_arrays  # noqa: E402

pytestmark = pytest.mark.gpu

W6 = synth.Workload("tiny_s6_prefetch", 1, 256, 128, 16, 2, 6, (2,), 1)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def clear_inputs(li, M, first_step):
    """A batch whose routing has no near tie (so the GPU's prediction equals the oracle's)."""
    for s in range(first_step, first_step + 50):
        x = synth.activations(0, 0, s, M, li.w.hidden)
        lg = oracle.router_logits(x, li.Wr, li.bias).astype(np.float64)
        srt = -np.sort(-lg, axis=1)
        if np.all(srt[:, li.w.top_k - 1] - srt[:, li.w.top_k] >= NEAR_TIE):
            return x
    raise AssertionError("no clear batch found")


@pytest.mark.parametrize("R", [1, 2, 4])
def test_prefetch_follows_oracle_and_makes_routes_hot(R):
    e2s0 = np.full(16, -1, dtype=np.int32)
    e2s0[[0, 3, 5, 8, 11, 14]] = np.arange(6)
    li = stack.LayerInputs(W6, 0, e2s=e2s0)
    lay = li.make_layer(max_tokens=8, out_f32=True, max_refills=R)
    M = 2
    x = clear_inputs(li, M, 300 + R)
    pred = oracle.moe_layer(x, li.Wr, li.bias, li.bank.numpy(), e2s0, W6.top_k, W6.hidden, W6.inter)["hist"]
    want_pairs, want_map = oracle.prefetch_step(np.zeros(16), np.full(16, -1, dtype=np.int64), e2s0, 6, pred, R)
    xd = stack.bf16_tensor(x)
    n = lay.prefetch(xd, M)
    torch.cuda.synchronize()
    assert n == len(want_pairs)
    m = lay.get_map()
    assert np.array_equal(m, want_map)
    bank = li.bank.numpy()
    for e, s, _ in want_pairs:
        assert np.array_equal(dev_bytes(lay.slot_ptr(s), W6.expert_bytes), bank[e])
    # the same input now routes to resident experts wherever the budget allowed
    out = torch.empty((M, W6.hidden), dtype=torch.float32, device="cuda")
    res = lay.route(xd, M)
    lay.forward_slots(xd, out, M)
    torch.cuda.synchronize()
    g = route_arrays(res, W6.experts, W6.top_k)
    o = oracle.moe_layer(x, li.Wr, li.bias, bank, m, W6.top_k, W6.hidden, W6.inter)
    compare_routing(g, o, o["logits"], W6.top_k, m)
    compare_values(out.cpu().numpy(), o["out_f32"], True)
    # the route is the prediction (same input, no near tie): its cold experts are the predicted ones left out
    assert set(g["cold_expert"].tolist()) == {int(e) for e in np.nonzero(pred)[0] if want_map[e] < 0}
    assert n == 0 or len(g["cold_expert"]) < sum(int(pred[e]) for e in range(16) if e2s0[e] < 0)
    lay.close()


def test_prefetch_with_every_expert_resident_does_nothing():
    li = stack.LayerInputs(synth.WORKLOADS["tiny_h256_i128_e16k2"], 0)
    lay = li.make_layer(max_tokens=8)
    assert lay.prefetch(stack.bf16_tensor(synth.activations(0, 0, 1, 1, 256)), 1) == 0
    lay.close()


def test_prefetch_refused_while_the_device_table_owns_the_slots():
    e2s0 = np.full(16, -1, dtype=np.int32)
    e2s0[:6] = np.arange(6)
    li = stack.LayerInputs(W6, 0, e2s=e2s0)
    lay = li.make_layer(max_tokens=8)
    lay.set_device_cache(True)
    with pytest.raises(moe.MoeError) as ei:
        lay.prefetch(stack.bf16_tensor(synth.activations(0, 0, 2, 1, 256)), 1)
    assert ei.value.code == moe.MOE_ESTATE
    with pytest.raises(moe.MoeError) as ei:
        lay.set_device_cache(False)
        lay.prefetch(stack.bf16_tensor(synth.activations(0, 0, 2, 9, 256)), 9)  # prefill sizes are not predicted
    assert ei.value.code == moe.MOE_EINVAL
    lay.close()
