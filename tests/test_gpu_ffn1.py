"""One-token decode in one launch (gate/up, SiLU·up, down and combine in one kernel) against the oracle,
beside the two-launch path, on shapes that cover its cases: K splits in a cluster or none, ragged hidden and
intermediate tiles, H tiles per CTA odd, even, and more than the pipeline holds, some or all routes cold."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import compare_routing, compare_values, route_arrays  # noqa: E402

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
GPTOSS = W["gptoss20b_h2880_e32k4_resident_m1"]
E512 = W["e512k10_h2048_i512_s256_m1"]
# (workload, layer): H tiles per CTA and K splits differ between them
SHAPES = [
    (W["tiny_h256_i128_e16k2"], 0),                                    # 1 split, 2 H tiles
    (synth.Workload("h512_i256_e64k8", 1, 512, 256, 64, 8, 64, (1,), 1), 0),   # 1 split, 4 H tiles
    (synth.Workload("h1024_i192_e16k2", 1, 1024, 192, 16, 2, 16, (1,), 1), 0),  # ragged I tile, 2 splits
    (GPTOSS, 5),                                                       # 3 splits, ragged H and I, 8/8/7 H tiles
    (E512, 2),                                                         # 4 splits, 4 H tiles each, bias
]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def forward(lay, x_bits, out_f32):
    M = x_bits.shape[0]
    x = stack.bf16_tensor(x_bits)
    out = torch.empty((M, x_bits.shape[1]), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    res = lay.route(x, M)
    lay.forward_slots(x, out, M)
    torch.cuda.synchronize()
    lay.check_error()
    return res, out.float().cpu().numpy()


def oracle_out(li, x_bits, e2s):
    w = li.w
    return oracle.moe_layer(x_bits, li.Wr, li.bias, li.bank.numpy(), e2s, w.top_k, w.hidden, w.inter)


@pytest.mark.parametrize("shape", range(len(SHAPES)))
@pytest.mark.parametrize("out_f32", [False, True])
def test_one_launch_matches_oracle_beside_two_launches(shape, out_f32):
    w, layer = SHAPES[shape]
    li = stack.LayerInputs(w, layer)
    x = synth.activations(0, layer, 90 + shape, 1, w.hidden)
    o = oracle_out(li, x, li.e2s)
    lay = li.make_layer(max_tokens=8, out_f32=out_f32)
    outs = {}
    for fused in (True, False, True):
        lay.decode_fusion(fused)
        res, out = forward(lay, x, out_f32)
        g = route_arrays(res, w.experts, w.top_k)
        excl = compare_routing(g, o, o["logits"], w.top_k, li.e2s)
        compare_values(out, o["out_f32"], out_f32, exclude=excl)
        if fused in outs:  # the arrival counters were reset: a second call gives the same bits
            assert np.array_equal(outs[fused], out)
        outs[fused] = out
    lay.close()


def test_one_launch_with_some_routes_cold():
    # 8 of 32 experts resident: fewer active units than the launch has room for
    w = synth.Workload("gptoss_s8", 1, GPTOSS.hidden, GPTOSS.inter, 32, 4, 8, (1,), 1)
    li = stack.LayerInputs(w, 1, e2s=np.arange(8).tolist() + [-1] * 24)
    hits = 0
    for s in range(4):
        x = synth.activations(0, 1, 120 + s, 1, w.hidden)
        ids = oracle_out(li, x, li.e2s)["ids"][0]  # routing does not depend on the map
        nh = 1 + s % 3  # 1-3 of the token's 4 experts hot
        e2s = np.full(32, -1, dtype=np.int32)
        e2s[ids[:nh]] = np.arange(nh)
        e2s[[e for e in range(32) if e not in ids][:8 - nh]] = np.arange(nh, 8)
        li.e2s = e2s
        o = oracle_out(li, x, e2s)
        lay = li.make_layer(max_tokens=8, out_f32=True)
        lay.decode_fusion(True)
        res, out = forward(lay, x, True)
        g = route_arrays(res, w.experts, w.top_k)
        excl = compare_routing(g, o, o["logits"], w.top_k, e2s)
        compare_values(out, o["out_f32"], True, exclude=excl)
        hits += int(g["counts"][0])
        lay.close()
    assert hits == 1 + 2 + 3 + 1


def test_one_launch_all_cold_outputs_zero():
    w = synth.Workload("gptoss_cold", 1, GPTOSS.hidden, GPTOSS.inter, 32, 4, 4, (1,), 1)
    li = stack.LayerInputs(w, 2, e2s=np.arange(4).tolist() + [-1] * 28)
    x = synth.activations(0, 2, 130, 1, w.hidden)
    ids = set(oracle_out(li, x, li.e2s)["ids"][0].tolist())
    e2s = np.full(32, -1, dtype=np.int32)
    e2s[[e for e in range(32) if e not in ids][:4]] = np.arange(4)  # resident experts the token does not use
    li.e2s = e2s
    lay = li.make_layer(max_tokens=8, out_f32=True)
    lay.decode_fusion(True)
    out_dev = torch.full((1, w.hidden), 7.0, dtype=torch.float32, device="cuda")
    xd = stack.bf16_tensor(x)
    res = lay.route(xd, 1)
    lay.forward_slots(xd, out_dev, 1)
    torch.cuda.synchronize()
    lay.check_error()
    g = route_arrays(res, w.experts, w.top_k)
    assert g["counts"][0] == 0 and g["counts"][1] == 4
    assert torch.count_nonzero(out_dev).item() == 0
    lay.close()


def test_one_launch_placement_gives_bit_identical_output():
    # sums run in expert order whatever slots the experts sit in
    w = GPTOSS
    x = synth.activations(0, 4, 140, 1, w.hidden)
    outs = []
    for perm_seed in (0, 1):
        e2s = np.random.default_rng(perm_seed).permutation(32).astype(np.int32)
        li = stack.LayerInputs(w, 4, e2s=e2s)
        lay = li.make_layer(max_tokens=8, out_f32=True)
        lay.decode_fusion(True)
        outs.append(forward(lay, x, True)[1])
        lay.close()
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("M", [1, 8])
def test_decode_route_pads_the_active_slots_with_minus_one(M):
    """A decode route writes act_slot[n_active .. min(S, M k)) = -1 (the expert kernels launched for up to
    min(S, M k) experts take an entry of -1 as 'no expert here'), on every call: a call with more active
    experts followed by one with fewer leaves no stale slot behind."""
    from parity import dev_i32

    w = synth.WORKLOADS["e512k10_h2048_i512_s256_m1"]
    li = stack.LayerInputs(w, 1)
    lay = li.make_layer(max_tokens=8)
    try:
        cap = min(w.slots, M * w.top_k)
        n_seen = set()
        for c in range(6):
            res = lay.route(stack.bf16_tensor(synth.activations(0, 1, 400 + c, M, w.hidden)), M)
            g = route_arrays(res, w.experts, w.top_k)
            n_act = int(g["counts"][2])
            n_seen.add(n_act)
            slots = dev_i32(res.act_slot, cap)
            assert np.array_equal(slots[:n_act], g["act_slot"])
            assert (slots[:n_act] >= 0).all() and (slots[n_act:] == -1).all()
        assert len(n_seen) > 1  # the calls had different numbers of active experts
    finally:
        lay.close()
