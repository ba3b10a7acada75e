"""GPU path (through the C ABI) against the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import (compare_routing, compare_values, outlier_tokens, route_arrays, route_weight_rtol,  # noqa: E402
                    combine_with_weights, two_term_e4m3_residual)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
TINY = W["tiny_h256_i128_e16k2"]
GPTOSS = W["gptoss20b_h2880_e32k4_resident_m1"]
E512 = W["e512k10_h2048_i512_s256_m1"]
E512_S384 = W["e512k10_h2048_i512_s384_m4m8"]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def run_layer(li, x_bits, M, out_f32=False, layer=None):
    """Routes and forwards M tokens on the GPU; returns (route arrays, output)."""
    w = li.w
    lay = layer or li.make_layer(max_tokens=max(M, 8), out_f32=out_f32)
    x = stack.bf16_tensor(x_bits)
    out = torch.empty((M, w.hidden), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    res = lay.route(x, M)
    lay.forward_slots(x, out, M)
    torch.cuda.synchronize()
    lay.check_error()
    g = route_arrays(res, w.experts, w.top_k)
    o = out.float().cpu().numpy()
    if layer is None:
        lay.close()
    return g, o


def oracle_layer(li, x_bits, e2s):
    w = li.w
    return oracle.moe_layer(x_bits, li.Wr, li.bias, li.bank.numpy(), e2s, w.top_k, w.hidden, w.inter)


def check_case(li, x_bits, out_f32, e2s=None, w_rtol=None):
    e2s = li.e2s if e2s is None else e2s
    M = x_bits.shape[0]
    g, out = run_layer(li, x_bits, M, out_f32=out_f32)
    o = oracle_layer(li, x_bits, e2s)
    assert g["mirror_ok"]
    excl = compare_routing(g, o, o["logits"], li.w.top_k, e2s, w_rtol=w_rtol)
    worst = compare_values(out, o["out_f32"], out_f32, exclude=excl)
    return g, o, out, worst, excl


# ---------------------------------------------------------------- tiny layer


@pytest.mark.parametrize("M", [1, 2, 3, 8])
@pytest.mark.parametrize("out_f32", [False, True])
def test_tiny_all_resident(M, out_f32):
    li = stack.LayerInputs(TINY, 0)
    x = synth.activations(0, 0, 10 + M, M, TINY.hidden)
    check_case(li, x, out_f32)


@pytest.mark.parametrize("shape,M", [(TINY, 1), (TINY, 8), (GPTOSS, 1), (GPTOSS, 8)])
@pytest.mark.parametrize("out_f32", [False, True])
def test_outlier_blocks_reach_the_inexact_activation_split(shape, M, out_f32):
    """Activations with outliers inside their 32-element blocks (ranges up to 2^18), where the two E4M3 terms
    of x on the tensor-core path are no longer exact, and h spans a wide range within its blocks: every
    output value within the 2e-3 metric, as for N(0, 1) inputs.  An outlier makes the fp32 partial sums of
    the token's logits, and so their rounding in either summation order, ~20x larger: the routing weights
    are compared with the oracle's within each token's own bound (route_weight_rtol), and the outputs with
    the oracle's expert outputs combined by the GPU's routing weights (otherwise a weight difference of a
    few 1e-5, times a large w y where experts' contributions cancel, decides the comparison)."""
    x = outlier_tokens(3, max(M, 3), shape.hidden)[:M] if M > 1 else outlier_tokens(3, 1, shape.hidden)
    assert np.any(two_term_e4m3_residual(x) != 0)  # the case really is the inexact one
    li = stack.LayerInputs(shape, 0)
    w = li.w
    rt = route_weight_rtol(x, li.Wr, li.bias)
    g, out = run_layer(li, x, M, out_f32=out_f32)
    o = oracle_layer(li, x, li.e2s)
    assert g["mirror_ok"]
    excl = compare_routing(g, o, o["logits"], w.top_k, li.e2s, w_rtol=rt)
    bank = li.bank.numpy()
    ys = np.stack([np.stack([oracle.expert_ffn(bank[e], w.hidden, w.inter, x[t]) for e in g["ids"][t]])
                   for t in range(M)])
    compare_values(out, combine_with_weights(g["ids"], g["w"], ys), out_f32, exclude=excl)


@pytest.mark.parametrize("M", [1, 5, 8])
def test_tiny_partial_map_returns_cold_routes(M):
    e2s = np.full(TINY.experts, -1, dtype=np.int32)
    e2s[[1, 4, 6, 9, 11, 15]] = np.arange(6)
    w = synth.Workload("tiny_s6", 1, 256, 128, 16, 2, 6, (M,), 1)
    li = stack.LayerInputs(w, 0, e2s=e2s)
    x = synth.activations(0, 0, 20 + M, M, w.hidden)
    g, o, out, _, excl = check_case(li, x, True, e2s)
    if M > 1:
        assert g["counts"][1] > 0  # some routes are cold


@pytest.mark.parametrize("M", [1, 8])
def test_narrow_expert_takes_the_cuda_core_kernels(M):
    # I = 64 has no full 128-column tile, so this shape runs the CUDA-core decode kernels
    w = synth.Workload("tiny_i64", 1, 256, 64, 16, 2, 16, (M,), 1)
    li = stack.LayerInputs(w, 0)
    x = synth.activations(0, 0, 70 + M, M, w.hidden)
    check_case(li, x, M == 8)


def test_tiny_all_cold_outputs_zero():
    w = synth.Workload("tiny_cold", 1, 256, 128, 16, 2, 2, (3,), 1)
    e2s = np.full(16, -1, dtype=np.int32)
    li = stack.LayerInputs(w, 0, e2s=e2s)
    x = synth.activations(0, 0, 30, 3, 256)
    g, out = run_layer(li, x, 3, out_f32=True)
    assert g["counts"][0] == 0 and g["counts"][1] == 6 and np.all(out == 0)


def test_slot_permutation_gives_bit_identical_output():
    # placement must not change the result (xinfer docs: byte-identical output for every offload fraction)
    w = synth.Workload("tiny_perm", 1, 256, 128, 16, 2, 16, (8,), 1)
    x = synth.activations(0, 0, 40, 8, 256)
    outs = []
    for perm_seed in (0, 1, 2):
        e2s = np.random.default_rng(perm_seed).permutation(16).astype(np.int32)
        li = stack.LayerInputs(w, 0, e2s=e2s)
        for out_f32 in (False, True):
            _, out = run_layer(li, x, 8, out_f32=out_f32)
            outs.append((out_f32, out))
    for f32 in (False, True):
        ref = [o for f, o in outs if f == f32]
        assert all(np.array_equal(ref[0], o) for o in ref[1:])


def test_repeated_calls_reuse_scratch():
    li = stack.LayerInputs(TINY, 0)
    lay = li.make_layer(max_tokens=8)
    for s, M in enumerate([1, 8, 3, 1, 8]):
        x = synth.activations(0, 0, 50 + s, M, TINY.hidden)
        g, out = run_layer(li, x, M, layer=lay)
        o = oracle_layer(li, x, li.e2s)
        excl = compare_routing(g, o, o["logits"], TINY.top_k, li.e2s)
        compare_values(out, o["out_f32"], False, exclude=excl)
    lay.close()


# ------------------------------------------------------------ full-size shapes


@pytest.mark.parametrize("layer", [0, 23])
def test_gptoss_shape_layer_m1(layer):
    li = stack.LayerInputs(GPTOSS, layer)
    x = synth.activations(0, layer, 0, 1, GPTOSS.hidden)
    g, o, out, worst, excl = check_case(li, x, False)
    assert g["counts"][2] == 4 and not excl


def test_gptoss_shape_batch_m8_f32():
    li = stack.LayerInputs(GPTOSS, 7)
    x = synth.activations(0, 7, 3, 8, GPTOSS.hidden)
    check_case(li, x, True)


def test_e512_s256_layer_m1():
    li = stack.LayerInputs(E512, 3)
    x = synth.activations(0, 3, 0, 1, E512.hidden)
    check_case(li, x, False)


@pytest.mark.parametrize("M", [4, 8])
def test_e512_s384_speculative_batches(M):
    li = stack.LayerInputs(E512_S384, 5)
    x = synth.activations(0, 5, 1, M, E512_S384.hidden)
    check_case(li, x, True)
    check_case(li, x, False)


def test_graph_replay_matches_eager_on_full_stack_sample():
    # the launch configuration the benchmark times: all layers in one CUDA graph
    st = stack.DecodeStack(GPTOSS, M=1, n_layers=3, n_inputs=2)
    st.capture()
    st.replay(1)
    torch.cuda.synchronize()
    g_out = st.out.float().cpu().numpy()
    for l in range(3):
        li = st.inputs[l]
        o = oracle_layer(li, st.x_host[1, l], li.e2s)
        compare_values(g_out[l], o["out_f32"], False)
    st.close()


# --------------------------------------------------------------- error paths


def test_pageable_host_bank_is_rejected():
    w = TINY
    Wr = torch.from_numpy(synth.router_weights(0, 0, w.experts, w.hidden)).cuda()
    bank = torch.zeros((w.experts, w.expert_bytes), dtype=torch.uint8)  # not pinned
    with pytest.raises(moe.MoeError) as ei:
        moe.Layer(w.hidden, w.inter, w.experts, w.top_k, w.slots, 8, Wr, None, bank, np.arange(16))
    assert ei.value.code == moe.MOE_EINVAL


def test_bad_descriptors_are_rejected():
    li = stack.LayerInputs(TINY, 0)
    Wr = torch.from_numpy(li.Wr).cuda()
    for kw, e2s in [(dict(hidden=250), np.arange(16)), (dict(top_k=0), np.arange(16)),
                    (dict(num_slots=1), np.arange(16)), (dict(), np.array([0, 0] + [-1] * 14))]:
        args = dict(hidden=256, inter=128, num_experts=16, top_k=2, num_slots=16, max_tokens=8)
        args.update(kw)
        with pytest.raises(moe.MoeError) as ei:
            moe.Layer(args["hidden"], args["inter"], args["num_experts"], args["top_k"], args["num_slots"],
                      args["max_tokens"], Wr, None, li.bank, e2s)
        assert ei.value.code == moe.MOE_EINVAL


def test_call_order_and_sizes_are_checked():
    li = stack.LayerInputs(TINY, 0)
    lay = li.make_layer(max_tokens=4)
    x = stack.bf16_tensor(synth.activations(0, 0, 60, 4, 256))
    out = torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        lay.forward_slots(x, out, 4)
    assert ei.value.code == moe.MOE_ESTATE
    with pytest.raises(moe.MoeError) as ei:
        lay.route(x, 5)
    assert ei.value.code == moe.MOE_EINVAL
    lay.route(x, 4)
    with pytest.raises(moe.MoeError) as ei:
        lay.forward_slots(x, out, 3)
    assert ei.value.code == moe.MOE_ESTATE
    lay.forward_slots(x, out, 4)
    torch.cuda.synchronize()
    lay.close()
