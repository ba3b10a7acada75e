"""NVFP4 experts (E2M1 codes, one E4M3 scale per 16 elements) on the GPU against the CPU oracle: routing exact,
outputs within the same tolerance as MXFP4, the slot cache copying NVFP4 records, and the MXFP4-only calls
refusing an NVFP4 layer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import (combine_with_weights, compare_routing, compare_values, dev_bytes, outlier_tokens,  # noqa: E402
                    route_arrays, route_weight_rtol)

pytestmark = pytest.mark.gpu

TINY_NV = synth.Workload("tiny_h256_i128_e16k2_nvfp4", 1, 256, 128, 16, 2, 16, (1,), 1, weight_format=1)
GPTOSS_NV = synth.WORKLOADS["gptoss20b_h2880_e32k4_resident_m1_nvfp4"]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def run_and_compare(li, x_bits, out_f32, e2s=None, layer=None):
    w = li.w
    e2s = li.e2s if e2s is None else e2s
    M = x_bits.shape[0]
    lay = layer or li.make_layer(max_tokens=8, out_f32=out_f32)
    x = stack.bf16_tensor(x_bits)
    out = torch.empty((M, w.hidden), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    res = lay.route(x, M)
    lay.forward_slots(x, out, M)
    torch.cuda.synchronize()
    lay.check_error()
    g = route_arrays(res, w.experts, w.top_k)
    o = oracle.moe_layer(x_bits, li.Wr, li.bias, li.bank.numpy(), e2s, w.top_k, w.hidden, w.inter, fmt="nvfp4")
    excl = compare_routing(g, o, o["logits"], w.top_k, e2s)
    compare_values(out.float().cpu().numpy(), o["out_f32"], out_f32, exclude=excl)
    if layer is None:
        lay.close()
    return g, o


@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("out_f32", [False, True])
def test_tiny_nvfp4_layer(M, out_f32):
    li = stack.LayerInputs(TINY_NV, 0)
    run_and_compare(li, synth.activations(0, 0, 200 + M, M, TINY_NV.hidden), out_f32)


@pytest.mark.parametrize("M", [1, 8])
def test_gptoss_shape_nvfp4(M):
    li = stack.LayerInputs(GPTOSS_NV, 3)
    g, _ = run_and_compare(li, synth.activations(0, 3, 210 + M, M, GPTOSS_NV.hidden), M == 8)
    assert g["counts"][2] > 0


@pytest.mark.parametrize("shape", [TINY_NV, GPTOSS_NV])
@pytest.mark.parametrize("fusion", [True, False])
def test_one_token_tensor_core_and_cuda_core_paths(shape, fusion):
    """M = 1 runs the one-launch tensor-core FFN (packed E2M1 x E2M1, UE4M3 scales per 16, x and h as 16 E2M1
    terms each); with decode fusion off the CUDA-core kernels.  Both against the oracle, both output types."""
    li = stack.LayerInputs(shape, 1)
    for out_f32 in (False, True):
        lay = li.make_layer(max_tokens=8, out_f32=out_f32)
        lay.decode_fusion(fusion)
        try:
            run_and_compare(li, synth.activations(0, 1, 240 + out_f32, 1, shape.hidden), out_f32, layer=lay)
        finally:
            lay.close()


@pytest.mark.parametrize("shape", [TINY_NV, GPTOSS_NV])
def test_one_token_outlier_activations(shape):
    """Outliers inside the 16-element blocks of x (and so a wide range within h's blocks) on the tensor-core
    path: routing weights within each token's own summation bound, outputs against the oracle's expert
    outputs combined with the GPU's weights, at the same 2e-3 metric."""
    li = stack.LayerInputs(shape, 2)
    w = li.w
    for seed in (3, 4, 5):
        x = outlier_tokens(seed, 3, w.hidden)[seed % 3:seed % 3 + 1]
        lay = li.make_layer(max_tokens=8, out_f32=True)
        try:
            xt = stack.bf16_tensor(x)
            out = torch.empty((1, w.hidden), dtype=torch.float32, device="cuda")
            res = lay.route(xt, 1)
            lay.forward_slots(xt, out, 1)
            torch.cuda.synchronize()
            lay.check_error()
            g = route_arrays(res, w.experts, w.top_k)
        finally:
            lay.close()
        o = oracle.moe_layer(x, li.Wr, li.bias, li.bank.numpy(), li.e2s, w.top_k, w.hidden, w.inter, fmt="nvfp4")
        excl = compare_routing(g, o, o["logits"], w.top_k, li.e2s, w_rtol=route_weight_rtol(x, li.Wr, li.bias))
        bank = li.bank.numpy()
        ys = np.stack([np.stack([oracle.expert_ffn(bank[e], w.hidden, w.inter, x[0], fmt="nvfp4")
                                 for e in g["ids"][0]])])
        compare_values(out.cpu().numpy(), combine_with_weights(g["ids"], g["w"], ys), True, exclude=excl)


def test_nvfp4_partial_map_cache_refills():
    # 6 of 16 experts resident; the host policy refills slots with NVFP4 records, later steps see them
    w = synth.Workload("tiny_nv_s6", 1, 256, 128, 16, 2, 6, (4,), 1, weight_format=1)
    e2s = np.full(16, -1, dtype=np.int32)
    e2s[[0, 3, 5, 8, 11, 14]] = np.arange(6)
    li = stack.LayerInputs(w, 0, e2s=e2s)
    lay = li.make_layer(max_tokens=8, out_f32=True)
    refills = 0
    for s in range(6):
        x = synth.activations(0, 0, 220 + s, 4, w.hidden)
        run_and_compare(li, x, True, e2s=lay.get_map(), layer=lay)
        refills += lay.cache_update()
        torch.cuda.synchronize()
    assert refills > 0
    m = lay.get_map()
    bank = li.bank.numpy()
    for e in np.nonzero(m >= 0)[0]:  # every resident slot holds its expert's NVFP4 record byte for byte
        assert np.array_equal(dev_bytes(lay.slot_ptr(int(m[e])), w.expert_bytes), bank[e])
    lay.close()


def test_mxfp4_only_calls_refuse_nvfp4():
    li = stack.LayerInputs(TINY_NV, 0)
    lay = li.make_layer(max_tokens=8)
    x = stack.bf16_tensor(synth.activations(0, 0, 230, 1, TINY_NV.hidden))
    out = torch.zeros((1, TINY_NV.hidden), dtype=torch.bfloat16, device="cuda")
    lay.route(x, 1)
    for call in (lambda: lay.forward_cold(x, out, 1), lambda: lay.forward_cold_gpu(x, out, 1),
                 lambda: lay.set_device_cache(True)):
        with pytest.raises(moe.MoeError) as ei:
            call()
        assert ei.value.code == moe.MOE_EINVAL
    stg = torch.empty(16 * TINY_NV.expert_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        lay.attach_staging(stg)
    assert ei.value.code == moe.MOE_EINVAL
    lay.close()
