"""NVFP4 experts (E2M1 codes, one E4M3 scale per 16 elements) on the GPU against the CPU oracle: routing exact,
outputs within the same tolerance as MXFP4, the slot cache copying NVFP4 records, and the MXFP4-only calls
refusing an NVFP4 layer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import compare_routing, compare_values, dev_bytes, route_arrays  # noqa: E402

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
