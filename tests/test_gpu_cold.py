"""Cold routes on host threads (moe_forward_cold): the GPU's hot sum plus the host's cold sum equals the
oracle's output with every expert resident, within the value tolerance; the result does not depend on the
number of host threads."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import bf16_half_ulp, compare_values, near_tie_tokens  # noqa: E402

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
TINY = W["tiny_h256_i128_e16k2"]
E512 = W["e512k10_h2048_i512_s256_m1"]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def hybrid(li, x_bits, out_f32=True, nthreads=0, lay=None, on_gpu=False):
    w = li.w
    M = x_bits.shape[0]
    own = lay is None
    lay = lay or li.make_layer(max_tokens=8, out_f32=out_f32)
    try:
        x = stack.bf16_tensor(x_bits)
        out = torch.empty((M, w.hidden), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
        res = lay.route(x, M)
        lay.forward_slots(x, out, M)
        if on_gpu:
            lay.forward_cold_gpu(x, out, M)
        else:
            lay.forward_cold(x, out, M, nthreads=nthreads)
        torch.cuda.synchronize()
        n_cold = int(stack.host_counts(res)[1])
        got = out.float().cpu().numpy()
    finally:
        if own:
            lay.close()
    return got, n_cold


def all_resident(li, x_bits):
    w = li.w
    return oracle.moe_layer(x_bits, li.Wr, li.bias, li.bank.numpy(), np.arange(w.experts, dtype=np.int32),
                            w.top_k, w.hidden, w.inter)


@pytest.mark.parametrize("on_gpu", [False, True])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_tiny_half_resident(M, on_gpu):
    e2s = np.full(TINY.experts, -1, dtype=np.int32)
    e2s[::2] = np.arange(TINY.experts // 2)  # even experts in slots, odd ones cold
    li = stack.LayerInputs(TINY, 0, e2s=e2s)
    x_bits = synth.activations(0, 0, 60 + M, M, TINY.hidden)
    got, n_cold = hybrid(li, x_bits, on_gpu=on_gpu)
    o = all_resident(li, x_bits)
    assert n_cold > 0
    compare_values(got, o["out_f32"], True, exclude=np.where(near_tie_tokens(o["logits"], TINY.top_k))[0])


@pytest.mark.parametrize("on_gpu", [False, True])
def test_tiny_all_cold(on_gpu):
    li = stack.LayerInputs(TINY, 0, e2s=np.full(TINY.experts, -1, dtype=np.int32))
    x_bits = synth.activations(0, 0, 70, 4, TINY.hidden)
    got, n_cold = hybrid(li, x_bits, on_gpu=on_gpu)
    assert n_cold == 4 * TINY.top_k
    o = all_resident(li, x_bits)
    compare_values(got, o["out_f32"], True, exclude=np.where(near_tie_tokens(o["logits"], TINY.top_k))[0])


@pytest.mark.parametrize("on_gpu", [False, True])
def test_e512_half_resident_m1(on_gpu):
    """The E=512 shape with its 256 slots by popularity rank: about a quarter of the routes are cold."""
    li = stack.LayerInputs(E512, 0)
    for s in range(3):
        x_bits = synth.activations(0, 0, 80 + s, 1, E512.hidden)
        got, n_cold = hybrid(li, x_bits, on_gpu=on_gpu)
        o = all_resident(li, x_bits)
        compare_values(got, o["out_f32"], True, exclude=np.where(near_tie_tokens(o["logits"], E512.top_k))[0])


def test_thread_count_does_not_change_the_result():
    e2s = np.full(TINY.experts, -1, dtype=np.int32)
    e2s[:4] = np.arange(4)
    li = stack.LayerInputs(TINY, 0, e2s=e2s)
    x_bits = synth.activations(0, 0, 90, 8, TINY.hidden)
    a, _ = hybrid(li, x_bits, nthreads=1)
    b, _ = hybrid(li, x_bits, nthreads=0)
    c, _ = hybrid(li, x_bits, nthreads=3)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_bf16_output():
    e2s = np.full(TINY.experts, -1, dtype=np.int32)
    e2s[1::2] = np.arange(TINY.experts // 2)
    li = stack.LayerInputs(TINY, 0, e2s=e2s)
    x_bits = synth.activations(0, 0, 95, 8, TINY.hidden)
    got, _ = hybrid(li, x_bits, out_f32=False)
    o = all_resident(li, x_bits)
    hot = oracle.moe_layer(x_bits, li.Wr, li.bias, li.bank.numpy(), e2s, TINY.top_k, TINY.hidden, TINY.inter)
    # the GPU rounds its hot sum to bf16, the cold sum is added and the total rounded again: beyond the value
    # tolerance, half a bf16 ulp of the hot part and half of the result
    ref = o["out_f32"].astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    allow = (2e-3 * np.maximum(np.abs(ref), 1e-2 * rms) + bf16_half_ulp(hot["out_f32"].astype(np.float64))
             + bf16_half_ulp(ref))
    keep = ~near_tie_tokens(o["logits"], TINY.top_k)
    assert np.all(np.abs(got - ref)[keep] <= allow[keep])


def test_cold_needs_the_last_route():
    li = stack.LayerInputs(TINY, 0)
    lay = li.make_layer(max_tokens=8, out_f32=True)
    try:
        x = stack.bf16_tensor(synth.activations(0, 0, 99, 2, TINY.hidden))
        out = torch.zeros((2, TINY.hidden), dtype=torch.float32, device="cuda")
        with pytest.raises(moe.MoeError):
            lay.forward_cold(x, out, 2)
    finally:
        lay.close()


def test_gpu_cold_in_a_graph_matches_eager():
    """route + forward_slots + forward_cold_gpu captured in a CUDA graph and replayed on new inputs gives
    the eager result bit for bit (no host step in the GPU cold path)."""
    e2s = np.full(TINY.experts, -1, dtype=np.int32)
    e2s[::3] = np.arange(len(e2s[::3]))
    li = stack.LayerInputs(TINY, 0, e2s=e2s)
    lay = li.make_layer(max_tokens=8, out_f32=True)
    try:
        M = 4
        x = torch.empty((M, TINY.hidden), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((M, TINY.hidden), dtype=torch.float32, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def body():
            lay.route(x, M, s)
            lay.forward_slots(x, out, M, s)
            lay.forward_cold_gpu(x, out, M, s)

        x.copy_(stack.bf16_tensor(synth.activations(0, 0, 120, M, TINY.hidden)))
        with torch.cuda.stream(s):
            body()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        for step in range(3):
            xb = synth.activations(0, 0, 130 + step, M, TINY.hidden)
            x.copy_(stack.bf16_tensor(xb))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            replayed = out.cpu().numpy().copy()
            with torch.cuda.stream(s):
                body()
            torch.cuda.synchronize()
            assert np.array_equal(replayed, out.cpu().numpy())
            o = all_resident(li, xb)
            compare_values(replayed, o["out_f32"], True, exclude=np.where(near_tie_tokens(o["logits"], TINY.top_k))[0])
    finally:
        lay.close()
