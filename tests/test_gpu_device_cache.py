"""Device-resident slot table on the GPU (xinfer docs "How it works", Decode): each decode step's map equals
the oracle's demand-filled LRU replay, filled slots hold their experts' bytes, every route is computed and the
output equals the oracle's with every expert resident, misses beyond the slots stay cold, and the whole step
replays inside a CUDA graph."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import compare_routing, compare_values, dev_bytes, near_tie_tokens, route_arrays  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL = synth.Workload("small_e16k2_s4_drift", 1, 256, 128, 16, 2, 4, (1, 4), 40, bias_tau=2.0, drift=True)
# mild skew: 8 tokens route to about 10 distinct experts, more than the 4 slots
SPREAD = synth.Workload("small_e16k2_s4_spread", 1, 256, 128, 16, 2, 4, (8,), 12, bias_tau=0.25, drift=True)
# gpt-oss-20B expert shape (H = I = 2880, 23 tiles of 128 rows per matrix, a ragged 64-row last tile)
GPTOSS = synth.Workload("gptoss_h2880_e32k4_s16", 1, 2880, 2880, 32, 4, 16, (1,), 6, bias_tau=0.25)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def least_popular_placement(seed, E, S, empty=0):
    """The S least popular experts in the slots (so that steps miss), the last `empty` slots left empty."""
    rank = synth.popularity_rank(seed, 0, E)
    e2s = np.where(rank >= E - S, rank - (E - S), -1).astype(np.int32)
    e2s[e2s >= S - empty] = -1
    return e2s


def slots_match_bank(lay, li, e2s):
    for e, s in enumerate(e2s):
        if s >= 0:
            got = dev_bytes(lay.slot_ptr(int(s)), li.w.expert_bytes)
            assert np.array_equal(got, li.bank.numpy()[e]), (e, s)


def oracle_hist(li, x_bits, bias, k):
    logits = oracle.router_logits(x_bits, li.Wr, bias)
    ids, _ = oracle.topk_softmax(logits, k)
    return np.bincount(ids.ravel(), minlength=li.Wr.shape[0]).astype(np.int32), logits


def run_steps(w, M, steps, seed=0, empty=0, cold_gpu=False, out_f32=True):
    """Drives a layer with the device table on through `steps` decode steps of drifting routing; yields
    (step, layer, inputs, replay, fills, GPU output, oracle result under the new map, GPU routing)."""
    li = stack.LayerInputs(w, 0, seed=seed, e2s=least_popular_placement(seed, w.experts, w.slots, empty))
    lay = li.make_layer(max_tokens=8, out_f32=out_f32)
    lay.set_device_cache(True)
    replay = oracle.DemandLRUReplay(li.e2s, w.slots)
    try:
        for st in range(steps):
            bias = synth.drifting_bias(seed, 0, w.experts, w.bias_tau, st, steps) if w.drift else li.bias
            lay.set_bias(torch.from_numpy(np.ascontiguousarray(bias, dtype=np.float32)).cuda())
            x_bits = synth.activations(seed, 0, 200 + st, M, w.hidden)
            x = stack.bf16_tensor(x_bits)
            out = torch.zeros((M, w.hidden), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
            res = lay.route(x, M)
            lay.forward_slots(x, out, M)
            if cold_gpu:
                lay.forward_cold_gpu(x, out, M)
            g = route_arrays(res, w.experts, w.top_k)
            hist, logits = oracle_hist(li, x_bits, bias, w.top_k)
            assert not near_tie_tokens(logits, w.top_k).any(), "seeded inputs must not hold near ties"
            fills = replay.step(hist)
            o = oracle.moe_layer(x_bits, li.Wr, bias, li.bank.numpy(), replay.e2s, w.top_k, w.hidden, w.inter)
            assert not compare_routing(g, o, o["logits"], w.top_k, replay.e2s)
            yield st, lay, li, replay, fills, out, o, g
    finally:
        lay.close()


@pytest.mark.parametrize("M,empty", [(1, 0), (4, 0), (2, 2)])
def test_device_table_follows_oracle_replay(M, empty):
    """Map after every step = the oracle's demand-filled LRU replay (misses left without a slot stay cold and
    the routing comparison checks the cold list); filled slots hold their experts' bytes; the hot output is
    the oracle's under the new map; the device counters add up."""
    n_fill = n_hit = n_cold = 0
    steps = 40
    for st, lay, li, replay, fills, out, o, g in run_steps(SMALL, M, steps, empty=empty):
        assert np.array_equal(lay.get_map(), replay.e2s), st
        for e, s in fills:
            got = dev_bytes(lay.slot_ptr(s), li.w.expert_bytes)
            assert np.array_equal(got, li.bank.numpy()[e]), (st, e, s)
        compare_values(out.cpu().numpy(), o["out_f32"], True)
        routed = np.nonzero(o["hist"])[0]
        filled = {f[0] for f in fills}
        n_fill += len(fills)
        n_hit += int(sum(1 for e in routed if e not in filled and replay.e2s[e] >= 0))
        n_cold += len({int(e) for e in o["cold_expert"]})
        if st == steps - 1:
            stats = lay.device_cache_stats()
            assert list(stats) == [steps, n_fill, n_hit, n_cold]
            slots_match_bank(lay, li, lay.get_map())
    assert n_fill > 0


def test_device_table_overflow_goes_cold_and_the_cold_path_completes_it():
    """M k > S: the misses without a slot stay cold this step; the GPU cold path adds them, and the sum
    equals the oracle's output with every expert resident."""
    w = SPREAD
    overflowed = 0
    for st, lay, li, replay, fills, out, o, g in run_steps(w, 8, 12, cold_gpu=True):
        o_all = oracle.moe_layer(synth.activations(0, 0, 200 + st, 8, w.hidden), li.Wr,
                                 synth.drifting_bias(0, 0, w.experts, w.bias_tau, st, 12), li.bank.numpy(),
                                 np.arange(w.experts, dtype=np.int32), w.top_k, w.hidden, w.inter)
        compare_values(out.cpu().numpy(), o_all["out_f32"], True)
        overflowed += int(g["counts"][1] > 0)
        assert np.array_equal(lay.get_map(), replay.e2s), st
    assert overflowed > 0


@pytest.mark.parametrize("out_f32", [True, False])
def test_device_table_output_is_bit_identical_to_every_expert_resident(out_f32):
    """Placement never changes the arithmetic (xinfer docs: byte-identical output for every offload
    fraction): with M k <= S the device table's output equals, bit for bit, that of a layer holding every
    expert."""
    w, M = SMALL, 2
    full = stack.LayerInputs(w, 0, seed=0, e2s=np.arange(w.experts, dtype=np.int32))
    ref = moe.Layer(w.hidden, w.inter, w.experts, w.top_k, w.experts, 8, torch.from_numpy(full.Wr).cuda(),
                    torch.from_numpy(full.bias).cuda(), full.bank, full.e2s, out_f32=out_f32)
    try:
        for st, lay, li, replay, fills, out, o, g in run_steps(w, M, 20, out_f32=out_f32):
            bias = synth.drifting_bias(0, 0, w.experts, w.bias_tau, st, 20)
            ref.set_bias(torch.from_numpy(bias).cuda())
            x = stack.bf16_tensor(synth.activations(0, 0, 200 + st, M, w.hidden))
            r = torch.zeros_like(out)
            ref.route(x, M)
            ref.forward_slots(x, r, M)
            torch.cuda.synchronize()
            assert torch.equal(out, r), st
    finally:
        ref.close()


def test_device_table_gptoss_shape():
    """gpt-oss-20B expert shape: fills of 13.2 MB records with their 23 x 23 scale atoms per matrix (ragged
    last tile), then the tensor-core FFN on the filled slots."""
    n_fill = 0
    for st, lay, li, replay, fills, out, o, g in run_steps(GPTOSS, 1, GPTOSS.steps, empty=1):
        assert np.array_equal(lay.get_map(), replay.e2s), st
        compare_values(out.cpu().numpy(), o["out_f32"], True)
        assert g["counts"][1] == 0  # k = 4 <= 16 slots: nothing stays cold
        n_fill += len(fills)
    assert n_fill > 0


def test_device_table_step_in_a_cuda_graph():
    """route (with the table step and the fill kernel) + forward_slots captured once and replayed on new
    inputs: the map follows the replay and the output the oracle, with no host step in between."""
    w, M = SMALL, 1
    li = stack.LayerInputs(w, 0, e2s=least_popular_placement(0, w.experts, w.slots))
    lay = li.make_layer(max_tokens=8, out_f32=True)
    try:
        lay.set_device_cache(True)
        replay = oracle.DemandLRUReplay(li.e2s, w.slots)
        x = torch.empty((M, w.hidden), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((M, w.hidden), dtype=torch.float32, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def body():
            lay.route(x, M, s)
            lay.forward_slots(x, out, M, s)

        def inputs(step):
            return synth.activations(0, 0, 300 + step, M, w.hidden)

        x.copy_(stack.bf16_tensor(inputs(0)))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            body()
        torch.cuda.synchronize()
        replay.step(oracle_hist(li, inputs(0), li.bias, w.top_k)[0])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        fills = 0
        for step in range(1, 25):
            xb = inputs(step)
            x.copy_(stack.bf16_tensor(xb))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            fills += len(replay.step(oracle_hist(li, xb, li.bias, w.top_k)[0]))
            assert np.array_equal(lay.get_map(), replay.e2s), step
            o = oracle.moe_layer(xb, li.Wr, li.bias, li.bank.numpy(), replay.e2s, w.top_k, w.hidden, w.inter)
            compare_values(out.cpu().numpy(), o["out_f32"], True)
        assert fills > 0
        slots_match_bank(lay, li, lay.get_map())
    finally:
        lay.close()


def test_device_table_hand_back_and_rejections():
    """While the table is on the host policy is refused; switching off hands the device's map to the host
    policy, which then refills from there."""
    w = SMALL
    li = stack.LayerInputs(w, 0, e2s=least_popular_placement(0, w.experts, w.slots))
    lay = li.make_layer(max_tokens=8, out_f32=True)
    try:
        lay.set_device_cache(True)
        x = stack.bf16_tensor(synth.activations(0, 0, 400, 1, w.hidden))
        out = torch.empty((1, w.hidden), dtype=torch.float32, device="cuda")
        lay.route(x, 1)
        lay.forward_slots(x, out, 1)
        with pytest.raises(moe.MoeError) as ei:
            lay.cache_update()
        assert ei.value.code == moe.MOE_ESTATE
        dev_map = lay.get_map()
        lay.set_device_cache(False)
        assert np.array_equal(lay.get_map(), dev_map)
        slots_match_bank(lay, li, dev_map)
        lay.route(x, 1)
        lay.forward_slots(x, out, 1)
        lay.cache_update()  # the host policy works from the handed-back map
        torch.cuda.synchronize()
        slots_match_bank(lay, li, lay.get_map())
    finally:
        lay.close()
