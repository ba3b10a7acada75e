"""Slot cache on the GPU: refills follow the oracle's replay, slot bytes equal
the bank's, outputs match the oracle under the map each step saw, and faults
injected on the host leave the map unchanged."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import compare_routing, compare_values, dev_bytes, near_tie_tokens, route_arrays  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL = synth.Workload("small_e16k2_s4_drift", 1, 256, 128, 16, 2, 4, (1, 4), 40, bias_tau=2.0, drift=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def slots_match_bank(lay, li, e2s):
    for e, s in enumerate(e2s):
        if s >= 0:
            got = dev_bytes(lay.slot_ptr(int(s)), li.w.expert_bytes)
            assert np.array_equal(got, li.bank.numpy()[e]), (e, s)


def least_popular_placement(seed, E, S):
    """Start from the S least popular experts so that routing misses and refills happen."""
    rank = synth.popularity_rank(seed, 0, E)
    return np.where(rank >= E - S, rank - (E - S), -1).astype(np.int32)


def drive(visibility, decay, steps, M, R=2, seed=0, policy="freq"):
    w = SMALL
    li = stack.LayerInputs(w, 0, seed=seed, e2s=least_popular_placement(seed, w.experts, w.slots))
    lay = li.make_layer(max_tokens=8, out_f32=True, max_refills=R, score_decay=decay, visibility=visibility)
    lay.set_policy({"freq": moe.MOE_POLICY_FREQ, "lru": moe.MOE_POLICY_LRU, "fifo": moe.MOE_POLICY_FIFO,
                    "slru": moe.MOE_POLICY_SLRU}[policy])
    replay = oracle.CacheReplay(li.e2s, w.slots, decay=decay, R=R, policy=policy)
    refills = 0
    for st in range(steps):
        bias = synth.drifting_bias(seed, 0, w.experts, w.bias_tau, st, steps)
        lay.set_bias(torch.from_numpy(bias).cuda())
        e2s_seen = lay.get_map()
        x_bits = synth.activations(seed, 0, 100 + st, M, w.hidden)
        x = stack.bf16_tensor(x_bits)
        out = torch.empty((M, w.hidden), dtype=torch.float32, device="cuda")
        res = lay.route(x, M)
        lay.forward_slots(x, out, M)
        g = route_arrays(res, w.experts, w.top_k)
        o = oracle.moe_layer(x_bits, li.Wr, bias, li.bank.numpy(), e2s_seen, w.top_k, w.hidden, w.inter)
        excl = compare_routing(g, o, o["logits"], w.top_k, e2s_seen)
        assert not excl
        compare_values(out.cpu().numpy(), o["out_f32"], True)
        n = lay.cache_update()
        refills += n
        yield st, lay, li, replay, o, n, e2s_seen
    assert refills > 0
    lay.close()


def test_deterministic_refills_follow_oracle_replay():
    for st, lay, li, replay, o, n, _ in drive(moe.MOE_VIS_DETERMINISTIC, 1.0, 40, 1):
        pairs = replay.step(o["hist"], st)
        assert n == len(pairs)
        assert np.array_equal(lay.get_map(), replay.e2s), st
        torch.cuda.synchronize()
        slots_match_bank(lay, li, lay.get_map())
        st_ = lay.stats()
        assert st_[1] == st_[0] * SMALL.expert_bytes


@pytest.mark.parametrize("policy", ["lru", "fifo", "slru"])
def test_recency_policies_follow_oracle_replay(policy):
    """LRU, FIFO and SLRU slots on the GPU: each step's refills and map equal the oracle's replay, and every
    refilled slot holds its expert's bytes."""
    for st, lay, li, replay, o, n, _ in drive(moe.MOE_VIS_DETERMINISTIC, 1.0, 40, 2, policy=policy):
        pairs = replay.step(o["hist"], st)
        assert n == len(pairs), st
        assert np.array_equal(lay.get_map(), replay.e2s), st
        torch.cuda.synchronize()
        slots_match_bank(lay, li, lay.get_map())


def test_set_policy_rejects_unknown():
    li = stack.LayerInputs(SMALL, 0)
    lay = li.make_layer(max_tokens=8)
    try:
        with pytest.raises(moe.MoeError):
            lay.set_policy(7)
    finally:
        lay.close()


def test_deterministic_lfru_decay_batches():
    for st, lay, li, replay, o, n, _ in drive(moe.MOE_VIS_DETERMINISTIC, 0.7, 30, 4):
        replay.step(o["hist"], st)
        assert np.array_equal(lay.get_map(), replay.e2s), st
    torch.cuda.synchronize()


def test_polled_refills_keep_map_consistent():
    seen_maps = []
    for st, lay, li, replay, o, n, e2s_seen in drive(moe.MOE_VIS_POLLED, 1.0, 40, 1):
        torch.cuda.synchronize()
        m = lay.get_map()
        res = m[m >= 0]
        assert len(set(res.tolist())) == len(res) <= SMALL.slots
        # every expert the device map points at has its own bytes in its slot (a victim's slot may
        # already hold the next expert, but the victim left the map before that copy started)
        slots_match_bank(lay, li, m)
        seen_maps.append(m.copy())
    assert len({m.tobytes() for m in seen_maps}) > 1


def test_injected_copy_fault_leaves_map_unchanged():
    w = SMALL
    li = stack.LayerInputs(w, 0, e2s=least_popular_placement(0, w.experts, w.slots))
    lay = li.make_layer(max_tokens=8, out_f32=True)
    out = torch.empty((1, w.hidden), dtype=torch.float32, device="cuda")
    hit = False
    for st in range(40):
        bias = synth.drifting_bias(0, 0, w.experts, w.bias_tau, st, 40)
        lay.set_bias(torch.from_numpy(bias).cuda())
        x = stack.bf16_tensor(synth.activations(0, 0, 200 + st, 1, w.hidden))
        lay.route(x, 1)
        lay.forward_slots(x, out, 1)
        before = lay.get_map()
        lay.inject_fault(moe.MOE_FAULT_COPY)
        try:
            lay.cache_update()
            lay.inject_fault(moe.MOE_FAULT_NONE)  # no refill was due: the fault was not consumed
        except moe.MoeError as e:
            assert e.code == moe.MOE_ECUDA and "injected" in str(e)
            assert np.array_equal(lay.get_map(), before)
            hit = True
            break
    assert hit
    # the layer keeps working after the failure
    x = stack.bf16_tensor(synth.activations(0, 0, 300, 1, w.hidden))
    lay.route(x, 1)
    lay.forward_slots(x, out, 1)
    torch.cuda.synchronize()
    lay.close()


def test_cache_update_needs_a_route():
    li = stack.LayerInputs(SMALL, 0)
    lay = li.make_layer(max_tokens=8)
    with pytest.raises(moe.MoeError) as ei:
        lay.cache_update()
    assert ei.value.code == moe.MOE_ESTATE
    lay.close()


def test_c4_prefill_then_decode_churn_follows_oracle_replay():
    """The gpt-oss-shaped prefill-then-decode workload: 16 of 32 slots, LFU, at most 2 refills per step,
    popularity drifting from order A to order B.  Step 0 is the 2048-token prefill on the staged bank; its
    routes count in the scores like any other.  Every decode step is checked against the oracle under the
    map it saw, every map against the oracle's policy replay, and every refilled slot against the bank."""
    w = synth.WORKLOADS["gptoss20b_prefill2048_s16_lfu_drift"]
    steps = 24  # the 256-step drift compressed, so that refills happen within the test
    li = stack.LayerInputs(w, 0)
    M_pf = w.prefill_tokens
    lay = li.make_layer(max_tokens=M_pf, out_f32=True, max_refills=2, score_decay=1.0,
                        visibility=moe.MOE_VIS_DETERMINISTIC)
    replay = oracle.CacheReplay(li.e2s, w.slots, decay=1.0, R=2)
    refills = 0
    try:
        staging = torch.empty(w.experts * w.expert_bytes, dtype=torch.uint8, device="cuda")
        lay.attach_staging(staging)
        lay.stage_all()
        # step 0: prefill
        bias = synth.drifting_bias(0, 0, w.experts, w.bias_tau, 0, steps)
        lay.set_bias(torch.from_numpy(bias).cuda())
        x_bits = synth.activations(0, 0, 0, M_pf, w.hidden)
        x = stack.bf16_tensor(x_bits)
        out = torch.empty((M_pf, w.hidden), dtype=torch.float32, device="cuda")
        res = lay.route(x, M_pf)
        lay.forward_slots(x, out, M_pf)
        g = route_arrays(res, w.experts, w.top_k)
        logits = oracle.router_logits(x_bits, li.Wr, bias)
        ids, _ = oracle.topk_softmax(logits, w.top_k)
        tie = near_tie_tokens(logits, w.top_k)
        same = np.array([set(g["ids"][t]) == set(ids[t]) for t in range(M_pf)])
        assert np.all(same | tie)
        if same.all():
            assert np.array_equal(g["hist"], np.bincount(ids.ravel(), minlength=w.experts))
        n = lay.cache_update()
        pairs = replay.step(g["hist"], 0)
        assert n == len(pairs) and np.array_equal(lay.get_map(), replay.e2s)
        refills += n
        del staging
        # decode steps
        out1 = torch.empty((1, w.hidden), dtype=torch.float32, device="cuda")
        for st in range(1, steps):
            bias = synth.drifting_bias(0, 0, w.experts, w.bias_tau, st, steps)
            lay.set_bias(torch.from_numpy(bias).cuda())
            e2s_seen = lay.get_map()
            x_bits = synth.activations(0, 0, 1000 + st, 1, w.hidden)
            x = stack.bf16_tensor(x_bits)
            res = lay.route(x, 1)
            lay.forward_slots(x, out1, 1)
            g = route_arrays(res, w.experts, w.top_k)
            o = oracle.moe_layer(x_bits, li.Wr, bias, li.bank.numpy(), e2s_seen, w.top_k, w.hidden, w.inter)
            excl = compare_routing(g, o, o["logits"], w.top_k, e2s_seen)
            compare_values(out1.cpu().numpy(), o["out_f32"], True, exclude=sorted(excl))
            n = lay.cache_update()
            pairs = replay.step(o["hist"], st)
            assert n == len(pairs), st
            assert np.array_equal(lay.get_map(), replay.e2s), st
            torch.cuda.synchronize()
            for e, slot, _victim in pairs:  # the refilled slots hold their new expert's bytes
                got = dev_bytes(lay.slot_ptr(slot), w.expert_bytes)
                assert np.array_equal(got, li.bank.numpy()[e]), (st, e, slot)
            refills += n
    finally:
        lay.close()
    assert refills > 0
