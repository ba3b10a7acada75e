"""Prefill (M > 8) on the tensor cores over the staged expert bank, against the oracle's prefill reading.

With every expert staged, every route is hot and the output is
  out[t] = sum over t's top-k experts in ascending expert order of w * y_e(x_t),
where y_e is the expert FFN with x and h passed through MXFP8 (32-element
E4M3 blocks, OCP MX v1.0 conversion rule) before their products with the
MXFP4 weights (oracle.expert_ffn_mxfp8).
"""
import numpy as np
import pytest
import torch

import oracle
from expert_offload_moe_gb300 import stack, synth

from parity import (compare_routing, compare_values, near_tie_tokens, oracle_ffn_mxfp8_task, outlier_tokens,
                    route_arrays, spawn_pool)

pytestmark = pytest.mark.gpu


def prefill_reference(li, x_bits, k, H, I, tokens, pool=None):
    """The oracle's prefill output for the listed tokens: fp32, experts summed in ascending order.  With a
    process pool the expert FFNs run in its workers (same function, records regenerated from the seed)."""
    logits = oracle.router_logits(x_bits, li.Wr, li.bias)
    ids, w = oracle.topk_softmax(logits, k)
    order = [(t, j) for t in tokens for j in np.argsort(ids[t], kind="stable")]
    if pool is None:
        bank = li.bank.numpy()
        ys = [oracle.expert_ffn_mxfp8(bank[ids[t][j]], H, I, x_bits[t]) for t, j in order]
    else:
        ys = pool.map(oracle_ffn_mxfp8_task, [(li.seed, li.layer, li.w.experts, H, I, int(ids[t][j]), x_bits[t])
                                             for t, j in order])
    out = np.zeros((len(tokens), H), dtype=np.float32)
    it = iter(zip(order, ys))
    for i, t in enumerate(tokens):
        acc = np.zeros(H, dtype=np.float32)
        for _ in range(k):
            (_, j), y = next(it)
            acc = (acc + np.float32(w[t][j]) * y).astype(np.float32)
        out[i] = acc
    return out, logits


def run_prefill(li, x_bits, M, out_f32=True, max_tokens=None, routes=False):
    w = li.w
    lay = li.make_layer(max_tokens=max_tokens or M, out_f32=out_f32)
    try:
        staging = torch.empty(w.experts * w.expert_bytes, dtype=torch.uint8, device="cuda")
        lay.attach_staging(staging)
        lay.stage_all()
        x = stack.bf16_tensor(x_bits)
        out = torch.empty((M, w.hidden), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
        res = lay.route(x, M)
        lay.forward_slots(x, out, M)
        torch.cuda.synchronize()
        lay.check_error()
        got = out.float().cpu().numpy()
        g = route_arrays(res, w.experts, w.top_k) if routes else None
    finally:
        lay.close()
    return (got, g) if routes else got


def tokens_covering_every_route_tile(g, tile=128):
    """A set of tokens that has a route in every (expert, 128-route tile) of the grouped GEMMs: the hot
    list is ordered by (expert, token) and each expert's routes are padded to whole tiles, so route r of
    expert e's segment lies in tile r // 128.  Greedy: the first token of each tile not yet covered."""
    covered, tokens = set(), []
    tiles_of = {}
    for e, off, cnt in zip(g["act_expert"], g["act_off"], g["act_cnt"]):
        for r in range(cnt):
            tiles_of.setdefault(int(g["hot_token"][off + r]), []).append((int(e), r // tile))
    for e, off, cnt in zip(g["act_expert"], g["act_off"], g["act_cnt"]):
        for r0 in range(0, cnt, tile):
            if (int(e), r0 // tile) in covered:
                continue
            t = int(g["hot_token"][off + r0])
            tokens.append(t)
            covered.update(tiles_of[t])
    n_tiles = sum((int(c) + tile - 1) // tile for c in g["act_cnt"])
    assert len(covered) == n_tiles
    return sorted(tokens), n_tiles


def _tiny():
    base = synth.WORKLOADS["tiny_h256_i128_e16k2"]
    return synth.Workload("tiny_prefill", 1, base.hidden, base.inter, base.experts, base.top_k, base.experts,
                          (16,), 1, bias_tau=0.25)


@pytest.mark.parametrize("M", [9, 40, 300])
def test_prefill_tiny_all_tokens(M):
    """Every token and column: M spans one and several 128-route tiles per expert (ragged last tiles)."""
    w = _tiny()
    li = stack.LayerInputs(w, 0)
    x_bits = synth.activations(0, 0, 11, M, w.hidden)
    got = run_prefill(li, x_bits, M)
    ref, logits = prefill_reference(li, x_bits, w.top_k, w.hidden, w.inter, range(M))
    compare_values(got, ref, True, exclude=np.where(near_tie_tokens(logits, w.top_k))[0])


def test_prefill_multi_tile_shape():
    """H = 704, I = 320: gate/up spans three 128-row tiles of I (the last one ragged) over 5.5 steps of K
    (the pipeline stages are reused, the last step is half empty); down spans a full 256-row tile of H
    and a ragged one over 2.5 steps of K.  Every token and column."""
    w = synth.Workload("prefill_h704_i320_e8k2", 1, 704, 320, 8, 2, 8, (16,), 1, bias_tau=0.25)
    li = stack.LayerInputs(w, 0)
    M = 300
    x_bits = synth.activations(0, 0, 14, M, w.hidden)
    got = run_prefill(li, x_bits, M)
    ref, logits = prefill_reference(li, x_bits, w.top_k, w.hidden, w.inter, range(M))
    compare_values(got, ref, True, exclude=np.where(near_tie_tokens(logits, w.top_k))[0])


def test_prefill_tiny_bf16_out():
    w = _tiny()
    li = stack.LayerInputs(w, 0)
    M = 64
    x_bits = synth.activations(0, 0, 12, M, w.hidden)
    got = run_prefill(li, x_bits, M, out_f32=False)
    ref, logits = prefill_reference(li, x_bits, w.top_k, w.hidden, w.inter, range(M))
    compare_values(got, ref, False, exclude=np.where(near_tie_tokens(logits, w.top_k))[0])


def test_prefill_gptoss_shape_every_route_tile():
    """The gpt-oss-20B-shaped prefill batch (2048 tokens, 32 experts, k = 4; ragged H = I = 2880) in the
    launch configuration the benchmark times, checked on a set of tokens that has a route in every
    (expert, 128-route tile) work item of the grouped GEMMs (plus the first and last token), every column,
    the oracle computing each token's experts one by one."""
    w = synth.WORKLOADS["gptoss20b_prefill2048_s16_lfu_drift"]
    li = stack.LayerInputs(w, 0)
    M = w.prefill_tokens
    x_bits = synth.activations(0, 0, 0, M, w.hidden)
    got, g = run_prefill(li, x_bits, M, routes=True)
    tokens, n_tiles = tokens_covering_every_route_tile(g)
    assert n_tiles >= 64  # about 256 routes per expert: two or three tiles each
    tokens = sorted(set(tokens) | {0, M - 1})
    with spawn_pool() as pool:
        ref, logits = prefill_reference(li, x_bits, w.top_k, w.hidden, w.inter, tokens, pool=pool)
    tie = near_tie_tokens(logits, w.top_k)
    keep = [i for i, t in enumerate(tokens) if not tie[t]]
    compare_values(got[tokens][keep], ref[keep], True)


@pytest.mark.parametrize("out_f32", [True, False])
def test_prefill_outlier_blocks(out_f32):
    """Activations with outliers inside their 32-element blocks: MXFP8 keeps 3 mantissa bits relative to
    each block's scale on both sides, and h spans a wide range within its blocks; every token and column."""
    w = _tiny()
    li = stack.LayerInputs(w, 0)
    M = 60
    x_bits = outlier_tokens(5, M, w.hidden)
    got = run_prefill(li, x_bits, M, out_f32=out_f32)
    ref, logits = prefill_reference(li, x_bits, w.top_k, w.hidden, w.inter, range(M))
    compare_values(got, ref, out_f32, exclude=np.where(near_tie_tokens(logits, w.top_k))[0])


def _route_case(w, M, seed_step, layer=0):
    """Prefill routing of M tokens against the oracle: every expert hot (slot = expert id), hot routes in
    (expert, token) order, no cold routes."""
    li = stack.LayerInputs(w, layer)
    x_bits = synth.activations(0, layer, seed_step, M, w.hidden)
    lay = li.make_layer(max_tokens=M)
    try:
        res = lay.route(stack.bf16_tensor(x_bits), M)
        g = route_arrays(res, w.experts, w.top_k)
    finally:
        lay.close()
    logits = oracle.router_logits(x_bits, li.Wr, li.bias)
    ids, wt = oracle.topk_softmax(logits, w.top_k)
    all_hot = np.arange(w.experts, dtype=np.int32)
    o = oracle.compact(ids, wt, all_hot)
    o.update(ids=ids, w=wt)
    assert g["mirror_ok"]
    assert g["counts"][1] == 0 and g["counts"][3] == M
    excl = compare_routing(g, o, logits, w.top_k, all_hot)
    return g, excl


@pytest.mark.parametrize("M", [9, 16, 17, 40, 300, 4096])
def test_prefill_routing_tiny(M):
    """Token tiles of 16: a partial first tile, exactly one, one plus one token, several, the maximum."""
    _route_case(_tiny(), M, 21)


def test_prefill_routing_gptoss_2048():
    w = synth.WORKLOADS["gptoss20b_prefill2048_s16_lfu_drift"]
    g, _ = _route_case(w, w.prefill_tokens, 0, layer=3)
    assert g["counts"][0] == w.prefill_tokens * w.top_k


def test_prefill_routing_e512_k10():
    """512 experts (sixteen 32-expert groups of router rows), k = 10, skewed popularity."""
    _route_case(synth.WORKLOADS["e512k10_h2048_i512_s256_m1"], 100, 5)


def test_prefill_needs_staging():
    w = _tiny()
    li = stack.LayerInputs(w, 0)
    lay = li.make_layer(max_tokens=16, out_f32=True)
    try:
        M = 12
        x = stack.bf16_tensor(synth.activations(0, 0, 13, M, w.hidden))
        out = torch.empty((M, w.hidden), dtype=torch.float32, device="cuda")
        lay.route(x, M)
        with pytest.raises(Exception):
            lay.forward_slots(x, out, M)
    finally:
        lay.close()


def test_prefill_needs_a_route_after_staging():
    """The route launch plans the prefill tiles only when the staging buffer is attached: routing first and
    attaching afterwards is refused, and routing again makes it run."""
    w = _tiny()
    li = stack.LayerInputs(w, 0)
    lay = li.make_layer(max_tokens=32, out_f32=True)
    try:
        M = 20
        x_bits = synth.activations(0, 0, 15, M, w.hidden)
        x = stack.bf16_tensor(x_bits)
        out = torch.empty((M, w.hidden), dtype=torch.float32, device="cuda")
        lay.route(x, M)
        staging = torch.empty(w.experts * w.expert_bytes, dtype=torch.uint8, device="cuda")
        lay.attach_staging(staging)
        lay.stage_all()
        with pytest.raises(Exception):
            lay.forward_slots(x, out, M)
        lay.route(x, M)
        lay.forward_slots(x, out, M)
        torch.cuda.synchronize()
        lay.check_error()
        ref, logits = prefill_reference(li, x_bits, w.top_k, w.hidden, w.inter, range(M))
        compare_values(out.cpu().numpy(), ref, True, exclude=np.where(near_tie_tokens(logits, w.top_k))[0])
    finally:
        lay.close()
