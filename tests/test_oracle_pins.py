"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it cannot agree with by
construction: a published format table, a bit-field definition, brute force
over a tiny input, a library matmul in float64 with a rigorous fp32 error
bound, a closed form, or a trace worked by hand.
"""
import itertools
import math
import os

import numpy as np
import pytest

from expert_offload_moe_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U32 = 2.0 ** -24  # fp32 unit roundoff


# ----------------------------------------------------------- independent decoders


def e2m1_from_bits(code):
    """OCP MX v1.0 E2M1: sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return s * mag


def decode_mxfp4_np(codes, scales, R, C):
    """float64 decode of an MXFP4 matrix from bit fields (independent of the oracle's table)."""
    codes = codes.reshape(R, C // 2)
    lo = (codes & 15).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    q = np.empty((R, C), dtype=np.int64)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    sign = np.where(q & 8, -1.0, 1.0)
    e = (q >> 1) & 3
    m = q & 1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, (e - 1)))
    sc = np.ldexp(1.0, scales.reshape(R, C // 32).astype(np.int64) - 127)
    return sign * mag * np.repeat(sc, 32, axis=1)


def bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sections(rec, H, I):
    offs = synth.section_offsets(H, I)
    return {k: rec[o:o + n] for k, (o, n) in offs.items()}


# ------------------------------------------------------------------- formats


def test_e2m1_table_matches_ocp_fixture_and_bit_fields(oracle_lib):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_ocp_mx_v1.txt")) if l[0] != "#"]
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s), float(val_s)
        got = oracle_lib.e2m1(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
        assert got == e2m1_from_bits(code)


@pytest.mark.parametrize("e", [0, 1, 2, 100, 120, 121, 122, 123, 124, 125, 126, 127, 128, 200, 254])
def test_e8m0_scales_exact(oracle_lib, e):
    assert oracle_lib.e8m0(e) == math.ldexp(1.0, e - 127)


def test_e8m0_nan(oracle_lib):
    assert math.isnan(oracle_lib.e8m0(255))


def test_mxfp4_exhaustive_codes_times_scales(oracle_lib):
    # every code in every position of a 32-element block, under several scales
    scales_list = [1, 120, 121, 122, 123, 124, 125, 126, 127, 200, 254]
    R = len(scales_list)
    C = 32
    codes = np.zeros((R, C // 2), dtype=np.uint8)
    vals = np.arange(C) % 16
    codes[:] = (vals[0::2] | (vals[1::2] << 4)).astype(np.uint8)
    scales = np.array(scales_list, dtype=np.uint8).reshape(R, 1)
    W = oracle_lib.mxfp4_dequant(codes, scales, R, C)
    ref = decode_mxfp4_np(codes, scales, R, C)
    # every finite product is exact in fp32; 6 * 2^127 overflows to inf in fp32 as it must
    with np.errstate(over="ignore"):
        assert np.array_equal(W, ref.astype(np.float32))
    assert W[-1, 4] == np.inf and W[-1, 15] == -np.inf and float(W[-1, 3]) == 1.5 * 2.0 ** 127


def test_mxfp4_nibble_order_and_block_scales(oracle_lib):
    # column 2c is the low nibble of byte c; scale b covers columns [32b, 32b+32)
    R, C = 2, 64
    codes = np.zeros((R, C // 2), dtype=np.uint8)
    codes[0, 0] = 0x72  # col 0 -> code 2 (1.0), col 1 -> code 7 (6.0)
    codes[1, 16] = 0x0B  # col 32 -> code 11 (-1.5), col 33 -> 0
    scales = np.array([[127, 126], [127, 129]], dtype=np.uint8)
    W = oracle_lib.mxfp4_dequant(codes, scales, R, C)
    assert W[0, 0] == 1.0 and W[0, 1] == 6.0 and np.count_nonzero(W[0]) == 2
    assert W[1, 32] == -1.5 * 4.0 and np.count_nonzero(W[1]) == 1


def test_bf16_round_nearest_even(oracle_lib):
    assert oracle_lib.f32_to_bf16(1.0) == 0x3F80
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    assert oracle_lib.f32_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even) -> up
    assert oracle_lib.f32_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle_lib.f32_to_bf16(-2.0) == 0xC000


# -------------------------------------------------------------------- router


def test_router_logits_within_fp32_bound(oracle_lib):
    H, E, M = 256, 16, 5
    x = synth.activations(0, 0, 0, M, H)
    Wr = synth.router_weights(0, 0, E, H)
    b = np.linspace(-1, 1, E).astype(np.float32)
    got = oracle_lib.router_logits(x, Wr, b).astype(np.float64)
    xf = bf16_to_f64(x)
    exact = xf @ Wr.astype(np.float64).T + b.astype(np.float64)
    bound = (H + 2) * U32 * (np.abs(xf) @ np.abs(Wr.astype(np.float64)).T + np.abs(b))
    assert np.all(np.abs(got - exact) <= bound)
    # a transposed or shifted operand is far outside the bound
    assert np.max(np.abs(got - exact)) < 1e-4


# --------------------------------------------------------------------- top-k


def brute_topk(l, k):
    E = len(l)
    sols = []
    for S in itertools.combinations(range(E), k):
        inside = set(S)
        ok = all(l[i] > l[j] or (l[i] == l[j] and i < j) for i in inside for j in range(E) if j not in inside)
        if ok:
            sols.append(S)
    assert len(sols) == 1
    return sorted(sols[0], key=lambda i: (-l[i], i))


def test_topk_brute_force_with_ties(oracle_lib):
    rng = np.random.default_rng(7)
    E, k = 16, 2
    logits = rng.standard_normal((64, E)).astype(np.float32)
    logits[32:] = np.round(logits[32:] * 2) / 2  # many exact ties
    logits[40] = 0.0  # all equal -> experts 0, 1
    ids, _ = oracle_lib.topk_softmax(logits, k)
    for t in range(logits.shape[0]):
        assert list(ids[t]) == brute_topk([float(v) for v in logits[t]], k), t
    assert list(ids[40]) == [0, 1]


@pytest.mark.parametrize("k", [1, 2, 4, 10])
def test_softmax_weights(oracle_lib, k):
    rng = np.random.default_rng(k)
    E = 32
    logits = (rng.standard_normal((16, E)) * 3).astype(np.float32)
    ids, w = oracle_lib.topk_softmax(logits, k)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 4 * k * U32)
    if k == 1:
        assert np.all(w == 1.0)
    # closed form against float64 on the selected logits
    sel = np.take_along_axis(logits, ids, 1).astype(np.float64)
    ref = np.exp(sel - sel.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-6, atol=1e-7)
    # weights follow the logit order
    assert np.all(np.diff(w, axis=1) <= 0)


def test_softmax_equal_logits(oracle_lib):
    logits = np.zeros((1, 8), dtype=np.float32)
    _, w = oracle_lib.topk_softmax(logits, 4)
    assert np.all(w == np.float32(0.25))


# ---------------------------------------------------------------- compaction


def test_compaction_against_brute_force_filter(oracle_lib):
    rng = np.random.default_rng(3)
    M, E, k = 8, 32, 4
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(M)], dtype=np.int32)
    w = rng.random((M, k)).astype(np.float32)
    e2s = np.full(E, -1, dtype=np.int32)
    resident = rng.choice(E, 12, replace=False)
    e2s[resident] = rng.permutation(12)
    r = oracle_lib.compact(ids, w, e2s)
    routes = [(t, int(ids[t, j]), float(w[t, j])) for t in range(M) for j in range(k)]
    hot = sorted([(e, t, wt) for t, e, wt in routes if e2s[e] >= 0])
    cold = sorted([(t, e, wt) for t, e, wt in routes if e2s[e] < 0])
    assert r["n_hot"] == len(hot) and r["n_cold"] == len(cold) and r["n_hot"] + r["n_cold"] == M * k
    assert [(int(a), int(b), float(c)) for a, b, c in zip(r["hot_expert"], r["hot_token"], r["hot_w"])] == hot
    assert list(r["hot_slot"]) == [int(e2s[e]) for e, _, _ in hot]
    assert [(int(a), int(b), float(c)) for a, b, c in zip(r["cold_token"], r["cold_expert"], r["cold_w"])] == cold
    act = sorted(set(e for e, _, _ in hot))
    assert list(r["act_expert"]) == act
    assert list(r["act_cnt"]) == [sum(1 for e2, _, _ in hot if e2 == e) for e in act]
    assert list(r["act_off"]) == list(np.concatenate([[0], np.cumsum(r["act_cnt"])[:-1]]))
    assert np.array_equal(r["hist"], np.bincount(ids.ravel(), minlength=E))


def test_compaction_all_cold_and_all_hot(oracle_lib):
    ids = np.array([[1, 0], [2, 3]], dtype=np.int32)
    w = np.full((2, 2), 0.5, dtype=np.float32)
    r = oracle_lib.compact(ids, w, np.full(4, -1, dtype=np.int32))
    assert r["n_hot"] == 0 and r["n_active"] == 0 and r["n_cold"] == 4
    assert list(r["cold_expert"]) == [0, 1, 2, 3] and list(r["cold_token"]) == [0, 0, 1, 1]
    r = oracle_lib.compact(ids, w, np.array([3, 2, 1, 0], dtype=np.int32))
    assert r["n_cold"] == 0 and list(r["hot_expert"]) == [0, 1, 2, 3] and list(r["hot_slot"]) == [3, 2, 1, 0]


# ---------------------------------------------------------------- expert FFN


def _expert_f64(rec, H, I):
    s = sections(rec, H, I)
    Wg = decode_mxfp4_np(s["wg_codes"], s["wg_scales"], I, H)
    Wu = decode_mxfp4_np(s["wu_codes"], s["wu_scales"], I, H)
    Wd = decode_mxfp4_np(s["wd_codes"], s["wd_scales"], H, I)
    return Wg, Wu, Wd


def test_gate_up_within_fp32_bound(oracle_lib):
    H, I = 256, 128  # H != I: a transposed operand cannot pass
    rec = synth.expert_records(0, 0, 16, H, I, experts=[5])[0]
    x = synth.activations(0, 0, 1, 1, H)[0]
    h = oracle_lib.expert_gate_up(rec, H, I, x).astype(np.float64)
    Wg, Wu, _ = _expert_f64(rec, H, I)
    xf = bf16_to_f64(x)
    g, u = Wg @ xf, Wu @ xf  # products are exact in float64; the sum nearly so
    dg = (H + 1) * U32 * (np.abs(Wg) @ np.abs(xf))
    du = (H + 1) * U32 * (np.abs(Wu) @ np.abs(xf))
    silu = g / (1.0 + np.exp(-g))
    ref = silu * u
    bound = 1.1 * dg * np.abs(u) + np.abs(silu) * du + 16 * U32 * np.abs(ref) + 1e-30
    assert np.all(np.abs(h - ref) <= bound)


def test_down_within_fp32_bound(oracle_lib):
    H, I = 256, 128
    rec = synth.expert_records(0, 0, 16, H, I, experts=[3])[0]
    h = np.random.default_rng(1).standard_normal(I).astype(np.float32)
    y = oracle_lib.expert_down(rec, H, I, h).astype(np.float64)
    _, _, Wd = _expert_f64(rec, H, I)
    exact = Wd @ h.astype(np.float64)
    bound = (I + 1) * U32 * (np.abs(Wd) @ np.abs(h.astype(np.float64)))
    assert np.all(np.abs(y - exact) <= bound)


def test_ffn_permutation_weights_pick_columns(oracle_lib):
    # Wg = Wu = 1.0 * P (a permutation): g_i = u_i = x[p(i)], so h_i = SiLU(x)x;
    # Wd = identity-like on the first I rows picks h back out.
    H, I = 64, 32
    perm = np.random.default_rng(0).permutation(H)[:I]
    rec = np.zeros(synth.expert_bytes(H, I), dtype=np.uint8)
    s = sections(rec, H, I)
    for name in ("wg", "wu"):
        codes = s[name + "_codes"].reshape(I, H // 2)
        for i, c in enumerate(perm):
            codes[i, c // 2] = 2 << (4 * (c & 1))  # code 2 = 1.0
        s[name + "_scales"][:] = 127
    dcodes = s["wd_codes"].reshape(H, I // 2)
    for r in range(I):
        dcodes[r, r // 2] = 2 << (4 * (r & 1))
    s["wd_scales"][:] = 128  # 2.0
    x = synth.activations(0, 0, 2, 1, H)[0]
    xf = bf16_to_f64(x).astype(np.float32)
    h = oracle_lib.expert_gate_up(rec, H, I, x)
    xp = xf[perm]
    ref_h = (xp / (np.float32(1) + np.exp(-xp))) * xp
    assert np.allclose(h, ref_h, rtol=4e-7, atol=0)
    y = oracle_lib.expert_ffn(rec, H, I, x)
    assert np.array_equal(y[:I], 2 * h) and np.all(y[I:] == 0)


def test_silu_closed_forms(oracle_lib):
    # SiLU(0) = 0; SiLU(g) -> g for large g; SiLU(g) -> 0 for very negative g
    H, I = 32, 32
    rec = np.zeros(synth.expert_bytes(H, I), dtype=np.uint8)
    s = sections(rec, H, I)
    s["wg_scales"][:] = 127
    s["wu_scales"][:] = 127
    gc = s["wg_codes"].reshape(I, H // 2)
    uc = s["wu_codes"].reshape(I, H // 2)
    uc[:, 0] = 2  # u_i = x_0
    gc[1, 0] = 7  # g_1 = 6 x_0
    gc[2, 0] = 15  # g_2 = -6 x_0
    x = np.zeros(H, dtype=np.uint16)
    x[0] = 0x4120  # 10.0
    h = oracle_lib.expert_gate_up(rec, H, I, x)
    assert h[0] == 0.0  # g = 0
    assert abs(h[1] - 60.0 * 10.0) <= 1e-4 * 600  # SiLU(60) ~ 60
    assert abs(h[2]) < 1e-20  # SiLU(-60) ~ 0


# ------------------------------------------------------- whole-layer invariants


def _tiny_layer(seed=0, M=3, tau=0.0):
    w = synth.WORKLOADS["tiny_h256_i128_e16k2"]
    H, I, E, k = w.hidden, w.inter, w.experts, w.top_k
    x = synth.activations(seed, 0, 0, M, H)
    Wr = synth.router_weights(seed, 0, E, H)
    b = synth.router_bias(seed, 0, E, tau)
    ex = synth.expert_records(seed, 0, E, H, I)
    return x, Wr, b, ex, H, I, E, k


def test_hot_plus_cold_equals_all_resident(oracle_lib):
    x, Wr, b, ex, H, I, E, k = _tiny_layer(M=6)
    full = oracle_lib.moe_layer(x, Wr, b, ex, np.arange(E, dtype=np.int32), k, H, I)
    e2s = np.full(E, -1, dtype=np.int32)
    e2s[::3] = np.arange(len(e2s[::3]))
    part = oracle_lib.moe_layer(x, Wr, b, ex, e2s, k, H, I)
    assert part["n_cold"] > 0 and part["n_hot"] > 0
    assert np.array_equal(part["ids"], full["ids"]) and np.array_equal(part["w"], full["w"])
    recon = part["out_f32"].astype(np.float64).copy()
    mag = np.zeros_like(recon)
    for t, e, wt in zip(part["cold_token"], part["cold_expert"], part["cold_w"]):
        y = oracle_lib.expert_ffn(ex[e], H, I, x[t]).astype(np.float64)
        recon[t] += wt * y
        mag[t] += np.abs(wt * y)
    for t, e, wt in zip(part["hot_token"], part["hot_expert"], part["hot_w"]):
        mag[t] += np.abs(wt * oracle_lib.expert_ffn(ex[e], H, I, x[t]).astype(np.float64))
    assert np.all(np.abs(recon - full["out_f32"]) <= 4 * (k + 1) * U32 * mag + 1e-30)


def test_single_route_output_is_expert_output(oracle_lib):
    # top_k = 1: the weight is exactly 1, the output is y of the chosen expert
    x, Wr, b, ex, H, I, E, _ = _tiny_layer(M=2)
    r = oracle_lib.moe_layer(x, Wr, b, ex, np.arange(E, dtype=np.int32), 1, H, I)
    for t in range(2):
        y = oracle_lib.expert_ffn(ex[r["ids"][t, 0]], H, I, x[t])
        assert np.array_equal(r["out_f32"][t], y)


def test_all_cold_layer_outputs_zero(oracle_lib):
    x, Wr, b, ex, H, I, E, k = _tiny_layer(M=2)
    r = oracle_lib.moe_layer(x, Wr, b, ex, np.full(E, -1, dtype=np.int32), k, H, I)
    assert r["n_hot"] == 0 and np.all(r["out_f32"] == 0) and r["n_cold"] == 2 * k


# ------------------------------------------------------------------ slot cache


def _read_trace(name):
    lines = [l.split() for l in open(os.path.join(GOLDEN, name)) if l.strip() and l[0] != "#"]
    hdr = lines[0]
    E, S, R, decay = int(hdr[1]), int(hdr[3]), int(hdr[5]), float(hdr[7])
    policy = hdr[9] if len(hdr) > 9 else "freq"
    init = [int(v) for v in lines[1][1:]]
    steps = []
    for l in lines[2:]:
        st = int(l[1])
        i_p, i_m = l.index("pairs"), l.index("map")
        hist = [int(v) for v in l[3:i_p]]
        pairs = [tuple(int(q) for q in p.split(":")) for p in l[i_p + 1:i_m]]
        mp = [int(v) for v in l[i_m + 1:]]
        steps.append((st, hist, pairs, mp))
    return E, S, R, decay, init, steps, policy


@pytest.mark.parametrize("trace", ["cache_lfu_trace.txt", "cache_lfru_trace.txt", "cache_lru_trace.txt",
                                   "cache_fifo_trace.txt", "cache_slru_trace.txt"])
def test_cache_policy_hand_worked_trace(oracle_lib, trace):
    E, S, R, decay, init, steps, policy = _read_trace(trace)
    rp = oracle_lib.CacheReplay(np.array(init, dtype=np.int32), S, decay=decay, R=R, policy=policy)
    for st, hist, pairs, mp in steps:
        got = rp.step(np.array(hist, dtype=np.int32), st)
        assert got == pairs, (trace, st)
        assert list(rp.e2s) == mp, (trace, st)


def test_cache_policy_never_exceeds_budget_and_keeps_map_injective(oracle_lib):
    rng = np.random.default_rng(11)
    E, S, R = 32, 16, 2
    rp = oracle_lib.CacheReplay(np.where(np.arange(E) < S, np.arange(E), -1).astype(np.int32), S, R=R)
    for st in range(200):
        hist = np.bincount(rng.choice(E, 4, replace=False, p=None), minlength=E).astype(np.int32)
        pairs = rp.step(hist, st)
        assert len(pairs) <= R
        res = rp.e2s[rp.e2s >= 0]
        assert len(res) == S and len(set(res.tolist())) == S
        assert all(rp.s2e[rp.e2s[e]] == e for e in range(E) if rp.e2s[e] >= 0)


@pytest.mark.parametrize("policy", ["lru", "fifo"])
def test_recency_policies_keep_budget_and_map(oracle_lib, policy):
    rng = np.random.default_rng(13)
    E, S, R = 32, 16, 2
    rp = oracle_lib.CacheReplay(np.where(np.arange(E) < S, np.arange(E), -1).astype(np.int32), S, R=R,
                                policy=policy)
    for st in range(200):
        hist = np.bincount(rng.choice(E, 4, replace=False), minlength=E).astype(np.int32)
        pairs = rp.step(hist, st)
        assert len(pairs) <= R
        res = rp.e2s[rp.e2s >= 0]
        assert len(res) == S and len(set(res.tolist())) == S
        for e, _slot, v in pairs:
            assert hist[e] > 0  # only experts this step routed come in
            if policy == "lru":
                assert hist[v] == 0  # LRU never evicts an expert this step routed


def test_slru_segments_keep_capacity_budget_and_map(oracle_lib):
    rng = np.random.default_rng(17)
    E, S, R = 32, 16, 2
    rp = oracle_lib.CacheReplay(np.where(np.arange(E) < S, np.arange(E), -1).astype(np.int32), S, R=R,
                                policy="slru")
    assert rp.pcap == 12
    for st in range(300):
        hist = np.bincount(rng.choice(E, 4, replace=False), minlength=E).astype(np.int32)
        before = rp.e2s.copy()
        pairs = rp.step(hist, st)
        assert len(pairs) <= R
        res = np.flatnonzero(rp.e2s >= 0)
        assert len(res) == S and len(set(rp.e2s[res].tolist())) == S
        assert int(rp.seg[res].sum()) <= rp.pcap and not rp.seg[rp.e2s < 0].any()
        for e, _slot, v in pairs:
            assert hist[e] > 0 and hist[v] == 0 and before[e] < 0 and rp.seg[e] == 0
        for e in np.flatnonzero((hist > 0) & (before >= 0)):
            # a hit is protected after the step unless demoted for the capacity, which only happens when
            # every protected expert was routed this step
            if not rp.seg[e]:
                assert all(hist[p] > 0 for p in np.flatnonzero(rp.seg))


def test_slru_without_a_protected_segment_is_lru(oracle_lib):
    # pcap = 0: no protected segment, victims by recency alone = the LRU replay, step for step
    rng = np.random.default_rng(19)
    E, S, R = 12, 5, 2
    init = np.where(np.arange(E) < S, np.arange(E), -1).astype(np.int32)
    a = oracle_lib.CacheReplay(init, S, R=R, policy="slru", pcap=0)
    b = oracle_lib.CacheReplay(init, S, R=R, policy="lru")
    for st in range(200):
        hist = np.bincount(rng.choice(E, 3, replace=False), minlength=E).astype(np.int32)
        assert a.step(hist, st) == b.step(hist, st)
        assert np.array_equal(a.e2s, b.e2s)


def test_lru_with_every_resident_routed_takes_no_pair(oracle_lib):
    rp = oracle_lib.CacheReplay(np.array([0, 1, -1], dtype=np.int32), 2, R=2, policy="lru")
    assert rp.step(np.array([1, 1, 1], dtype=np.int32), 0) == []
    rp = oracle_lib.CacheReplay(np.array([0, 1, -1], dtype=np.int32), 2, R=2, policy="fifo")
    assert rp.step(np.array([1, 1, 1], dtype=np.int32), 0) == [(2, 0, 0)]


def test_cache_in_flight_experts_are_skipped(oracle_lib):
    rp = oracle_lib.CacheReplay(np.array([0, 1, -1, -1], dtype=np.int32), 2, R=2)
    fl = np.array([0, 0, 1, 0], dtype=np.uint8)  # expert 2's copy has not landed
    pairs = rp.step(np.array([0, 0, 5, 3], dtype=np.int32), 0, in_flight=fl)
    assert pairs == [(3, 0, 0)]


# ------------------------------------------------------- prefill activation format


def e4m3_from_bits(code):
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * m / 8.0 * 2.0 ** -6
    return s * (1 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_exhaustive_and_fixture(oracle_lib):
    for c in range(256):
        a, b = oracle_lib.e4m3(c), e4m3_from_bits(c)
        assert (math.isnan(a) and math.isnan(b)) or a == b, c
    for l in open(os.path.join(GOLDEN, "e4m3_points.txt")):
        if l[0] == "#":
            continue
        c, v = l.split()
        assert oracle_lib.e4m3(int(c, 16)) == float(v)


def test_e4m3_encode_round_trip_rne_and_saturation(oracle_lib):
    for c in range(256):
        v = e4m3_from_bits(c)
        if math.isnan(v) or v == 0:
            continue
        assert oracle_lib.e4m3(oracle_lib.e4m3_encode(v)) == v
    assert oracle_lib.e4m3(oracle_lib.e4m3_encode(1.0625)) == 1.0  # tie -> even mantissa
    assert oracle_lib.e4m3(oracle_lib.e4m3_encode(1.1875)) == 1.25
    assert oracle_lib.e4m3(oracle_lib.e4m3_encode(500.0)) == 448.0
    assert oracle_lib.e4m3(oracle_lib.e4m3_encode(-1e9)) == -448.0


def test_mxfp8_block_rule(oracle_lib):
    # powers of two within the block's range come back exactly
    v = np.array([2.0 ** j for j in range(-6, 2)] * 4, dtype=np.float32)
    sc, codes = oracle_lib.mxfp8_block(v)
    assert sc == 127 + (1 - 8)  # floor(log2 2) - 8 = -7
    back = np.array([oracle_lib.e4m3(c) for c in codes]) * 2.0 ** (sc - 127)
    assert np.array_equal(back, v)
    # an all-equal block
    sc, codes = oracle_lib.mxfp8_block(np.full(32, 1.5, dtype=np.float32))
    assert sc == 127 - 8 and all(oracle_lib.e4m3(c) * 2.0 ** (sc - 127) == 1.5 for c in codes)
    # zeros
    sc, codes = oracle_lib.mxfp8_block(np.zeros(32, dtype=np.float32))
    assert sc == 0 and np.all(codes == 0)



# ------------------------------------------------- prefill expert FFN (MXFP8 activations)


def e4m3_rne_np(s):
    """Round float64 values to the E4M3 grid, nearest with ties to an even mantissa, saturating at
    +-448; computed from the format's spacing (3 mantissa bits, normal from 2^-6, subnormal step
    2^-9), not from a code table."""
    s = np.asarray(s, dtype=np.float64)
    a = np.abs(s)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.where(a >= 2.0 ** -6, np.ldexp(1.0, (np.maximum(e, -6) - 3).astype(np.int64)), 2.0 ** -9)
    q = np.round(a / step) * step  # numpy rounds halves to even: the even integer is the even mantissa
    return np.sign(s) * np.minimum(q, 448.0)


def mxfp8_quant_np(v):
    """OCP MX v1.0 MXFP8 conversion of a float64 vector in blocks of 32: shared exponent
    X = floor(log2 max|v|) - 8 (8 = E4M3's largest exponent), X = -127 for a zero block,
    elements E4M3(v / 2^X).  Returns the dequantised values and X per block."""
    v = np.asarray(v, dtype=np.float64).reshape(-1, 32)
    amax = np.abs(v).max(axis=1)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    X = np.where(amax > 0, np.clip(ex - 1 - 8, -127, 127), -127)
    sc = np.ldexp(1.0, X)[:, None]
    return (e4m3_rne_np(v / sc) * sc).reshape(-1), X


def test_mxfp8_quantiser_restatement_agrees_with_the_oracle_block_rule(oracle_lib):
    # the numpy quantiser used below against the oracle's block rule, on bf16-exact blocks of many
    # magnitudes (any disagreement here would make the FFN pin below meaningless)
    rng = np.random.default_rng(7)
    for t in range(200):
        v = (rng.standard_normal(32) * 2.0 ** rng.integers(-20, 20, size=32)).astype(np.float32)
        if t % 5 == 0:
            v[rng.integers(0, 32)] = 0
        sc, codes = oracle_lib.mxfp8_block(v)
        back = np.array([e4m3_from_bits(int(c)) for c in codes]) * 2.0 ** (int(sc) - 127)
        ref, X = mxfp8_quant_np(v.astype(np.float64))
        assert int(sc) - 127 == X[0]
        assert np.array_equal(back, ref)


def _ffn_mxfp8_reference(rec, H, I, x):
    """float64 restatement of the prefill reading of the expert FFN from independent decoders:
    xq = MXFP8(x) in 32-element blocks along H; g = Wg xq, u = Wu xq; h = SiLU(g) u;
    hq = MXFP8(h) in 32-element blocks along I; y = Wd hq.

    The oracle forms h in fp32, so an element of h that lies within the fp32 error bound of an E4M3
    rounding boundary may legitimately round either way.  Returns y for the float64 h, the bound
    on |y_oracle - y| (fp32 summation of both contractions plus the spread of those ambiguous
    elements), and the number of ambiguous elements."""
    Wg, Wu, Wd = _expert_f64(rec, H, I)
    xf = bf16_to_f64(x)
    xq, _ = mxfp8_quant_np(xf)
    g, u = Wg @ xq, Wu @ xq
    dg = (H + 1) * U32 * (np.abs(Wg) @ np.abs(xq))
    du = (H + 1) * U32 * (np.abs(Wu) @ np.abs(xq))
    sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    h = silu * u
    # mean value theorem: |SiLU(g') - SiLU(g)| <= (|SiLU'(g)| + 1/2 |g' - g|) |g' - g|, as |SiLU''| <= 1/2
    dsilu = (np.abs(sig * (1.0 + g * (1.0 - sig))) + 0.5 * dg) * dg
    dh = dsilu * (np.abs(u) + du) + np.abs(silu) * du + 16 * U32 * np.abs(h) + 1e-30
    hq, X = mxfp8_quant_np(h)
    lo, Xlo = mxfp8_quant_np(h - dh)
    hi, Xhi = mxfp8_quant_np(h + dh)
    amax_lo = np.maximum(np.abs(h) - dh, 0).reshape(-1, 32).max(axis=1)
    amax_hi = (np.abs(h) + dh).reshape(-1, 32).max(axis=1)
    _, e_lo = np.frexp(amax_lo)
    _, e_hi = np.frexp(amax_hi)
    assert np.array_equal(e_lo, e_hi), "a block scale of h is ambiguous at this seed"
    # the quantiser is monotone within a fixed block scale, so every admissible hq lies in [qlo, qhi]
    qlo = np.minimum(lo, hi)
    qhi = np.maximum(lo, hi)
    spread = qhi - qlo
    y = Wd @ hq
    bound = (I + 1) * U32 * (np.abs(Wd) @ np.maximum(np.abs(qlo), np.abs(qhi))) + np.abs(Wd) @ spread + 1e-30
    return y, bound, int(np.count_nonzero(spread)), h, hq


@pytest.mark.parametrize("H,I", [(256, 128), (128, 256), (320, 96)])
def test_ffn_mxfp8_against_float64_restatement(oracle_lib, H, I):
    # H != I both ways: a block axis or a transposed operand taken the wrong way cannot pass
    rec = synth.expert_records(3, 1, 8, H, I, experts=[6])[0]
    x = synth.activations(3, 1, 0, 1, H)[0]
    y = oracle_lib.expert_ffn_mxfp8(rec, H, I, x).astype(np.float64)
    ref, bound, n_amb, h, hq = _ffn_mxfp8_reference(rec, H, I, x)
    assert n_amb <= I // 16
    assert np.all(np.abs(y - ref) <= bound)
    # the bound is tight enough to tell the readings apart: leaving h unquantised, or quantising
    # x per element instead of per block, moves y far outside it
    Wg, Wu, Wd = _expert_f64(rec, H, I)
    assert np.mean(np.abs(Wd @ h - ref) > bound) > 0.5
    xf = bf16_to_f64(x)
    x_elem = np.concatenate([mxfp8_quant_np(np.repeat(v, 32))[0][:1] for v in xf])
    g2, u2 = Wg @ x_elem, Wu @ x_elem
    y2 = Wd @ mxfp8_quant_np(g2 / (1 + np.exp(-g2)) * u2)[0]
    assert np.mean(np.abs(y2 - ref) > bound) > 0.5


def test_ffn_mxfp8_gate_and_up_scales_are_their_own(oracle_lib):
    # Wg and Wu identical in codes but with different block scales: taking one section's scales
    # for the other changes h by a power of two per block
    H, I = 128, 64
    rec = synth.expert_records(5, 0, 4, H, I, experts=[1])[0].copy()
    s = sections(rec, H, I)
    s["wu_codes"][:] = s["wg_codes"]
    s["wu_scales"][:] = 120 + (s["wg_scales"].astype(np.int64) - 120 + 3) % 8
    x = synth.activations(5, 0, 0, 1, H)[0]
    y = oracle_lib.expert_ffn_mxfp8(rec, H, I, x).astype(np.float64)
    ref, bound, _, _, _ = _ffn_mxfp8_reference(rec, H, I, x)
    assert np.all(np.abs(y - ref) <= bound)


def _mxfp8_exact_token(rng, H):
    """bf16 values that MXFP8 represents exactly: each 32-block holds one +-3 (so X = 1 - 8 = -7) and
    other values m/8 * 2^e with m in 8..15, e in [-6, 1] (inside E4M3's normal range at that scale)."""
    v = (rng.integers(8, 16, size=H) / 8.0) * np.ldexp(1.0, rng.integers(-6, 2, size=H))
    v *= np.where(rng.random(H) < 0.5, -1.0, 1.0)
    v[::32] = np.where(rng.random(H // 32) < 0.5, -3.0, 3.0)
    bits = synth.bf16_bits_rne(v.astype(np.float32))
    assert np.array_equal(bf16_to_f64(bits), v)
    return bits


def test_ffn_mxfp8_equals_decode_ffn_on_mxfp8_exact_values(oracle_lib):
    # x exactly MXFP8-representable and h exactly MXFP8-representable: the prefill reading must give
    # the decode FFN's result bit for bit (quantisation is the identity there).
    # Wg row i picks 6 * 2^a_i * x_0 with x_0 = 3, so g_i = 18 * 2^a_i >= 18 and SiLU(g_i) = g_i in
    # fp32 (exp(-18) < 2^-25); Wu row i picks +-2^b_i * x_j for an x_j that is a power of two, so
    # h_i = g_i u_i has at most 4 significant bits.  Within each 32-block of h the exponents span
    # 5 binades, inside E4M3's range below the block maximum.
    H, I = 128, 96
    rng = np.random.default_rng(11)
    x = _mxfp8_exact_token(rng, H)
    x[0] = 0x4040  # x_0 = +3
    xf = bf16_to_f64(x)
    pow2 = [c for c in range(H) if c % 32 and np.log2(abs(xf[c])) == np.round(np.log2(abs(xf[c])))]
    assert len(pow2) >= 4
    rec = synth.expert_records(9, 0, 4, H, I, experts=[2])[0].copy()
    s = sections(rec, H, I)
    gc = s["wg_codes"].reshape(I, H // 2)
    uc = s["wu_codes"].reshape(I, H // 2)
    gs = s["wg_scales"].reshape(I, H // 32)
    us = s["wu_scales"].reshape(I, H // 32)
    gc[:] = 0
    uc[:] = 0
    for i in range(I):
        gc[i, 0] = 7  # code 7 = 6.0 in the low nibble: column 0
        gs[i, 0] = 127 + rng.integers(0, 3)
        c = pow2[rng.integers(0, len(pow2))]
        uc[i, c // 2] = (2 | (8 if rng.random() < 0.5 else 0)) << (4 * (c & 1))  # +-1.0
        us[i, c // 32] = 127 - rng.integers(0, 3)
    h = oracle_lib.expert_gate_up(rec, H, I, x).astype(np.float64)
    hq, _ = mxfp8_quant_np(h)
    assert np.array_equal(hq, h)  # the construction really is MXFP8-exact
    y8 = oracle_lib.expert_ffn_mxfp8(rec, H, I, x)
    y = oracle_lib.expert_ffn(rec, H, I, x)
    assert np.array_equal(y8.view(np.uint32), y.view(np.uint32))


# ---------------------------------------------------------------- demand-filled LRU slot table

def _read_demand_trace(name):
    lines = [l.split() for l in open(os.path.join(GOLDEN, name)) if l.strip() and l[0] != "#"]
    E, S = int(lines[0][1]), int(lines[0][3])
    init = [int(v) for v in lines[1][1:]]
    steps = []
    for l in lines[2:]:
        i_f, i_m = l.index("fills"), l.index("map")
        steps.append(([int(v) for v in l[3:i_f]], [tuple(int(q) for q in p.split(":")) for p in l[i_f + 1:i_m]],
                      [int(v) for v in l[i_m + 1:]]))
    return E, S, init, steps


def test_demand_lru_hand_worked_trace(oracle_lib):
    E, S, init, steps = _read_demand_trace("cache_demand_lru_trace.txt")
    rp = oracle_lib.DemandLRUReplay(np.array(init, dtype=np.int32), S)
    for i, (hist, fills, mp) in enumerate(steps):
        assert rp.step(np.array(hist, dtype=np.int32)) == fills, i
        assert list(rp.e2s) == mp, i


@pytest.mark.parametrize("S,init_fill", [(4, 4), (8, 3), (1, 1)])
def test_demand_lru_one_expert_per_step_is_a_textbook_lru_cache(oracle_lib, S, init_fill):
    # With one routed expert per step there are no ties within a step: the resident set must follow a
    # textbook LRU cache of capacity S (least recently used first out; initial experts in slot order count as
    # used before any step, the lower slot earlier), and the fills must be exactly its misses.
    from collections import OrderedDict
    rng = np.random.default_rng(21)
    E = 12
    init = np.full(E, -1, dtype=np.int32)
    init[:init_fill] = np.arange(init_fill)
    rp = oracle_lib.DemandLRUReplay(init, S)
    book = OrderedDict((e, None) for e in range(init_fill))
    for st in range(400):
        e = int(rng.zipf(1.3) - 1) % E
        hist = np.zeros(E, dtype=np.int32)
        hist[e] = 1 + int(rng.integers(0, 3))
        fills = rp.step(hist)
        miss = e not in book
        if miss:
            if len(book) == S:
                book.popitem(last=False)
            book[e] = None
        else:
            book.move_to_end(e)
        assert [f[0] for f in fills] == ([e] if miss else []), st
        assert set(np.nonzero(rp.e2s >= 0)[0].tolist()) == set(book), st


def test_demand_lru_invariants_on_random_steps(oracle_lib):
    rng = np.random.default_rng(23)
    E, S = 40, 12
    init = np.where(np.arange(E) < 10, np.arange(E), -1).astype(np.int32)  # two slots start empty
    rp = oracle_lib.DemandLRUReplay(init, S)
    for st in range(300):
        M, k = int(rng.integers(1, 5)), 4
        hist = np.zeros(E, dtype=np.int32)
        for _ in range(M):
            hist[rng.choice(E, k, replace=False)] += 1
        e2s0, s2e0, stamp0 = rp.e2s.copy(), rp.s2e.copy(), rp.stamp.copy()
        fills = rp.step(hist)
        routed = set(np.nonzero(hist)[0].tolist())
        hits = {e for e in routed if e2s0[e] >= 0}
        misses = routed - hits
        # every miss that can be served is, and only those
        free = [s for s in range(S) if s2e0[s] < 0 or hist[s2e0[s]] == 0]
        assert len(fills) == min(len(misses), len(free)), st
        assert {f[0] for f in fills} <= misses and len({f[1] for f in fills}) == len(fills), st
        # served misses: most routes first; victims: slots this step did not route, empty first, oldest stamp
        served = [f[0] for f in fills]
        assert all(hist[a] >= hist[b] for a, b in zip(served, served[1:])), st
        if len(fills) < len(misses):
            assert min(hist[e] for e in served) >= max(hist[e] for e in misses - set(served)), st
        key = {s: (-2 if s2e0[s] < 0 else stamp0[s]) for s in free}
        used = [f[1] for f in fills]
        assert all(s in key for s in used), st
        assert max((key[s] for s in used), default=-3) <= min((key[s] for s in free if s not in used),
                                                               default=1 << 40), st
        # map: injective, s2e its inverse, every hit unchanged, every routed expert resident when it fits
        res = rp.e2s[rp.e2s >= 0]
        assert len(set(res.tolist())) == len(res)
        assert all(rp.s2e[rp.e2s[e]] == e for e in range(E) if rp.e2s[e] >= 0)
        assert all(rp.e2s[e] == e2s0[e] for e in hits), st
        if len(routed) <= S:
            assert all(rp.e2s[e] >= 0 for e in routed), st
        # stamps: every slot used this step carries the step
        assert all(rp.stamp[rp.e2s[e]] == st for e in routed if rp.e2s[e] >= 0), st


# --------------------------------------------------------------------- NVFP4


def decode_nvfp4_np(codes, scales, R, C):
    """float64 decode of an NVFP4 matrix from bit fields: E2M1 codes (low nibble first), one E4M3 scale per
    16 columns, both decoded by this file's bit-field decoders (pinned to the OCP fixtures above)."""
    codes = codes.reshape(R, C // 2)
    q = np.empty((R, C), dtype=np.int64)
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    mag = np.vectorize(e2m1_from_bits)(q)
    sc = np.vectorize(e4m3_from_bits)(scales.reshape(R, C // 16).astype(np.int64))
    return mag * np.repeat(sc, 16, axis=1)


def test_nvfp4_exhaustive_codes_times_e4m3_scales(oracle_lib):
    # every (code, scale byte) pair: element = E2M1(code) * E4M3(scale), NaN scales give NaN
    codes = np.array([(2 * j) | ((2 * j + 1) << 4) for j in range(8)], dtype=np.uint8)  # codes 0..15, one row
    for sb in range(256):
        scales = np.array([sb], dtype=np.uint8)
        W = oracle_lib.nvfp4_dequant(codes, scales, 1, 16)[0]
        for c in range(16):
            ref = e2m1_from_bits(c) * e4m3_from_bits(sb)
            assert (math.isnan(ref) and math.isnan(W[c])) or W[c] == ref, (c, sb)


def test_nvfp4_sixteen_column_blocks_and_nibble_order(oracle_lib):
    # a scale per 16 columns (not 32) and rows not transposed: distinct scales on every block of a 3 x 64 matrix
    rng = np.random.default_rng(7)
    R, C = 3, 64
    codes = rng.integers(0, 256, R * C // 2, dtype=np.uint8)
    scales = np.array([0x30 + 3 * i for i in range(R * C // 16)], dtype=np.uint8)
    W = oracle_lib.nvfp4_dequant(codes, scales, R, C).astype(np.float64)
    assert np.array_equal(W, decode_nvfp4_np(codes, scales, R, C))


def test_nvfp4_record_size(oracle_lib):
    for H, I in [(256, 128), (2880, 2880), (2048, 512)]:
        assert oracle_lib.expert_bytes(H, I, "nvfp4") == 3 * I * H * 9 // 16 == synth.expert_bytes(H, I, 1)
        assert oracle_lib.expert_bytes(H, I) == 3 * I * H * 17 // 32 == synth.expert_bytes(H, I)


def test_nvfp4_ffn_within_fp32_bound(oracle_lib):
    H, I = 256, 128
    rec = synth.expert_records(0, 0, 16, H, I, experts=[2], weight_format=1)[0]
    x = synth.activations(0, 0, 5, 1, H)[0]
    y = oracle_lib.expert_ffn(rec, H, I, x, "nvfp4").astype(np.float64)
    offs = synth.section_offsets(H, I, 1)
    sec = {k: rec[o:o + n] for k, (o, n) in offs.items()}
    Wg = decode_nvfp4_np(sec["wg_codes"], sec["wg_scales"], I, H)
    Wu = decode_nvfp4_np(sec["wu_codes"], sec["wu_scales"], I, H)
    Wd = decode_nvfp4_np(sec["wd_codes"], sec["wd_scales"], H, I)
    xf = bf16_to_f64(x)
    g, u = Wg @ xf, Wu @ xf
    h = g / (1.0 + np.exp(-g)) * u
    ref = Wd @ h
    # fp32 sums of H and I terms: a loose but sure bound, relative to the sum of magnitudes
    dh = 4 * (H + 8) * U32 * ((np.abs(Wg) @ np.abs(xf)) * np.abs(u) + np.abs(g) * (np.abs(Wu) @ np.abs(xf)))
    bound = (I + 8) * U32 * (np.abs(Wd) @ np.abs(h)) + np.abs(Wd) @ dh + 1e-30
    assert np.all(np.abs(y - ref) <= bound)


def test_nvfp4_unit_scales_equal_mxfp4_unit_scales(oracle_lib):
    # with every scale 1 (E4M3 0x38, E8M0 127) the two formats hold the same matrices: same layer output, bit for bit
    H, I, E, k = 256, 128, 8, 2
    mx = synth.expert_records(0, 1, E, H, I)
    nv = np.empty((E, synth.expert_bytes(H, I, 1)), dtype=np.uint8)
    om, on = synth.section_offsets(H, I), synth.section_offsets(H, I, 1)
    for name in ("wg", "wu", "wd"):
        (o1, n1), (o2, n2) = om[name + "_codes"], on[name + "_codes"]
        nv[:, o2:o2 + n2] = mx[:, o1:o1 + n1]
        (s1, l1), (s2, l2) = om[name + "_scales"], on[name + "_scales"]
        mx[:, s1:s1 + l1] = 127
        nv[:, s2:s2 + l2] = 0x38
    x = synth.activations(0, 1, 9, 3, H)
    Wr = synth.router_weights(0, 1, E, H)
    e2s = np.arange(E, dtype=np.int32)
    a = oracle_lib.moe_layer(x, Wr, None, mx, e2s, k, H, I)
    b = oracle_lib.moe_layer(x, Wr, None, nv, e2s, k, H, I, fmt="nvfp4")
    assert np.array_equal(a["out_f32"], b["out_f32"]) and np.abs(a["out_f32"]).max() > 0


# ------------------------------------------------------------ next-layer prefetch


def test_prefetch_hand_worked_cases(oracle_lib):
    # E = 6, S = 3, experts 0, 1, 2 in slots 0, 1, 2
    e2s = [0, 1, 2, -1, -1, -1]
    zero, never = np.zeros(6), np.full(6, -1, dtype=np.int64)
    # predicted: 2 (resident), 3 twice, 4 once -> 3 then 4 come in; victims 0 then 1 (ties: lower slot)
    pairs, m = oracle_lib.prefetch_step(zero, never, e2s, 3, [0, 0, 1, 2, 1, 0], 2)
    assert pairs == [(3, 0, 0), (4, 1, 1)] and list(m) == [-1, -1, 2, 0, 1, -1]
    # R = 1 keeps the most predicted; the victim is the lowest score (expert 1), not the lowest slot
    pairs, _ = oracle_lib.prefetch_step([5.0, 1.0, 3.0, 0, 0, 0], never, e2s, 3, [0, 0, 0, 1, 3, 1], 1)
    assert pairs == [(4, 1, 1)]
    # equal predictions: higher score first, then lower id; equal scores: least recently routed victim
    pairs, _ = oracle_lib.prefetch_step([2.0, 2.0, 2.0, 1.0, 4.0, 1.0], [7, 3, 5, -1, -1, -1], e2s, 3,
                                        [0, 0, 0, 1, 1, 1], 3)
    assert pairs == [(4, 1, 1), (3, 2, 2), (5, 0, 0)]
    # an expert in flight is neither a candidate nor a victim; predicted residents are never victims
    pairs, _ = oracle_lib.prefetch_step(zero, never, e2s, 3, [1, 0, 1, 1, 1, 0], 3,
                                        in_flight=np.array([0, 0, 0, 1, 0, 0], dtype=np.uint8))
    assert pairs == [(4, 1, 1)]


def test_prefetch_invariants_on_random_steps(oracle_lib):
    rng = np.random.default_rng(11)
    for _ in range(300):
        E = int(rng.integers(4, 40))
        S = int(rng.integers(1, E + 1))
        e2s = np.full(E, -1, dtype=np.int32)
        e2s[rng.choice(E, S, replace=False)] = rng.permutation(S)
        score = rng.integers(0, 5, E).astype(np.float64)
        last = rng.integers(-1, 6, E).astype(np.int64)
        pred = np.where(rng.random(E) < 0.3, rng.integers(1, 4, E), 0).astype(np.int32)
        fl = (rng.random(E) < 0.1).astype(np.uint8)
        R = int(rng.integers(0, 5))
        pairs, m = oracle_lib.prefetch_step(score, last, e2s, S, pred, R, in_flight=fl)
        cands = [e for e in range(E) if pred[e] > 0 and e2s[e] < 0 and not fl[e]]
        vics = [e for e in range(E) if e2s[e] >= 0 and pred[e] == 0 and not fl[e]]
        assert len(pairs) == min(R, len(cands), len(vics))
        for ce, sl, ve in pairs:
            assert ce in cands and ve in vics and e2s[ve] == sl and m[ce] == sl and m[ve] == -1
        assert all(m[e] == e2s[e] for e in range(E) if pred[e] > 0 and e2s[e] >= 0)  # predicted residents stay
        slots = m[m >= 0]
        assert len(slots) == len(set(slots.tolist())) == S  # injective, every slot still used


def test_prefetching_the_exact_routes_makes_them_resident(oracle_lib):
    # when the prediction is the step's routing and R covers the misses, the step then finds every route hot
    rng = np.random.default_rng(5)
    for _ in range(50):
        E, S, k = 16, 8, 3
        e2s = np.full(E, -1, dtype=np.int32)
        e2s[rng.choice(E, S, replace=False)] = rng.permutation(S)
        routed = rng.choice(E, k, replace=False)
        pred = np.zeros(E, dtype=np.int32)
        pred[routed] = 1
        _, m = oracle_lib.prefetch_step(np.zeros(E), np.full(E, -1, dtype=np.int64), e2s, S, pred, k)
        assert all(m[e] >= 0 for e in routed)



def test_residual_stream_inputs_are_seeded_and_correlated():
    # the next-layer prefetch line's stand-in for a residual stream: x_l = rho x_(l-1) + sqrt(1 - rho^2) e_l
    a = synth.activations_residual(0, 3, 6, 2, 2048, 0.9)
    assert np.array_equal(a, synth.activations_residual(0, 3, 6, 2, 2048, 0.9))
    x = bf16_to_f64(a)
    for l in range(1, 6):
        c = np.corrcoef(x[l - 1].ravel(), x[l].ravel())[0, 1]
        assert abs(c - 0.9) < 0.02
        assert abs(np.std(x[l]) - 1.0) < 0.05
    assert abs(np.corrcoef(x[0].ravel(), x[5].ravel())[0, 1] - 0.9 ** 5) < 0.03
