"""Comparison helpers for the GPU parity tests (GPU result vs CPU oracle)."""
from __future__ import annotations

import ctypes

import numpy as np

NEAR_TIE = 1e-4  # k-th vs (k+1)-th logit gap below which a token's routing is not compared exactly
# fp32 logits summed in another order differ by a random walk of roundings: about u * 0.02 * H / sqrt(2)
# ~ 2.4e-6 per side for H = 2880 (router rows ~N(0, 0.02^2), x ~N(0, 1), u = 2^-24), so up to ~1.5e-5
# at 4 sigma over thousands of tokens (far inside NEAR_TIE).  The softmax turns logit differences d
# into relative weight differences of at most 2 max|d|: 5e-5 covers that with margin.
W_RTOL, W_ATOL = 5e-5, 1e-8
REL_TOL = 2e-3
RHO = 1e-2  # per-token floor: RHO * RMS of the token's oracle row


class _DevArray:
    """Exposes a raw device pointer to torch through __cuda_array_interface__."""

    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 3, "strides": None}


def dev_bytes(ptr, n):
    import torch

    if n == 0:
        return np.zeros(0, dtype=np.uint8)
    return torch.as_tensor(_DevArray(ptr, n, "|u1"), device="cuda").cpu().numpy().copy()


def dev_i32(ptr, n):
    import torch

    if n == 0:
        return np.zeros(0, dtype=np.int32)
    return torch.as_tensor(_DevArray(ptr, n, "<i4"), device="cuda").cpu().numpy().copy()


def dev_f32(ptr, n):
    return dev_i32(ptr, n).view(np.float32)


def _host(ptr, n, ct):
    if n == 0:
        return np.zeros(0)
    return np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(ct)), (n,)).copy()


def route_arrays(res, E, k):
    """Reads a moe_route_result back to numpy (synchronises)."""
    import torch

    torch.cuda.synchronize()
    counts = dev_i32(res.counts, 4)
    n_hot, n_cold, n_act, M = (int(c) for c in counts)
    out = {
        "counts": counts,
        "ids": dev_i32(res.topk_ids, M * k).reshape(M, k),
        "w": dev_f32(res.topk_w, M * k).reshape(M, k),
        "hot_expert": dev_i32(res.hot_expert, n_hot), "hot_token": dev_i32(res.hot_token, n_hot),
        "hot_w": dev_f32(res.hot_w, n_hot),
        "act_expert": dev_i32(res.act_expert, n_act), "act_slot": dev_i32(res.act_slot, n_act),
        "act_off": dev_i32(res.act_off, n_act), "act_cnt": dev_i32(res.act_cnt, n_act),
        "cold_token": dev_i32(res.cold_token, n_cold), "cold_expert": dev_i32(res.cold_expert, n_cold),
        "cold_w": dev_f32(res.cold_w, n_cold),
        "hist": dev_i32(res.hist, E),
    }
    # the page-locked mirror must equal the device arrays
    out["mirror_ok"] = (np.array_equal(_host(res.h_counts, 4, ctypes.c_int32), counts)
                        and np.array_equal(_host(res.h_hist, E, ctypes.c_int32), out["hist"])
                        and np.array_equal(_host(res.h_cold_token, n_cold, ctypes.c_int32), out["cold_token"])
                        and np.array_equal(_host(res.h_cold_expert, n_cold, ctypes.c_int32), out["cold_expert"])
                        and np.array_equal(_host(res.h_cold_w, n_cold, ctypes.c_float), out["cold_w"]))
    return out


def near_tie_tokens(logits, k):
    s = -np.sort(-logits.astype(np.float64), axis=1)
    if s.shape[1] <= k:
        return np.zeros(s.shape[0], dtype=bool)
    return (s[:, k - 1] - s[:, k]) < NEAR_TIE


def route_weight_rtol(x_bits, Wr, bias=None):
    """Per-token relative tolerance of the routing weights, from the token's own logit sums.

    Two fp32 sums of the same products in different orders differ by a random walk of roundings, each
    of size u |S_i| for the partial sums S_i: about u sqrt(sum_i S_i^2) per side.  The softmax turns
    logit differences d into relative weight differences of at most 2 max|d|; at 4 sigma, with both sides'
    walks: 8 sqrt(2) u max_e sqrt(sum_i S_ei^2), the partial sums taken in ascending order in float64,
    never below W_RTOL.  For N(0, 1) tokens at H = 2880 it gives 5e-5 to 7e-5 (about W_RTOL); an outlier
    of 2^10 in one block makes the later partial sums ~20x larger (~1.5e-3), one outlier of up to 2^12 in
    every block ~100x (up to ~2e-2, where the softmax is so peaked that all but the top weight are tiny).
    The output values are still held to 2e-3, so a weight error that mattered would show there."""
    x = ((np.asarray(x_bits).astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
    W = np.asarray(Wr, dtype=np.float64)
    out = np.empty(x.shape[0])
    for t in range(x.shape[0]):
        S = np.cumsum(x[t][None, :] * W, axis=1)
        if bias is not None:
            S = S + np.asarray(bias, dtype=np.float64)[:, None]
        walk = np.sqrt((S * S).sum(axis=1)).max()
        out[t] = max(W_RTOL, 8 * np.sqrt(2) * 2.0 ** -24 * walk)
    return out


def combine_with_weights(ids, w, ys):
    """Oracle combine of the given expert outputs with the given routing weights: per token, the fp32 sum in
    ascending expert order of w_e * y_e.  ids, w: [M, k]; ys: [M, k, H] (fp32)."""
    M, k = ids.shape
    out = np.zeros((M, ys.shape[2]), dtype=np.float32)
    for t in range(M):
        acc = np.zeros(ys.shape[2], dtype=np.float32)
        for j in np.argsort(ids[t], kind="stable"):
            acc = (acc + np.float32(w[t][j]) * ys[t][j].astype(np.float32)).astype(np.float32)
        out[t] = acc
    return out


def compare_routing(g, o, logits, k, e2s, w_rtol=None):
    """Routing indices, compaction and miss lists: bit-exact except near-tie tokens.  ``w_rtol``: per-token
    relative tolerance of the routing weights (default W_RTOL for every token; see route_weight_rtol).

    Returns the set of excluded tokens (near ties whose selection differs)."""
    M = o["ids"].shape[0]
    rt = np.full(M, W_RTOL) if w_rtol is None else np.asarray(w_rtol, dtype=np.float64)
    tie = near_tie_tokens(logits, k)
    excluded = set()
    for t in range(M):
        same = set(g["ids"][t].tolist()) == set(o["ids"][t].tolist())
        if not same:
            assert tie[t], f"token {t}: GPU experts {sorted(g['ids'][t])} vs oracle {sorted(o['ids'][t])}"
            excluded.add(t)
            continue
        gw = dict(zip(g["ids"][t].tolist(), g["w"][t].tolist()))
        ow = dict(zip(o["ids"][t].tolist(), o["w"][t].tolist()))
        for e in ow:
            assert abs(gw[e] - ow[e]) <= W_ATOL + rt[t] * abs(ow[e]), (t, e, gw[e], ow[e], rt[t])

    def keep(tokens):
        return np.array([t not in excluded for t in tokens], dtype=bool)

    if not excluded:
        assert np.array_equal(g["hist"], o["hist"])
        assert g["counts"][0] == o["n_hot"] and g["counts"][1] == o["n_cold"] and g["counts"][2] == o["n_active"]
        assert np.array_equal(g["act_expert"], o["act_expert"]) and np.array_equal(g["act_slot"], o["act_slot"])
        assert np.array_equal(g["act_off"], o["act_off"]) and np.array_equal(g["act_cnt"], o["act_cnt"])
    kg, ko = keep(g["hot_token"]), keep(o["hot_token"])
    assert np.array_equal(g["hot_expert"][kg], o["hot_expert"][ko])
    assert np.array_equal(g["hot_token"][kg], o["hot_token"][ko])
    ow = o["hot_w"][ko]
    assert np.all(np.abs(g["hot_w"][kg] - ow) <= W_ATOL + rt[o["hot_token"][ko]] * np.abs(ow))
    kg, ko = keep(g["cold_token"]), keep(o["cold_token"])
    assert np.array_equal(g["cold_token"][kg], o["cold_token"][ko])
    assert np.array_equal(g["cold_expert"][kg], o["cold_expert"][ko])
    ow = o["cold_w"][ko]
    assert np.all(np.abs(g["cold_w"][kg] - ow) <= W_ATOL + rt[o["cold_token"][ko]] * np.abs(ow))
    assert all(e2s[e] < 0 for e in g["cold_expert"]) and all(e2s[e] >= 0 for e in g["hot_expert"])
    return excluded


def bf16_half_ulp(r):
    a = np.abs(r.astype(np.float32)).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))  # half of 2^(e-7)


def compare_values(gpu, ref_f32, out_f32, exclude=()):
    """|g - r| <= 2e-3 * max(|r|, rho_t) (+ half a bf16 ulp of r for bf16 outputs).

    rho_t = 1e-2 * RMS of token t's oracle row guards outputs that cancel to
    near zero; r is the oracle's fp32 value before rounding.  Returns the
    largest ratio of error to allowance."""
    g = gpu.astype(np.float64)
    r = ref_f32.astype(np.float64)
    rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True))
    allow = REL_TOL * np.maximum(np.abs(r), RHO * rms)
    if not out_f32:
        allow = allow + bf16_half_ulp(r)
    allow = np.maximum(allow, 1e-30)
    ratio = np.abs(g - r) / allow
    for t in exclude:
        ratio[t] = 0
    worst = float(ratio.max()) if ratio.size else 0.0
    assert worst <= 1.0, f"max error/allowance {worst:.3f} at {np.unravel_index(ratio.argmax(), ratio.shape)}"
    return worst


# ---------------------------------------------------------------- inputs with outliers (test inputs only)


def outlier_tokens(seed, M, H):
    """bf16 bits [M, H] of N(0, 1) activations with outliers, cycling over three patterns per token:
    0. one 32-element block holds a single +-2^10 among values N(0, 1) * 2^-8 (a 2^18 range: the two E4M3
       terms of x cannot hold the small ones exactly);
    1. every block holds one outlier +-2^e (e in 4..12) among values N(0, 1) * 2^-6;
    2. alternate blocks scaled by 2^8 and 2^-8 (each block ordinary inside, wide range across blocks).
    The outliers make g, u and hence h span a wide range within 32-row blocks too."""
    from expert_offload_moe_gb300 import synth

    rng = np.random.default_rng(np.random.SeedSequence([seed, 77]))
    x = rng.standard_normal((M, H))
    nb = H // 32
    for t in range(M):
        blocks = x[t].reshape(nb, 32)
        mode = t % 3
        if mode == 0:
            b = (7 * t + 3) % nb
            blocks[b] *= 2.0 ** -8
            blocks[b, (5 * t) % 32] = (1 if t % 2 else -1) * 2.0 ** 10
        elif mode == 1:
            blocks *= 2.0 ** -6
            cols = rng.integers(0, 32, nb)
            blocks[np.arange(nb), cols] = rng.choice([-1.0, 1.0], nb) * np.ldexp(1.0, rng.integers(4, 13, nb))
        else:
            blocks[0::2] *= 2.0 ** 8
            blocks[1::2] *= 2.0 ** -8
    return synth.bf16_bits_rne(x.astype(np.float32))


def _e4m3_round(v):
    """Nearest E4M3 value (ties to even mantissa), from the format's spacing; no saturation needed here."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.where(a >= 2.0 ** -6, np.ldexp(1.0, (np.maximum(e, -6) - 3).astype(np.int64)), 2.0 ** -9)
    return np.sign(v) * np.round(a / step) * step


def two_term_e4m3_residual(x_bits):
    """What two E4M3 terms with one power-of-two scale per 32-element block (the largest magnitude of the
    block's residual below 2^8 after scaling) leave of each bf16 value: zero where the split is exact."""
    r = ((x_bits.astype(np.uint32) << 16).view(np.float32)).astype(np.float64).reshape(-1, 32)
    for _ in range(2):
        amax = np.abs(r).max(axis=1, keepdims=True)
        X = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 7, -127)
        r = r - _e4m3_round(r / 2.0 ** X) * 2.0 ** X
    return r.reshape(x_bits.shape)


# ---------------------------------------------------------------- oracle work spread over host processes


def oracle_ffn_mxfp8_task(args):
    """One expert's prefill FFN for one token in a worker process (the record regenerated from its seed)."""
    import oracle
    from expert_offload_moe_gb300 import synth

    seed, layer, E, H, I, e, x_row = args
    rec = synth.expert_records(seed, layer, E, H, I, experts=[e])[0]
    return oracle.expert_ffn_mxfp8(rec, H, I, x_row)


def spawn_pool(n=None):
    """A process pool started with spawn (safe after the parent has used the GPU)."""
    import multiprocessing as mp
    import os

    return mp.get_context("spawn").Pool(n or min(16, os.cpu_count() or 1))
