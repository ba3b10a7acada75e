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


def compare_routing(g, o, logits, k, e2s):
    """Routing indices, compaction and miss lists: bit-exact except near-tie tokens.

    Returns the set of excluded tokens (near ties whose selection differs)."""
    M = o["ids"].shape[0]
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
            assert abs(gw[e] - ow[e]) <= W_ATOL + W_RTOL * abs(ow[e]), (t, e, gw[e], ow[e])

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
    assert np.allclose(g["hot_w"][kg], o["hot_w"][ko], rtol=W_RTOL, atol=W_ATOL)
    kg, ko = keep(g["cold_token"]), keep(o["cold_token"])
    assert np.array_equal(g["cold_token"][kg], o["cold_token"][ko])
    assert np.array_equal(g["cold_expert"][kg], o["cold_expert"][ko])
    assert np.allclose(g["cold_w"][kg], o["cold_w"][ko], rtol=W_RTOL, atol=W_ATOL)
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
