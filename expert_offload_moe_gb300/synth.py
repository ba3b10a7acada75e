"""Seeded synthetic inputs for the decode-time MoE layer with GPU expert slots.

This module only draws random numbers and lays bytes out in the documented
expert record format; it holds none of the layer's arithmetic (no decoding,
no routing, no products).  Both the CPU oracle (under ``oracle/``) and the
CUDA path take their inputs from here, and nothing else is shared between
them.

The pages measure real models (gpt-oss-20B, an E=512/k=10 Qwen3-Next-style
model) on real prompts; none of that is available, so every tensor below is a
seeded stand-in with the pages' shapes:

* activations  ``x``      bf16 bits, RNE of N(0, 1)
* router       ``Wr``     fp32 N(0, 0.02), ``[E, H]``
* router bias  ``b``      ``tau * log(p_rank(e))`` with Zipf(s=1) popularity
                          ``p_r = (1/r) / sum_j (1/j)`` over a seeded rank
                          permutation (0 when ``tau == 0``)
* experts      MXFP4      every E2M1 nibble uniform over its 16 codes, every
                          E8M0 scale byte uniform over {120, ..., 127}

Expert record layout (``expert_bytes = 3 * I * H * 17 / 32``), one record per
expert, the same bytes in the pinned host bank and in a GPU slot::

    [Wg codes  I x H/2][Wg scales I x H/32]
    [Wu codes  I x H/2][Wu scales I x H/32]
    [Wd codes  H x I/2][Wd scales H x I/32]

Codes are row-major; byte ``c`` of a row holds column ``2c`` in its low nibble
and column ``2c+1`` in its high nibble.  Scale byte ``b`` of a row covers
columns ``[32b, 32b+32)``.

NVFP4 records (``weight_format=1``) have the same codes and one E4M3 scale byte
per 16 columns (``expert_bytes = 3 * I * H * 9 / 16``); scale bytes are
positive normal E4M3 values with exponent field uniform over {1, ..., 7} and
mantissa uniform, i.e. between 2^-6 and 1.875, a range like the MXFP4 scales'.

Seeds follow ``SeedSequence([seed, layer, tensor_id, step])``.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# tensor ids inside a SeedSequence key
T_X, T_ROUTER, T_RANK, T_EXPERTS, T_RANK_B, T_X_RESID = 1, 2, 3, 4, 5, 6


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one synthetic workload (a stack of independent MoE layers)."""

    name: str
    layers: int
    hidden: int
    inter: int
    experts: int
    top_k: int
    slots: int
    tokens: tuple  # decode batch sizes M exercised
    steps: int
    bias_tau: float = 0.0
    prefill_tokens: int = 0
    drift: bool = False  # bias drifts between two popularity orders over the steps
    weight_format: int = 0  # 0 = MXFP4, 1 = NVFP4

    @property
    def expert_bytes(self) -> int:
        return expert_bytes(self.hidden, self.inter, self.weight_format)


WORKLOADS = {
    w.name: w
    for w in [
        # tiny single layer: every expert resident, one token
        Workload("tiny_h256_i128_e16k2", 1, 256, 128, 16, 2, 16, (1,), 4),
        # gpt-oss-20B-shaped stack, every expert resident, M=1 decode
        Workload("gptoss20b_h2880_e32k4_resident_m1", 24, 2880, 2880, 32, 4, 32, (1,), 512),
        # E=512 / k=10 stack, half the experts in slots, popularity-skewed routing
        Workload("e512k10_h2048_i512_s256_m1", 48, 2048, 512, 512, 10, 256, (1,), 64, bias_tau=0.25),
        # same shape, 3/4 of the experts in slots, speculative-verify batches
        Workload("e512k10_h2048_i512_s384_m4m8", 48, 2048, 512, 512, 10, 384, (4, 8), 64, bias_tau=0.25),
        # gpt-oss shape: 2048-token prefill, then decode with 16 of 32 slots and LFU refill
        Workload("gptoss20b_prefill2048_s16_lfu_drift", 24, 2880, 2880, 32, 4, 16, (1,), 256,
                 bias_tau=0.25, prefill_tokens=2048, drift=True),
        # the gpt-oss decode stack with NVFP4 experts (16-element E4M3 scales)
        Workload("gptoss20b_h2880_e32k4_resident_m1_nvfp4", 24, 2880, 2880, 32, 4, 32, (1,), 512, weight_format=1),
    ]
}


def scale_block(weight_format: int = 0) -> int:
    return 16 if weight_format == 1 else 32


def expert_bytes(hidden: int, inter: int, weight_format: int = 0) -> int:
    return 3 * inter * hidden // 2 + 3 * inter * hidden // scale_block(weight_format)


def section_offsets(hidden: int, inter: int, weight_format: int = 0) -> dict:
    """Byte offsets of the six sections of one expert record."""
    gc = inter * hidden // 2
    gs = inter * hidden // scale_block(weight_format)
    off = {}
    o = 0
    for name, size in (("wg_codes", gc), ("wg_scales", gs), ("wu_codes", gc), ("wu_scales", gs),
                       ("wd_codes", gc), ("wd_scales", gs)):
        off[name] = (o, size)
        o += size
    return off


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def _bits(*key) -> np.random.PCG64:
    return np.random.PCG64(np.random.SeedSequence([int(k) for k in key]))


def bf16_bits_rne(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (input generation only)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def activations(seed: int, layer: int, step: int, M: int, H: int) -> np.ndarray:
    """bf16 bit patterns [M, H] of RNE(N(0,1))."""
    g = _rng(seed, layer, T_X, step).standard_normal((M, H), dtype=np.float32)
    return bf16_bits_rne(g)


def activations_residual(seed: int, step: int, L: int, M: int, H: int, rho: float) -> np.ndarray:
    """[L, M, H] bf16 bits whose layers are correlated like a residual stream:
    x_0 ~ N(0, 1), x_l = rho x_(l-1) + sqrt(1 - rho^2) e_l with fresh e_l ~ N(0, 1) (float64, then RNE)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0, T_X_RESID, step]))
    x = rng.standard_normal((M, H))
    out = np.empty((L, M, H), dtype=np.uint16)
    for l in range(L):
        if l:
            x = rho * x + np.sqrt(1.0 - rho * rho) * rng.standard_normal((M, H))
        out[l] = bf16_bits_rne(x.astype(np.float32))
    return out


def router_weights(seed: int, layer: int, E: int, H: int) -> np.ndarray:
    return (_rng(seed, layer, T_ROUTER).standard_normal((E, H), dtype=np.float32) * np.float32(0.02)).astype(np.float32)


def popularity_rank(seed: int, layer: int, E: int, order: int = 0) -> np.ndarray:
    """rank[e] in [0, E): a seeded permutation; rank 0 is the most popular expert."""
    tid = T_RANK if order == 0 else T_RANK_B
    perm = _rng(seed, layer, tid).permutation(E)  # perm[r] = expert with rank r
    rank = np.empty(E, dtype=np.int64)
    rank[perm] = np.arange(E)
    return rank


def zipf_log_popularity(E: int) -> np.ndarray:
    """log p_r for Zipf(s=1) over ranks r = 1..E (float64)."""
    r = np.arange(1, E + 1, dtype=np.float64)
    p = (1.0 / r) / np.sum(1.0 / r)
    return np.log(p)


def router_bias(seed: int, layer: int, E: int, tau: float, order: int = 0) -> np.ndarray:
    if tau == 0.0:
        return np.zeros(E, dtype=np.float32)
    lp = zipf_log_popularity(E)
    return (tau * lp[popularity_rank(seed, layer, E, order)]).astype(np.float32)


def drifting_bias(seed: int, layer: int, E: int, tau: float, step: int, steps: int) -> np.ndarray:
    """(1 - a) * b_A + a * b_B with a = step / (steps - 1), orders A and B seeded 0 and 1."""
    a = step / max(steps - 1, 1)
    bA = router_bias(seed, layer, E, tau, 0).astype(np.float64)
    bB = router_bias(seed, layer, E, tau, 1).astype(np.float64)
    return ((1.0 - a) * bA + a * bB).astype(np.float32)


def expert_to_slot_by_rank(seed: int, layer: int, E: int, S: int, order: int = 0) -> np.ndarray:
    """Static placement: expert of popularity rank r < S sits in slot r; others are cold (-1)."""
    if S >= E:
        return np.arange(E, dtype=np.int32)
    rank = popularity_rank(seed, layer, E, order)
    return np.where(rank < S, rank, -1).astype(np.int32)


def fill_expert_records(out: np.ndarray, seed: int, layer: int, H: int, I: int, first: int = 0,
                        weight_format: int = 0) -> None:
    """Fill ``out`` ([n, expert_bytes] uint8) with experts first..first+n-1 of a layer."""
    eb = expert_bytes(H, I, weight_format)
    assert out.ndim == 2 and out.shape[1] == eb and out.dtype == np.uint8
    offs = section_offsets(H, I, weight_format)
    for j in range(out.shape[0]):
        e = first + j
        raw = _bits(seed, layer, T_EXPERTS, e).random_raw((eb + 7) // 8).view(np.uint8)[:eb]
        rec = out[j]
        rec[:] = raw
        for name in ("wg_scales", "wu_scales", "wd_scales"):
            o, n = offs[name]
            if weight_format == 1:  # E4M3: exponent field 1..7, any mantissa, sign 0
                rec[o:o + n] = (((rec[o:o + n] >> 3) % 7 + 1) << 3) | (rec[o:o + n] & 7)
            else:
                rec[o:o + n] = (rec[o:o + n] & 7) + 120


def expert_records(seed: int, layer: int, E: int, H: int, I: int, experts=None, weight_format: int = 0) -> np.ndarray:
    """[n, expert_bytes] uint8 records for the listed experts (default: all E)."""
    ids = list(range(E)) if experts is None else list(experts)
    out = np.empty((len(ids), expert_bytes(H, I, weight_format)), dtype=np.uint8)
    for j, e in enumerate(ids):
        fill_expert_records(out[j:j + 1], seed, layer, H, I, first=e, weight_format=weight_format)
    return out


def zipf_expected_hit_rate(E: int, S: int, tau: float) -> float:
    """Rough prior only (used in docs): mass of the top-S experts under p^tau."""
    lp = zipf_log_popularity(E) * tau
    w = np.exp(lp - lp.max())
    return float(w[:S].sum() / w.sum())


__all__ = [
    "Workload", "WORKLOADS", "scale_block", "expert_bytes", "section_offsets", "bf16_bits_rne", "activations",
    "activations_residual", "router_weights", "popularity_rank", "router_bias", "drifting_bias", "expert_to_slot_by_rank",
    "fill_expert_records", "expert_records", "zipf_log_popularity", "zipf_expected_hit_rate",
]
