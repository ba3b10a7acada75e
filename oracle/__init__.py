"""CPU oracle for the decode-time MoE layer with GPU expert slots.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` load it; the product path never does.

``build()`` compiles ``oracle.c`` with gcc into ``liboracle.so`` beside it
(plain C, ``-O2 -ffp-contract=off``, no fast-math) and the wrappers below pass
numpy arrays to it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        _declare(_lib)
    return _lib


P = ctypes.c_void_p
I32 = ctypes.c_int
F32 = ctypes.c_float


def _declare(L):
    L.oracle_e2m1.argtypes, L.oracle_e2m1.restype = [ctypes.c_uint8], F32
    L.oracle_e8m0.argtypes, L.oracle_e8m0.restype = [ctypes.c_uint8], F32
    L.oracle_e4m3.argtypes, L.oracle_e4m3.restype = [ctypes.c_uint8], F32
    L.oracle_e4m3_encode.argtypes, L.oracle_e4m3_encode.restype = [F32], ctypes.c_uint8
    L.oracle_f32_to_bf16.argtypes, L.oracle_f32_to_bf16.restype = [F32], ctypes.c_uint16
    L.oracle_mxfp4_dequant.argtypes = [P, P, I32, I32, P]
    L.oracle_mxfp4_dequant.restype = None
    L.oracle_nvfp4_dequant.argtypes = [P, P, I32, I32, P]
    L.oracle_nvfp4_dequant.restype = None
    L.oracle_expert_bytes_fmt.argtypes, L.oracle_expert_bytes_fmt.restype = [I32, I32, I32], ctypes.c_size_t
    L.oracle_expert_ffn_fmt.argtypes = [P, I32, I32, I32, P, P]
    L.oracle_expert_ffn_fmt.restype = None
    L.oracle_moe_layer_fmt.argtypes = [P, I32, I32, I32, I32, I32, I32, P, P, P, P, P, P] + [P] * 16
    L.oracle_moe_layer_fmt.restype = None
    L.oracle_router_logits.argtypes = [P, I32, I32, P, P, I32, P]
    L.oracle_router_logits.restype = None
    L.oracle_topk_softmax.argtypes = [P, I32, I32, I32, P, P]
    L.oracle_topk_softmax.restype = None
    L.oracle_compact.argtypes = [P, P, I32, I32, P, I32] + [P] * 13
    L.oracle_compact.restype = None
    L.oracle_expert_gate_up.argtypes = [P, I32, I32, P, P]
    L.oracle_expert_gate_up.restype = None
    L.oracle_expert_down.argtypes = [P, I32, I32, P, P]
    L.oracle_expert_down.restype = None
    L.oracle_expert_ffn.argtypes = [P, I32, I32, P, P]
    L.oracle_expert_ffn.restype = None
    L.oracle_expert_ffn_mxfp8.argtypes = [P, I32, I32, P, P]
    L.oracle_expert_ffn_mxfp8.restype = None
    L.oracle_moe_layer.argtypes = [P, I32, I32, I32, I32, I32, P, P, P, P, P, P] + [P] * 16
    L.oracle_moe_layer.restype = None
    L.oracle_cache_step.argtypes = [P, P, P, P, I32, I32, P, ctypes.c_int64, ctypes.c_double, I32, P, P, P, P]
    L.oracle_cache_step.restype = I32
    L.oracle_cache_step_recency.argtypes = [I32, P, P, P, P, P, I32, I32, P, ctypes.c_int64, ctypes.c_double, I32,
                                            P, P, P, P]
    L.oracle_cache_step_recency.restype = I32
    L.oracle_cache_step_slru.argtypes = [P, P, P, P, P, I32, I32, P, ctypes.c_int64, ctypes.c_double, I32, I32, P,
                                         P, P, P]
    L.oracle_cache_step_slru.restype = I32
    L.oracle_demand_lru_step.argtypes = [P, P, P, I32, I32, P, ctypes.c_int64, P, P]
    L.oracle_demand_lru_step.restype = I32
    L.oracle_prefetch_step.argtypes = [P, P, P, P, I32, I32, P, I32, P, P, P, P]
    L.oracle_prefetch_step.restype = I32
    L.oracle_mxfp8_block.argtypes = [P, I32, P]
    L.oracle_mxfp8_block.restype = ctypes.c_uint8


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e8m0(e: int) -> float:
    return lib().oracle_e8m0(e)


def e4m3(code: int) -> float:
    return lib().oracle_e4m3(code)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(v)


def f32_to_bf16(v: float) -> int:
    return lib().oracle_f32_to_bf16(v)


def mxfp4_dequant(codes, scales, R, C):
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    W = np.empty((R, C), dtype=np.float32)
    lib().oracle_mxfp4_dequant(_p(codes), _p(scales), R, C, _p(W))
    return W


def nvfp4_dequant(codes, scales, R, C):
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    W = np.empty((R, C), dtype=np.float32)
    lib().oracle_nvfp4_dequant(_p(codes), _p(scales), R, C, _p(W))
    return W


FORMATS = {"mxfp4": 0, "nvfp4": 1}


def expert_bytes(H, I, fmt="mxfp4"):
    return int(lib().oracle_expert_bytes_fmt(H, I, FORMATS[fmt]))


def router_logits(x_bf16, Wr, bias=None):
    x = _c(x_bf16, np.uint16)
    Wr = _c(Wr, np.float32)
    M, H = x.shape
    E = Wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((M, E), dtype=np.float32)
    lib().oracle_router_logits(_p(x), M, H, _p(Wr), _p(b), E, _p(out))
    return out


def topk_softmax(logits, k):
    logits = _c(logits, np.float32)
    M, E = logits.shape
    ids = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float32)
    lib().oracle_topk_softmax(_p(logits), M, E, k, _p(ids), _p(w))
    return ids, w


def compact(ids, w, e2s):
    ids, w, e2s = _c(ids, np.int32), _c(w, np.float32), _c(e2s, np.int32)
    M, k = ids.shape
    E = e2s.shape[0]
    n = M * k
    r = {name: np.zeros(n, dtype=np.int32) for name in
         ("hot_expert", "hot_slot", "hot_token", "act_expert", "act_slot", "act_off", "act_cnt",
          "cold_token", "cold_expert")}
    r["hot_w"] = np.zeros(n, dtype=np.float32)
    r["cold_w"] = np.zeros(n, dtype=np.float32)
    r["hist"] = np.zeros(E, dtype=np.int32)
    counts = np.zeros(3, dtype=np.int32)
    lib().oracle_compact(_p(ids), _p(w), M, k, _p(e2s), E, _p(r["hot_expert"]), _p(r["hot_slot"]),
                         _p(r["hot_token"]), _p(r["hot_w"]), _p(r["act_expert"]), _p(r["act_slot"]),
                         _p(r["act_off"]), _p(r["act_cnt"]), _p(r["cold_token"]), _p(r["cold_expert"]),
                         _p(r["cold_w"]), _p(r["hist"]), _p(counts))
    return _trim(r, counts)


def _trim(r, counts):
    n_hot, n_cold, n_act = (int(c) for c in counts)
    out = {"n_hot": n_hot, "n_cold": n_cold, "n_active": n_act, "hist": r["hist"]}
    for name in ("hot_expert", "hot_slot", "hot_token", "hot_w"):
        out[name] = r[name][:n_hot].copy()
    for name in ("act_expert", "act_slot", "act_off", "act_cnt"):
        out[name] = r[name][:n_act].copy()
    for name in ("cold_token", "cold_expert", "cold_w"):
        out[name] = r[name][:n_cold].copy()
    return out


def expert_gate_up(rec, H, I, x_row):
    rec, x = _c(rec, np.uint8), _c(x_row, np.uint16)
    h = np.empty(I, dtype=np.float32)
    lib().oracle_expert_gate_up(_p(rec), H, I, _p(x), _p(h))
    return h


def expert_down(rec, H, I, h):
    rec, h = _c(rec, np.uint8), _c(h, np.float32)
    y = np.empty(H, dtype=np.float32)
    lib().oracle_expert_down(_p(rec), H, I, _p(h), _p(y))
    return y


def expert_ffn(rec, H, I, x_row, fmt="mxfp4"):
    rec, x = _c(rec, np.uint8), _c(x_row, np.uint16)
    y = np.empty(H, dtype=np.float32)
    lib().oracle_expert_ffn_fmt(_p(rec), H, I, FORMATS[fmt], _p(x), _p(y))
    return y


def expert_ffn_mxfp8(rec, H, I, x_row):
    rec, x = _c(rec, np.uint8), _c(x_row, np.uint16)
    y = np.empty(H, dtype=np.float32)
    lib().oracle_expert_ffn_mxfp8(_p(rec), H, I, _p(x), _p(y))
    return y


def moe_layer(x_bf16, Wr, bias, experts, e2s, k, H, I, fmt="mxfp4"):
    """Whole layer.  ``experts``: [E, expert_bytes] uint8 indexed by expert id; ``fmt``: "mxfp4" / "nvfp4"."""
    x = _c(x_bf16, np.uint16)
    Wr = _c(Wr, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    experts = _c(experts, np.uint8)
    e2s = _c(e2s, np.int32)
    M = x.shape[0]
    E = Wr.shape[0]
    n = M * k
    out_f32 = np.empty((M, H), dtype=np.float32)
    out_bf16 = np.empty((M, H), dtype=np.uint16)
    ids = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float32)
    logits = np.empty((M, E), dtype=np.float32)
    r = {name: np.zeros(n, dtype=np.int32) for name in
         ("hot_expert", "hot_slot", "hot_token", "act_expert", "act_slot", "act_off", "act_cnt",
          "cold_token", "cold_expert")}
    r["hot_w"] = np.zeros(n, dtype=np.float32)
    r["cold_w"] = np.zeros(n, dtype=np.float32)
    r["hist"] = np.zeros(E, dtype=np.int32)
    counts = np.zeros(3, dtype=np.int32)
    lib().oracle_moe_layer_fmt(_p(x), M, H, I, E, k, FORMATS[fmt], _p(Wr), _p(b), _p(experts), _p(e2s), _p(out_f32),
                           _p(out_bf16), _p(ids), _p(w), _p(r["hot_expert"]), _p(r["hot_slot"]),
                           _p(r["hot_token"]), _p(r["hot_w"]), _p(r["act_expert"]), _p(r["act_slot"]),
                           _p(r["act_off"]), _p(r["act_cnt"]), _p(r["cold_token"]), _p(r["cold_expert"]),
                           _p(r["cold_w"]), _p(r["hist"]), _p(counts), _p(logits))
    out = _trim(r, counts)
    out.update(out_f32=out_f32, out_bf16=out_bf16, ids=ids, w=w, logits=logits)
    return out


POLICIES = {"freq": 0, "lru": 1, "fifo": 2, "slru": 3}


def slru_protected_cap(S):
    """Protected segment of the SLRU reading: four fifths of the slots (rounded down)."""
    return (4 * S) // 5


class CacheReplay:
    """Step-by-step replay of the slot cache policy for one layer.  policy: "freq" (decayed frequency:
    LFU / LFRU), "lru", "fifo" or "slru" (segmented LRU; ``pcap`` protected slots, default four fifths)."""

    def __init__(self, e2s, S, decay=1.0, R=2, policy="freq", pcap=None):
        self.e2s = _c(e2s, np.int32).copy()
        self.E = self.e2s.shape[0]
        self.S = S
        self.s2e = np.full(S, -1, dtype=np.int32)
        for e, s in enumerate(self.e2s):
            if s >= 0:
                self.s2e[s] = e
        self.score = np.zeros(self.E, dtype=np.float64)
        self.last = np.full(self.E, -1, dtype=np.int64)
        self.decay = float(decay)
        self.R = int(R)
        self.policy = POLICIES[policy]
        self.loaded = np.full(self.E, -1, dtype=np.int64)
        self.seg = np.zeros(self.E, dtype=np.uint8)  # SLRU: 1 = protected segment
        self.pcap = slru_protected_cap(S) if pcap is None else int(pcap)

    def step(self, hist, step, in_flight=None):
        hist = _c(hist, np.int32)
        pe = np.zeros(max(self.R, 1), dtype=np.int32)
        ps = np.zeros_like(pe)
        pv = np.zeros_like(pe)
        fl = None if in_flight is None else _c(in_flight, np.uint8)
        if self.policy == 0:
            n = lib().oracle_cache_step(_p(self.score), _p(self.last), _p(self.e2s), _p(self.s2e), self.E,
                                        self.S, _p(hist), int(step), self.decay, self.R, _p(fl), _p(pe),
                                        _p(ps), _p(pv))
        elif self.policy == 3:
            n = lib().oracle_cache_step_slru(_p(self.score), _p(self.last), _p(self.seg), _p(self.e2s),
                                             _p(self.s2e), self.E, self.S, _p(hist), int(step), self.decay, self.R,
                                             self.pcap, _p(fl), _p(pe), _p(ps), _p(pv))
        else:
            n = lib().oracle_cache_step_recency(self.policy, _p(self.score), _p(self.last), _p(self.loaded),
                                                _p(self.e2s), _p(self.s2e), self.E, self.S, _p(hist), int(step),
                                                self.decay, self.R, _p(fl), _p(pe), _p(ps), _p(pv))
        return [(int(pe[i]), int(ps[i]), int(pv[i])) for i in range(n)]


class DemandLRUReplay:
    """Step-by-step replay of the demand-filled LRU slot table (xinfer docs "How it works", Decode): every
    routed expert without a slot is given the least-recently-used slot that this step did not route, in
    the same step.  ``step(hist)`` returns the fills as (expert, slot) pairs; the step clock starts at 0."""

    def __init__(self, e2s, S):
        self.e2s = _c(e2s, np.int32).copy()
        self.E = self.e2s.shape[0]
        self.S = S
        self.s2e = np.full(S, -1, dtype=np.int32)
        for e, s in enumerate(self.e2s):
            if s >= 0:
                self.s2e[s] = e
        self.stamp = np.full(S, -1, dtype=np.int64)
        self.clock = 0

    def step(self, hist):
        hist = _c(hist, np.int32)
        fe = np.zeros(max(self.S, 1), dtype=np.int32)
        fs = np.zeros_like(fe)
        n = lib().oracle_demand_lru_step(_p(self.e2s), _p(self.s2e), _p(self.stamp), self.E, self.S, _p(hist),
                                         self.clock, _p(fe), _p(fs))
        self.clock += 1
        return [(int(fe[i]), int(fs[i])) for i in range(n)]


def mxfp8_block(v):
    v = _c(v, np.float32)
    codes = np.empty(v.shape[0], dtype=np.uint8)
    sc = lib().oracle_mxfp8_block(_p(v), v.shape[0], _p(codes))
    return int(sc), codes


def prefetch_step(score, last, e2s, S, pred, R, in_flight=None):
    """One next-layer prefetch decision (see oracle_prefetch_step).  Returns (pairs, new e2s); the inputs
    are not modified."""
    score, last = _c(score, np.float64), _c(last, np.int64)
    e2s = _c(e2s, np.int32).copy()
    E = e2s.shape[0]
    s2e = np.full(S, -1, dtype=np.int32)
    for e, s in enumerate(e2s):
        if s >= 0:
            s2e[s] = e
    pred = _c(pred, np.int32)
    fl = None if in_flight is None else _c(in_flight, np.uint8)
    pe = np.zeros(max(R, 1), dtype=np.int32)
    ps, pv = np.zeros_like(pe), np.zeros_like(pe)
    n = lib().oracle_prefetch_step(_p(score), _p(last), _p(e2s), _p(s2e), E, S, _p(pred), int(R), _p(fl), _p(pe),
                                   _p(ps), _p(pv))
    return [(int(pe[i]), int(ps[i]), int(pv[i])) for i in range(n)], e2s
