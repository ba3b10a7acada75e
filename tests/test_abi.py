"""The C-ABI library builds, loads without a GPU, exports every declared
symbol, and its host-side slot-cache policy agrees with the oracle's."""
import os
import re

import numpy as np
import pytest

from expert_offload_moe_gb300 import build as moe_build
from expert_offload_moe_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def declared_symbols():
    text = ""
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            text += open(os.path.join(ROOT, "include", f)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_calls():
    syms = declared_symbols()
    for name in ("moe_layer_create", "moe_route", "moe_forward_slots", "moe_cache_update", "moe_destroy"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing
    assert set(declared_symbols()) <= set(moe.EXPORTED)


def test_null_arguments_are_rejected_without_a_gpu(lib):
    assert lib.moe_layer_create(None, None, None, None, None, None, None) == moe.MOE_EINVAL
    assert lib.moe_route(None, None, 1, None, None) == moe.MOE_EINVAL
    assert lib.moe_forward_slots(None, None, None, 1, None) == moe.MOE_EINVAL
    assert lib.moe_cache_update(None, None, None) == moe.MOE_EINVAL
    assert lib.moe_prefetch(None, None, 1, None, None) == moe.MOE_EINVAL
    assert lib.moe_debug_decode_fusion(None, 1) == moe.MOE_EINVAL
    assert lib.moe_debug_stream_read(None, 16, None, 0, None) == moe.MOE_EINVAL
    assert lib.moe_debug_mma_peak(8, 0, None, None) == moe.MOE_EINVAL
    assert lib.moe_destroy(None) == moe.MOE_OK


def _random_trace(rng, E, k, steps, drift=False):
    for st in range(steps):
        p = np.exp(-0.15 * ((np.arange(E) + (st // 7 if drift else 0)) % E))
        p /= p.sum()
        hist = np.zeros(E, dtype=np.int32)
        for _ in range(rng.integers(1, 4)):
            for e in rng.choice(E, k, replace=False, p=p):
                hist[e] += 1
        yield st, hist


@pytest.mark.parametrize("decay,R,E,S", [(1.0, 2, 32, 16), (0.5, 2, 32, 16), (0.9, 1, 16, 4), (1.0, 4, 64, 48)])
def test_library_policy_matches_oracle_replay(lib, oracle_lib, decay, R, E, S):
    rng = np.random.default_rng(int(decay * 10) + R)
    e2s0 = np.full(E, -1, dtype=np.int32)
    e2s0[rng.choice(E, S, replace=False)] = rng.permutation(S)
    rp = oracle_lib.CacheReplay(e2s0, S, decay=decay, R=R)
    score = np.zeros(E, dtype=np.float64)
    last = np.full(E, -1, dtype=np.int64)
    e2s = e2s0.copy()
    s2e = np.full(S, -1, dtype=np.int32)
    s2e[e2s[e2s >= 0]] = np.nonzero(e2s >= 0)[0]
    n_pairs = 0
    for st, hist in _random_trace(rng, E, 4, 300, drift=True):
        a = moe.policy_step(score, last, e2s, s2e, hist, st, decay, R)
        b = rp.step(hist, st)
        assert a == b, st
        assert np.array_equal(e2s, rp.e2s) and np.array_equal(s2e, rp.s2e)
        n_pairs += len(a)
    assert n_pairs > 0


def test_library_policy_with_in_flight_matches_oracle(lib, oracle_lib):
    rng = np.random.default_rng(5)
    E, S, R = 24, 8, 2
    e2s0 = np.where(np.arange(E) < S, np.arange(E), -1).astype(np.int32)
    rp = oracle_lib.CacheReplay(e2s0, S, R=R)
    score, last = np.zeros(E), np.full(E, -1, dtype=np.int64)
    e2s, s2e = e2s0.copy(), np.arange(S, dtype=np.int32)
    for st, hist in _random_trace(rng, E, 3, 100, drift=True):
        fl = (rng.random(E) < 0.2).astype(np.uint8)
        assert moe.policy_step(score, last, e2s, s2e, hist, st, 1.0, R, in_flight=fl) == rp.step(hist, st, fl)
        assert np.array_equal(e2s, rp.e2s)


def test_library_policy_golden_trace(lib):
    lines = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "cache_lfu_trace.txt"))
             if l.strip() and l[0] != "#"]
    E, S, R = int(lines[0][1]), int(lines[0][3]), int(lines[0][5])
    e2s = np.array([int(v) for v in lines[1][1:]], dtype=np.int32)
    s2e = np.full(S, -1, dtype=np.int32)
    s2e[e2s[e2s >= 0]] = np.nonzero(e2s >= 0)[0]
    score, last = np.zeros(E), np.full(E, -1, dtype=np.int64)
    for l in lines[2:]:
        st = int(l[1])
        i_p, i_m = l.index("pairs"), l.index("map")
        hist = np.array([int(v) for v in l[3:i_p]], dtype=np.int32)
        want = [tuple(int(q) for q in p.split(":")) for p in l[i_p + 1:i_m]]
        assert moe.policy_step(score, last, e2s, s2e, hist, st, 1.0, R) == want
        assert list(e2s) == [int(v) for v in l[i_m + 1:]]


def test_policy_rejects_bad_arguments(lib):
    with pytest.raises(moe.MoeError):
        moe.policy_step(np.zeros(4), np.zeros(4, dtype=np.int64), np.zeros(4, dtype=np.int32),
                        np.zeros(8, dtype=np.int32), np.zeros(4, dtype=np.int32), 0, 1.0, 1)


@pytest.mark.parametrize("policy,R,E,S", [("lru", 2, 32, 16), ("fifo", 2, 32, 16), ("lru", 1, 16, 4),
                                          ("fifo", 4, 64, 48)])
def test_library_recency_policies_match_oracle_replay(lib, oracle_lib, policy, R, E, S):
    rng = np.random.default_rng(len(policy) * 7 + R)
    e2s0 = np.full(E, -1, dtype=np.int32)
    e2s0[rng.choice(E, S, replace=False)] = rng.permutation(S)
    rp = oracle_lib.CacheReplay(e2s0, S, R=R, policy=policy)
    code = {"lru": moe.MOE_POLICY_LRU, "fifo": moe.MOE_POLICY_FIFO}[policy]
    score, last, loaded = np.zeros(E), np.full(E, -1, dtype=np.int64), np.full(E, -1, dtype=np.int64)
    e2s = e2s0.copy()
    s2e = np.full(S, -1, dtype=np.int32)
    s2e[e2s[e2s >= 0]] = np.nonzero(e2s >= 0)[0]
    n_pairs = 0
    for st, hist in _random_trace(rng, E, 4, 300, drift=True):
        fl = (rng.random(E) < 0.1).astype(np.uint8)
        a = moe.policy_step_recency(code, score, last, loaded, e2s, s2e, hist, st, 1.0, R, in_flight=fl)
        b = rp.step(hist, st, fl)
        assert a == b, st
        assert np.array_equal(e2s, rp.e2s) and np.array_equal(s2e, rp.s2e)
        n_pairs += len(a)
    assert n_pairs > 0


@pytest.mark.parametrize("name,code", [("cache_lru_trace.txt", 1), ("cache_fifo_trace.txt", 2)])
def test_library_recency_golden_traces(lib, name, code):
    lines = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", name)) if l.strip() and l[0] != "#"]
    E, S, R = int(lines[0][1]), int(lines[0][3]), int(lines[0][5])
    e2s = np.array([int(v) for v in lines[1][1:]], dtype=np.int32)
    s2e = np.full(S, -1, dtype=np.int32)
    s2e[e2s[e2s >= 0]] = np.nonzero(e2s >= 0)[0]
    score, last, loaded = np.zeros(E), np.full(E, -1, dtype=np.int64), np.full(E, -1, dtype=np.int64)
    for l in lines[2:]:
        st = int(l[1])
        i_p, i_m = l.index("pairs"), l.index("map")
        hist = np.array([int(v) for v in l[3:i_p]], dtype=np.int32)
        want = [tuple(int(q) for q in p.split(":")) for p in l[i_p + 1:i_m]]
        assert moe.policy_step_recency(code, score, last, loaded, e2s, s2e, hist, st, 1.0, R) == want, st
        assert list(e2s) == [int(v) for v in l[i_m + 1:]]


def test_recency_policy_rejects_bad_arguments(lib):
    E, S = 4, 2
    with pytest.raises(moe.MoeError):  # FIFO needs loaded[]
        moe.policy_step_recency(moe.MOE_POLICY_FIFO, np.zeros(E), np.zeros(E, dtype=np.int64), None,
                                np.array([0, 1, -1, -1], dtype=np.int32), np.array([0, 1], dtype=np.int32),
                                np.zeros(E, dtype=np.int32), 0, 1.0, 1)
    with pytest.raises(moe.MoeError):  # not a recency policy
        moe.policy_step_recency(moe.MOE_POLICY_FREQ, np.zeros(E), np.zeros(E, dtype=np.int64),
                                np.zeros(E, dtype=np.int64), np.array([0, 1, -1, -1], dtype=np.int32),
                                np.array([0, 1], dtype=np.int32), np.zeros(E, dtype=np.int32), 0, 1.0, 1)


@pytest.mark.parametrize("R,E,S,pcap", [(2, 32, 16, None), (1, 16, 4, None), (4, 64, 48, None), (2, 32, 16, 0),
                                         (2, 32, 16, 16), (3, 12, 5, 2)])
def test_library_slru_matches_oracle_replay(lib, oracle_lib, R, E, S, pcap):
    rng = np.random.default_rng(R * 31 + E + S)
    e2s0 = np.full(E, -1, dtype=np.int32)
    e2s0[rng.choice(E, S, replace=False)] = rng.permutation(S)
    rp = oracle_lib.CacheReplay(e2s0, S, R=R, policy="slru", pcap=pcap)
    score, last = np.zeros(E), np.full(E, -1, dtype=np.int64)
    seg = np.zeros(E, dtype=np.uint8)
    e2s = e2s0.copy()
    s2e = np.full(S, -1, dtype=np.int32)
    s2e[e2s[e2s >= 0]] = np.nonzero(e2s >= 0)[0]
    n_pairs = 0
    for st, hist in _random_trace(rng, E, 4, 300, drift=True):
        fl = (rng.random(E) < 0.1).astype(np.uint8)
        a = moe.policy_step_slru(score, last, seg, e2s, s2e, hist, st, 1.0, R, rp.pcap, in_flight=fl)
        b = rp.step(hist, st, fl)
        assert a == b, st
        assert np.array_equal(e2s, rp.e2s) and np.array_equal(s2e, rp.s2e) and np.array_equal(seg, rp.seg)
        n_pairs += len(a)
    assert n_pairs > 0


def test_library_slru_golden_trace(lib):
    lines = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "cache_slru_trace.txt"))
             if l.strip() and l[0] != "#"]
    E, S, R = int(lines[0][1]), int(lines[0][3]), int(lines[0][5])
    e2s = np.array([int(v) for v in lines[1][1:]], dtype=np.int32)
    s2e = np.full(S, -1, dtype=np.int32)
    s2e[e2s[e2s >= 0]] = np.nonzero(e2s >= 0)[0]
    score, last, seg = np.zeros(E), np.full(E, -1, dtype=np.int64), np.zeros(E, dtype=np.uint8)
    for l in lines[2:]:
        st = int(l[1])
        i_p, i_m = l.index("pairs"), l.index("map")
        hist = np.array([int(v) for v in l[3:i_p]], dtype=np.int32)
        want = [tuple(int(q) for q in p.split(":")) for p in l[i_p + 1:i_m]]
        assert moe.policy_step_slru(score, last, seg, e2s, s2e, hist, st, 1.0, R, (4 * S) // 5) == want, st
        assert list(e2s) == [int(v) for v in l[i_m + 1:]]


def test_slru_rejects_bad_arguments(lib):
    E, S = 4, 2
    args = (np.zeros(E), np.zeros(E, dtype=np.int64), np.zeros(E, dtype=np.uint8),
            np.array([0, 1, -1, -1], dtype=np.int32), np.array([0, 1], dtype=np.int32), np.zeros(E, dtype=np.int32),
            0, 1.0, 1)
    for pcap in (-1, S + 1):
        with pytest.raises(moe.MoeError):
            moe.policy_step_slru(*args, pcap)
    assert lib.moe_layer_set_policy(None, moe.MOE_POLICY_SLRU) == moe.MOE_EINVAL


@pytest.mark.parametrize("R,E,S", [(2, 32, 16), (1, 16, 4), (4, 64, 48), (3, 8, 8)])
def test_library_prefetch_step_matches_oracle(lib, oracle_lib, R, E, S):
    rng = np.random.default_rng(R * 100 + E)
    for _ in range(200):
        e2s = np.full(E, -1, dtype=np.int32)
        e2s[rng.choice(E, S, replace=False)] = rng.permutation(S)
        s2e = np.full(S, -1, dtype=np.int32)
        s2e[e2s[e2s >= 0]] = np.nonzero(e2s >= 0)[0]
        score = rng.integers(0, 4, E).astype(np.float64)
        last = rng.integers(-1, 5, E).astype(np.int64)
        pred = np.where(rng.random(E) < 0.25, rng.integers(1, 4, E), 0).astype(np.int32)
        fl = (rng.random(E) < 0.1).astype(np.uint8)
        want, want_map = oracle_lib.prefetch_step(score, last, e2s, S, pred, R, in_flight=fl)
        got = moe.prefetch_step(score, last, e2s, s2e, pred, R, in_flight=fl)
        assert got == want and np.array_equal(e2s, want_map)
        assert all(s2e[e2s[e]] == e for e in range(E) if e2s[e] >= 0)


def test_prefetch_step_rejects_bad_arguments(lib):
    E, S = 4, 2
    e2s = np.array([0, 1, -1, -1], dtype=np.int32)
    s2e = np.array([0, 1], dtype=np.int32)
    with pytest.raises(moe.MoeError):  # R < 0
        moe.prefetch_step(np.zeros(E), np.zeros(E, dtype=np.int64), e2s, s2e, np.ones(E, dtype=np.int32), -1)
    with pytest.raises(moe.MoeError):  # more slots than experts
        moe.prefetch_step(np.zeros(E), np.zeros(E, dtype=np.int64), e2s, np.zeros(8, dtype=np.int32),
                          np.ones(E, dtype=np.int32), 1)
    assert moe.prefetch_step(np.zeros(E), np.zeros(E, dtype=np.int64), e2s, s2e, np.zeros(E, dtype=np.int32), 2) == []
