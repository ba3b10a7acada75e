"""ctypes binding of ``libmoe.so`` (include/moe.h), same call names.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  If the library
has not been built, ``lib()`` raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA, MOE_ETIMEOUT, MOE_ESTATE = range(6)
MOE_OUT_BF16, MOE_OUT_F32 = 0, 1
MOE_VIS_DETERMINISTIC, MOE_VIS_POLLED = 0, 1
MOE_FAULT_NONE, MOE_FAULT_COPY = 0, 1
MOE_POLICY_FREQ, MOE_POLICY_LRU, MOE_POLICY_FIFO, MOE_POLICY_SLRU = 0, 1, 2, 3
MOE_FMT_MXFP4, MOE_FMT_NVFP4 = 0, 1

EXPORTED = [
    "moe_layer_create", "moe_route", "moe_forward_slots", "moe_cache_update", "moe_destroy", "moe_last_error",
    "moe_layer_set_bias", "moe_layer_attach_staging", "moe_layer_stage_all", "moe_debug_get_map",
    "moe_debug_slot_ptr", "moe_debug_inject_fault", "moe_debug_stats", "moe_debug_profile",
    "moe_debug_profile_read", "moe_debug_check_error", "moe_policy_step", "moe_route_noalloc", "moe_forward_cold",
    "moe_forward_cold_gpu", "moe_host_expert_ffn", "moe_policy_step_recency", "moe_layer_set_policy",
    "moe_layer_set_device_cache", "moe_debug_device_cache", "moe_debug_decode_fusion", "moe_prefetch_step",
    "moe_prefetch", "moe_debug_stream_read", "moe_debug_mma_peak", "moe_policy_step_slru", "moe_ep_local_map",
]


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"moe status {code}: {msg}")
        self.code = code


class LayerDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("num_slots", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("max_refills_per_step", ctypes.c_int32),
                ("score_decay", ctypes.c_float), ("visibility", ctypes.c_int32), ("weight_format", ctypes.c_int32)]


_P = ctypes.c_void_p


class RouteBuffers(ctypes.Structure):
    """Caller-owned device buffers for moe_route_noalloc (device pointers)."""

    _fields_ = [(n, _P) for n in (
        "topk_ids", "topk_w", "hot_expert", "hot_token", "hot_w", "act_expert", "act_slot", "act_off",
        "act_cnt", "cold_token", "cold_expert", "cold_w", "hist", "counts")]


class RouteResult(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int32)] + [(n, _P) for n in (
        "topk_ids", "topk_w", "hot_expert", "hot_token", "hot_w", "act_expert", "act_slot", "act_off",
        "act_cnt", "cold_token", "cold_expert", "cold_w", "hist", "counts", "h_counts", "h_cold_token",
        "h_cold_expert", "h_cold_w", "h_hist", "done")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m expert_offload_moe_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        i32, p = ctypes.c_int32, _P
        L.moe_layer_create.argtypes = [ctypes.POINTER(LayerDesc), p, p, p, p, p, ctypes.POINTER(p)]
        L.moe_route.argtypes = [p, p, i32, p, ctypes.POINTER(RouteResult)]
        L.moe_forward_slots.argtypes = [p, p, p, i32, p]
        L.moe_forward_cold.argtypes = [p, p, p, i32, i32, p]
        L.moe_forward_cold_gpu.argtypes = [p, p, p, i32, p]
        L.moe_policy_step_recency.argtypes = [i32, p, p, p, p, p, i32, i32, p, ctypes.c_int64, ctypes.c_double,
                                              i32, p, p, p, p]
        L.moe_layer_set_policy.argtypes = [p, i32]
        L.moe_policy_step_slru.argtypes = [p, p, p, p, p, i32, i32, p, ctypes.c_int64, ctypes.c_double, i32, i32,
                                           p, p, p, p]
        L.moe_layer_set_device_cache.argtypes = [p, i32]
        L.moe_debug_device_cache.argtypes = [p, p]
        L.moe_host_expert_ffn.argtypes = [p, i32, i32, p, p]
        L.moe_cache_update.argtypes = [p, p, ctypes.POINTER(i32)]
        L.moe_destroy.argtypes = [p]
        L.moe_last_error.argtypes = []
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_layer_set_bias.argtypes = [p, p, p]
        L.moe_layer_attach_staging.argtypes = [p, p, ctypes.c_size_t]
        L.moe_layer_stage_all.argtypes = [p, p]
        L.moe_debug_get_map.argtypes = [p, p]
        L.moe_debug_slot_ptr.argtypes = [p, i32, ctypes.POINTER(p)]
        L.moe_debug_inject_fault.argtypes = [p, i32]
        L.moe_debug_stats.argtypes = [p, p]
        L.moe_debug_profile.argtypes = [p, i32]
        L.moe_debug_decode_fusion.argtypes = [p, i32]
        L.moe_prefetch_step.argtypes = [p, p, p, p, i32, i32, p, i32, p, p, p, p]
        L.moe_prefetch.argtypes = [p, p, i32, p, ctypes.POINTER(i32)]
        L.moe_debug_profile_read.argtypes = [p, p]
        L.moe_debug_check_error.argtypes = [p, ctypes.POINTER(i32)]
        L.moe_debug_stream_read.argtypes = [p, ctypes.c_size_t, p, i32, p]
        L.moe_debug_mma_peak.argtypes = [i32, i32, p, p]
        L.moe_ep_local_map.argtypes = [i32, i32, i32, p, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.moe_route_noalloc.argtypes = [p, i32, i32, p, p, i32, i32, p, ctypes.POINTER(RouteBuffers), p]
        L.moe_policy_step.argtypes = [p, p, p, p, i32, i32, p, ctypes.c_int64, ctypes.c_double, i32, p, p, p, p]
        for name in EXPORTED:
            if name != "moe_last_error":
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def check(rc):
    if rc != MOE_OK:
        raise MoeError(rc, lib().moe_last_error().decode())
    return rc


def stream_ptr(stream):
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return _P(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Layer:
    """One MoE layer: owns the slot bank, router copy, map and scratch on the GPU.

    ``router_w`` / ``router_bias``: fp32 CUDA tensors [E, H] / [E] (copied);
    ``host_bank``: page-locked uint8 CPU tensor [E, expert_bytes] (borrowed);
    ``expert_to_slot``: int32 sequence [E].
    """

    def __init__(self, hidden, inter, num_experts, top_k, num_slots, max_tokens, router_w, router_bias,
                 host_bank, expert_to_slot, out_f32=False, max_refills=2, score_decay=1.0,
                 visibility=MOE_VIS_DETERMINISTIC, stream=None, weight_format=0):
        import numpy as np

        self.h = None
        self.desc = LayerDesc(hidden, inter, num_experts, top_k, num_slots, max_tokens,
                              MOE_OUT_F32 if out_f32 else MOE_OUT_BF16, max_refills, score_decay, visibility,
                              weight_format)
        self._host_bank = host_bank  # keep the borrowed bank alive
        self._e2s = np.ascontiguousarray(np.asarray(expert_to_slot, dtype=np.int32))
        h = _P()
        bias_ptr = None if router_bias is None else _P(router_bias.data_ptr())
        check(lib().moe_layer_create(ctypes.byref(self.desc), _P(router_w.data_ptr()), bias_ptr,
                                     _P(host_bank.data_ptr()), self._e2s.ctypes.data_as(_P), stream_ptr(stream),
                                     ctypes.byref(h)))
        self.h = h
        self.res = RouteResult()

    def route(self, x, M, stream=None):
        check(lib().moe_route(self.h, _P(x.data_ptr()), M, stream_ptr(stream), ctypes.byref(self.res)))
        return self.res

    def forward_slots(self, x, out, M, stream=None):
        check(lib().moe_forward_slots(self.h, _P(x.data_ptr()), _P(out.data_ptr()), M, stream_ptr(stream)))

    def forward_cold(self, x, out, M, nthreads=0, stream=None):
        """Cold routes of the last route on host threads, added to ``out`` (blocks the calling thread)."""
        check(lib().moe_forward_cold(self.h, _P(x.data_ptr()), _P(out.data_ptr()), M, nthreads, stream_ptr(stream)))

    def set_policy(self, policy):
        """Slot policy for later cache updates: MOE_POLICY_FREQ (default), MOE_POLICY_LRU or MOE_POLICY_FIFO."""
        check(lib().moe_layer_set_policy(self.h, int(policy)))

    def set_device_cache(self, enable=True):
        """Decode calls keep and run the slot table on the GPU (demand-filled LRU, misses copied in by a kernel
        in the same step), or hand it back to the host policy.  Synchronises the device."""
        check(lib().moe_layer_set_device_cache(self.h, 1 if enable else 0))

    def device_cache_stats(self):
        """[steps, experts filled, hit experts, misses left cold] of the device slot table (synchronises)."""
        import numpy as np

        s = np.zeros(4, dtype=np.int64)
        check(lib().moe_debug_device_cache(self.h, s.ctypes.data_as(_P)))
        return s

    def forward_cold_gpu(self, x, out, M, stream=None):
        """Cold routes of the last route on the GPU, reading the host bank in place, added to ``out``."""
        check(lib().moe_forward_cold_gpu(self.h, _P(x.data_ptr()), _P(out.data_ptr()), M, stream_ptr(stream)))

    def cache_update(self, stream=None):
        n = ctypes.c_int32(0)
        check(lib().moe_cache_update(self.h, stream_ptr(stream), ctypes.byref(n)))
        return n.value

    def set_bias(self, bias, stream=None):
        check(lib().moe_layer_set_bias(self.h, None if bias is None else _P(bias.data_ptr()), stream_ptr(stream)))

    def attach_staging(self, buf):
        check(lib().moe_layer_attach_staging(self.h, None if buf is None else _P(buf.data_ptr()),
                                             0 if buf is None else buf.numel() * buf.element_size()))

    def stage_all(self, stream=None):
        check(lib().moe_layer_stage_all(self.h, stream_ptr(stream)))

    def get_map(self):
        import numpy as np

        out = np.empty(self.desc.num_experts, dtype=np.int32)
        check(lib().moe_debug_get_map(self.h, out.ctypes.data_as(_P)))
        return out

    def slot_ptr(self, slot):
        p = _P()
        check(lib().moe_debug_slot_ptr(self.h, slot, ctypes.byref(p)))
        return p.value

    def inject_fault(self, fault):
        check(lib().moe_debug_inject_fault(self.h, fault))

    def stats(self):
        import numpy as np

        s = np.zeros(4, dtype=np.int64)
        check(lib().moe_debug_stats(self.h, s.ctypes.data_as(_P)))
        return s

    def check_error(self):
        """Raises MoeError(MOE_ETIMEOUT) if a tensor-core kernel gave up a bounded wait since the last check."""
        code = ctypes.c_int32(0)
        check(lib().moe_debug_check_error(self.h, ctypes.byref(code)))

    def prefetch(self, x, M, stream=None):
        """Next-layer prefetch: this layer's router predicts its experts from ``x`` (the current layer's input)
        and the predicted experts missing from its slots are copied in now.  Returns the refills issued."""
        n = ctypes.c_int32(0)
        check(lib().moe_prefetch(self.h, _P(x.data_ptr()), M, stream_ptr(stream), ctypes.byref(n)))
        return n.value

    def decode_fusion(self, enable):
        check(lib().moe_debug_decode_fusion(self.h, 1 if enable else 0))

    def profile(self, enable):
        check(lib().moe_debug_profile(self.h, 1 if enable else 0))

    def profile_read(self):
        import numpy as np

        out = np.zeros(4, dtype=np.float64)
        check(lib().moe_debug_profile_read(self.h, out.ctypes.data_as(_P)))
        return out

    def close(self):
        if getattr(self, "h", None):
            lib().moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def route_noalloc(x, M, router_w, router_bias, E, top_k, expert_to_slot_dev, bufs: dict, stream=None):
    """moe_route_noalloc: routes into the caller's device tensors in ``bufs`` (keys as RouteBuffers)."""
    rb = RouteBuffers(*[_P(bufs[n].data_ptr()) for n, _ in RouteBuffers._fields_])
    H = x.shape[-1]
    check(lib().moe_route_noalloc(_P(x.data_ptr()), M, H, _P(router_w.data_ptr()),
                                  None if router_bias is None else _P(router_bias.data_ptr()), E, top_k,
                                  _P(expert_to_slot_dev.data_ptr()), ctypes.byref(rb), stream_ptr(stream)))


def policy_step(score, last, e2s, s2e, hist, step, decay, R, in_flight=None):
    """The library's slot-cache decision on numpy arrays (updated in place)."""
    import numpy as np

    E, S = e2s.shape[0], s2e.shape[0]
    pe, ps, pv = (np.zeros(max(R, 1), dtype=np.int32) for _ in range(3))
    fl = None if in_flight is None else np.ascontiguousarray(in_flight, dtype=np.uint8)
    hist = np.ascontiguousarray(hist, dtype=np.int32)
    n = lib().moe_policy_step(score.ctypes.data_as(_P), last.ctypes.data_as(_P), e2s.ctypes.data_as(_P),
                              s2e.ctypes.data_as(_P), E, S, hist.ctypes.data_as(_P),
                              int(step), float(decay), int(R), None if fl is None else fl.ctypes.data_as(_P),
                              pe.ctypes.data_as(_P), ps.ctypes.data_as(_P), pv.ctypes.data_as(_P))
    if n < 0:
        raise MoeError(MOE_EINVAL, "moe_policy_step rejected its arguments")
    return [(int(pe[i]), int(ps[i]), int(pv[i])) for i in range(n)]


def policy_step_recency(policy, score, last, loaded, e2s, s2e, hist, step, decay, R, in_flight=None):
    """The library's LRU / FIFO slot decision on numpy arrays (updated in place)."""
    import numpy as np

    E, S = e2s.shape[0], s2e.shape[0]
    pe, ps, pv = (np.zeros(max(R, 1), dtype=np.int32) for _ in range(3))
    fl = None if in_flight is None else np.ascontiguousarray(in_flight, dtype=np.uint8)
    hist = np.ascontiguousarray(hist, dtype=np.int32)
    n = lib().moe_policy_step_recency(int(policy), score.ctypes.data_as(_P), last.ctypes.data_as(_P),
                                      None if loaded is None else loaded.ctypes.data_as(_P), e2s.ctypes.data_as(_P),
                                      s2e.ctypes.data_as(_P), E, S, hist.ctypes.data_as(_P), int(step), float(decay),
                                      int(R), None if fl is None else fl.ctypes.data_as(_P), pe.ctypes.data_as(_P),
                                      ps.ctypes.data_as(_P), pv.ctypes.data_as(_P))
    if n < 0:
        raise MoeError(MOE_EINVAL, "moe_policy_step_recency rejected its arguments")
    return [(int(pe[i]), int(ps[i]), int(pv[i])) for i in range(n)]


def policy_step_slru(score, last, seg, e2s, s2e, hist, step, decay, R, pcap, in_flight=None):
    """The library's segmented-LRU slot decision on numpy arrays (updated in place)."""
    import numpy as np

    E, S = e2s.shape[0], s2e.shape[0]
    pe, ps, pv = (np.zeros(max(R, 1), dtype=np.int32) for _ in range(3))
    fl = None if in_flight is None else np.ascontiguousarray(in_flight, dtype=np.uint8)
    hist = np.ascontiguousarray(hist, dtype=np.int32)
    n = lib().moe_policy_step_slru(score.ctypes.data_as(_P), last.ctypes.data_as(_P), seg.ctypes.data_as(_P),
                                   e2s.ctypes.data_as(_P), s2e.ctypes.data_as(_P), E, S, hist.ctypes.data_as(_P),
                                   int(step), float(decay), int(R), int(pcap),
                                   None if fl is None else fl.ctypes.data_as(_P), pe.ctypes.data_as(_P),
                                   ps.ctypes.data_as(_P), pv.ctypes.data_as(_P))
    if n < 0:
        raise MoeError(MOE_EINVAL, "moe_policy_step_slru rejected its arguments")
    return [(int(pe[i]), int(ps[i]), int(pv[i])) for i in range(n)]


def prefetch_step(score, last, e2s, s2e, pred, R, in_flight=None):
    """The library's next-layer prefetch decision on numpy arrays (e2s / s2e updated in place)."""
    import numpy as np

    E, S = e2s.shape[0], s2e.shape[0]
    pe, ps, pv = (np.zeros(max(R, 1), dtype=np.int32) for _ in range(3))
    fl = None if in_flight is None else np.ascontiguousarray(in_flight, dtype=np.uint8)
    pred = np.ascontiguousarray(pred, dtype=np.int32)
    n = lib().moe_prefetch_step(score.ctypes.data_as(_P), last.ctypes.data_as(_P), e2s.ctypes.data_as(_P),
                                s2e.ctypes.data_as(_P), E, S, pred.ctypes.data_as(_P), int(R),
                                None if fl is None else fl.ctypes.data_as(_P), pe.ctypes.data_as(_P),
                                ps.ctypes.data_as(_P), pv.ctypes.data_as(_P))
    if n < 0:
        raise MoeError(MOE_EINVAL, "moe_prefetch_step rejected its arguments")
    return [(int(pe[i]), int(ps[i]), int(pv[i])) for i in range(n)]


def host_expert_ffn(record, H, I, x_bits):
    """The library's host expert FFN (the one its cold-route workers run) on one record: fp32 [H]."""
    import numpy as np

    rec = np.ascontiguousarray(record, dtype=np.uint8)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    y = np.empty(H, dtype=np.float32)
    check(lib().moe_host_expert_ffn(rec.ctypes.data_as(_P), H, I, x.ctypes.data_as(_P), y.ctypes.data_as(_P)))
    return y


def stream_read(src, nbytes, sink, stream=None, nblocks=0):
    """One launch of the library's streaming-read probe over ``nbytes`` bytes at device pointer ``src``."""
    check(lib().moe_debug_stream_read(_P(int(src)), nbytes, _P(int(sink)), nblocks, stream_ptr(stream)))


def mma_peak(iters, err, stream=None, nblocks=0):
    """One launch of the library's block-scaled MMA probe (nblocks x iters x 4 MMAs of 128 x 256 x 32)."""
    check(lib().moe_debug_mma_peak(iters, nblocks, _P(int(err)), stream_ptr(stream)))


def mma_peak_flops(iters, nblocks):
    return float(nblocks) * iters * 4 * 2 * 128 * 256 * 32


def ep_local_map(E, world, rank):
    """moe_ep_local_map: (expert_to_slot int32 [E] of the rank's shard, first expert, expert count)."""
    import numpy as np

    e2s = np.empty(E, dtype=np.int32)
    first, count = ctypes.c_int32(0), ctypes.c_int32(0)
    rc = lib().moe_ep_local_map(int(E), int(world), int(rank), e2s.ctypes.data_as(_P), ctypes.byref(first),
                                ctypes.byref(count))
    if rc != MOE_OK:
        raise MoeError(rc, f"moe_ep_local_map({E}, {world}, {rank}) rejected its arguments")
    return e2s, first.value, count.value
