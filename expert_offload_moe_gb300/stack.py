"""A stack of independent MoE layers built from the seeded workloads, and the
decode step over it (route + forward for every layer), optionally captured
as one CUDA graph.

Layers are independent instances with their own fresh N(0,1) input each step
(chaining them without attention and norms would overflow); this is how the
workloads are timed and checked.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import moe, synth


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device != "cpu" else t


def pinned_bank(seed: int, layer: int, E: int, H: int, I: int, weight_format: int = 0) -> torch.Tensor:
    eb = synth.expert_bytes(H, I, weight_format)
    bank = torch.empty((E, eb), dtype=torch.uint8, pin_memory=True)
    synth.fill_expert_records(bank.numpy(), seed, layer, H, I, first=0, weight_format=weight_format)
    return bank


def host_counts(res) -> np.ndarray:
    """The page-locked mirror of (n_hot, n_cold, n_active, M) of a route result."""
    return np.ctypeslib.as_array(ctypes.cast(res.h_counts, ctypes.POINTER(ctypes.c_int32)), (4,)).copy()


class LayerInputs:
    """Everything one layer of a workload needs (host copies kept for the oracle)."""

    def __init__(self, w: synth.Workload, layer: int, seed: int = 0, e2s=None, bias_order=0):
        self.w, self.layer, self.seed = w, layer, seed
        H, I, E = w.hidden, w.inter, w.experts
        self.Wr = synth.router_weights(seed, layer, E, H)
        self.bias = synth.router_bias(seed, layer, E, w.bias_tau, bias_order)
        self.e2s = synth.expert_to_slot_by_rank(seed, layer, E, w.slots) if e2s is None else np.asarray(e2s, np.int32)
        self.bank = pinned_bank(seed, layer, E, H, I, w.weight_format)

    def make_layer(self, max_tokens=8, out_f32=False, **kw) -> moe.Layer:
        w = self.w
        return moe.Layer(w.hidden, w.inter, w.experts, w.top_k, w.slots, max_tokens,
                         torch.from_numpy(self.Wr).cuda(), torch.from_numpy(self.bias).cuda(), self.bank,
                         self.e2s, out_f32=out_f32, weight_format=w.weight_format, **kw)


class DecodeStack:
    """L layers of one workload with M-token decode steps over resident inputs."""

    def __init__(self, w: synth.Workload, M: int = 1, n_layers: int | None = None, seed: int = 0,
                 n_inputs: int = 1, out_f32: bool = False, max_tokens: int = 8, cold_on_gpu: bool = False):
        """cold_on_gpu: each layer also computes its cold routes on the GPU from the host bank in place."""
        self.w, self.M, self.seed = w, M, seed
        self.cold_on_gpu = cold_on_gpu
        self.L = w.layers if n_layers is None else n_layers
        self.inputs = [LayerInputs(w, l, seed) for l in range(self.L)]
        self.layers = [li.make_layer(max_tokens=max_tokens, out_f32=out_f32) for li in self.inputs]
        H = w.hidden
        # n_inputs steps of fresh activations per layer, resident in HBM: [n_inputs, L, M, H]
        xs = np.stack([np.stack([synth.activations(seed, l, s, M, H) for l in range(self.L)])
                       for s in range(n_inputs)])
        self.x_host = xs
        self.x_all = bf16_tensor(xs)
        self.x_cur = torch.empty((self.L, M, H), dtype=torch.bfloat16, device="cuda")
        dt = torch.float32 if out_f32 else torch.bfloat16
        self.out = torch.empty((self.L, M, H), dtype=dt, device="cuda")
        self.graph = None
        self.graph_stream = None

    def _body(self, stream):
        for l, layer in enumerate(self.layers):
            layer.route(self.x_cur[l], self.M, stream)
            layer.forward_slots(self.x_cur[l], self.out[l], self.M, stream)
            if self.cold_on_gpu:
                layer.forward_cold_gpu(self.x_cur[l], self.out[l], self.M, stream)

    def load_inputs(self, i: int):
        self.x_cur.copy_(self.x_all[i % self.x_all.shape[0]], non_blocking=True)

    def step(self, i: int = 0):
        """One decode step over every layer (eager launches on the current stream)."""
        self.load_inputs(i)
        self._body(torch.cuda.current_stream())

    def capture(self):
        """Captures the step body (all layers) as one CUDA graph."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(2):
                self._body(s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self._body(s)
        torch.cuda.synchronize()
        self.graph, self.graph_stream = g, s
        return g

    def replay(self, i: int = 0):
        self.load_inputs(i)
        self.graph.replay()

    def close(self):
        for l in self.layers:
            l.close()
        self.layers = []


class EPShard:
    """One rank's shard of an expert-parallel layer (xinfer docs "Options": each rank loads and offloads its own
    expert shard; NCCL combines the rank-local MoE results).  The router is replicated; the layer holds only
    the rank's contiguous range of experts (moe_ep_local_map), computes the routes to them and returns the
    rest as its cold list; ``forward`` then sums the ranks' fp32 outputs with one all-reduce."""

    def __init__(self, inputs: LayerInputs, world: int, rank: int, max_tokens: int = 8):
        w = inputs.w
        self.world, self.rank = world, rank
        self.e2s, self.first, self.count = moe.ep_local_map(w.experts, world, rank)
        self.layer = moe.Layer(w.hidden, w.inter, w.experts, w.top_k, self.count, max_tokens,
                               torch.from_numpy(inputs.Wr).cuda(), torch.from_numpy(inputs.bias).cuda(), inputs.bank,
                               self.e2s, out_f32=True, weight_format=w.weight_format)

    def forward(self, x: torch.Tensor, M: int, out: torch.Tensor, group=None, stream=None, reduce: bool = True):
        """Routes and computes this rank's routes into ``out`` (fp32 [M, H]), then (reduce, world > 1) all-reduces
        it over the ranks.  Returns the route result (its cold list = the other ranks' routes)."""
        res = self.layer.route(x, M, stream)
        self.layer.forward_slots(x, out, M, stream)
        if reduce and self.world > 1:
            torch.distributed.all_reduce(out, group=group)
        return res

    def close(self):
        self.layer.close()


def ep_host_partial(bank: np.ndarray, e2s_local: np.ndarray, ids: np.ndarray, w: np.ndarray, x_bits: np.ndarray,
                    H: int, I: int) -> np.ndarray:
    """A rank's share of an expert-parallel layer on the host: for each token, the fp32 sum in ascending expert
    order of w * FFN_e(x) over its routes to the experts this rank holds (e2s_local[e] >= 0), each FFN run by
    the library's host expert FFN (the one its cold-route workers use).  [M, H] fp32."""
    M, k = ids.shape
    out = np.zeros((M, H), dtype=np.float32)
    for t in range(M):
        for j in np.argsort(ids[t], kind="stable"):
            e = int(ids[t][j])
            if e2s_local[e] >= 0:
                y = moe.host_expert_ffn(bank[e], H, I, x_bits[t])
                out[t] = (out[t] + np.float32(w[t][j]) * y).astype(np.float32)
    return out


class PrefillStack:
    """L layers of one workload with the whole expert bank staged on the device, and the M-token prefill
    step over it (route + forward of every layer on the tensor cores)."""

    def __init__(self, w: synth.Workload, M: int | None = None, n_layers: int | None = None, seed: int = 0,
                 n_inputs: int = 2, out_f32: bool = False):
        self.w, self.seed = w, seed
        self.M = w.prefill_tokens if M is None else M
        self.L = w.layers if n_layers is None else n_layers
        self.layers, self.staging = [], []
        H, M = w.hidden, self.M
        for l in range(self.L):
            li = LayerInputs(w, l, seed)
            lay = li.make_layer(max_tokens=M, out_f32=out_f32)
            buf = torch.empty(w.experts * w.expert_bytes, dtype=torch.uint8, device="cuda")
            lay.attach_staging(buf)
            lay.stage_all()
            self.layers.append(lay)
            self.staging.append(buf)
            del li  # the pinned host bank is only needed until staged
        torch.cuda.synchronize()
        # n_inputs fresh activation batches per layer, resident in HBM: [n_inputs, L, M, H]
        self.x_all = torch.empty((n_inputs, self.L, M, H), dtype=torch.bfloat16, device="cuda")
        for s in range(n_inputs):
            for l in range(self.L):
                self.x_all[s, l].copy_(bf16_tensor(synth.activations(seed, l, s, M, H), device="cpu"))
        dt = torch.float32 if out_f32 else torch.bfloat16
        self.out = torch.empty((self.L, M, H), dtype=dt, device="cuda")

    def step(self, i: int = 0, stream=None):
        """One prefill step: every layer routes and runs its own batch i (eager launches)."""
        x = self.x_all[i % self.x_all.shape[0]]
        for l, layer in enumerate(self.layers):
            layer.route(x[l], self.M, stream)
            layer.forward_slots(x[l], self.out[l], self.M, stream)

    def close(self):
        for l in self.layers:
            l.close()
        self.layers, self.staging = [], []
