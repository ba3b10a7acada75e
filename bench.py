#!/usr/bin/env python3
"""Decode-time MoE layer with GPU expert slots: throughput on one GB300.

Workload (default): the gpt-oss-20B-shaped stack -- 24 independent layers,
hidden 2880, expert intermediate 2880, 32 experts, top-4, every expert in a
GPU slot, M=1 decode, each layer with its own fresh N(0,1) bf16 input every
step, MXFP4 experts (~10 GB).  A step = route + forward of all 24 layers for
one token (one CUDA-graph replay), so tokens/s = steps / time.

Printed (rank 0, one JSON line): value (tokens/s with inputs resident in HBM),
e2e (host inputs copied in and outputs copied back each step), roofline of
the dominant kernel (gate/up GEMV, HBM-bound), the oracle as a CPU baseline,
clocks sampled during the timed region, and the kernel launch count.

`--impl reference` times the CPU oracle instead (the slow, plain reference),
on a bounded sample of the same workload.

Other lines (not the default): `--workload gptoss20b_prefill2048_s16_lfu_drift`
times the 2048-token prefill of every layer (tensor-core roofline of the
gate/up GEMM); `--cold-on-gpu` / `--cold-on-host` time decode with the cold
routes computed as well (on the GPU from the host bank in place, or on the
host cores).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "gptoss20b_h2880_e32k4_resident_m1"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
METRIC = "MoE-layer decode tokens/s (M=1)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--layers", type=int, default=None, help="fewer layers (debug only; not a valid result)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-layers", type=int, default=1, help="layers per oracle step (reference arm sample)")
    ap.add_argument("--cold-on-host", action="store_true",
                    help="decode with the cold routes computed on the host cores (moe_forward_cold) as well")
    ap.add_argument("--policy-sweep", action="store_true",
                    help="hot-route hit rate and refills of each slot policy on the drifting decode workload")
    ap.add_argument("--cold-on-gpu", action="store_true",
                    help="decode with the cold routes computed on the GPU from the host bank in place as well")
    ap.add_argument("--tokens", type=int, default=None,
                    help="decode batch M (default: the workload's first; e.g. 8 for the M=8 speculative-verify line)")
    ap.add_argument("--two-launch", action="store_true",
                    help="M = 1 decode with separate gate/up and down launches instead of the one-launch FFN")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)), "measured"
    return PEAKS_FALLBACK, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_token_seconds(w, n_layers, seed=0):
    """The oracle, as it stands, on one host core: seconds for one token through n_layers layers."""
    import oracle
    from expert_offload_moe_gb300 import synth

    oracle.build()
    t_total = 0.0
    for l in range(n_layers):
        Wr = synth.router_weights(seed, l, w.experts, w.hidden)
        b = synth.router_bias(seed, l, w.experts, w.bias_tau)
        ex = synth.expert_records(seed, l, w.experts, w.hidden, w.inter, weight_format=w.weight_format)
        e2s = synth.expert_to_slot_by_rank(seed, l, w.experts, w.slots)
        x = synth.activations(seed, l, 0, 1, w.hidden)
        t0 = time.perf_counter()
        oracle.moe_layer(x, Wr, b, ex, e2s, w.top_k, w.hidden, w.inter, fmt="nvfp4" if w.weight_format else "mxfp4")
        t_total += time.perf_counter() - t0
        del ex
    return t_total


def cpu_baseline(w, n_layers):
    t = oracle_token_seconds(w, n_layers)
    per_token = t / n_layers * w.layers
    return {"value": 1.0 / per_token, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"1 token through {n_layers} of {w.layers} layers (single-threaded C oracle, "
                      f"{t:.1f} s), time scaled to the {w.layers}-layer stack"}


def _oracle_layer_worker(args):
    """One worker process: the oracle for token 0 of one layer, after a shared start time (for the pool)."""
    name, layer, start_at = args
    import oracle
    from expert_offload_moe_gb300 import synth

    w = synth.WORKLOADS[name]
    oracle.build()
    Wr = synth.router_weights(0, layer, w.experts, w.hidden)
    b = synth.router_bias(0, layer, w.experts, w.bias_tau)
    ex = synth.expert_records(0, layer, w.experts, w.hidden, w.inter, weight_format=w.weight_format)
    e2s = synth.expert_to_slot_by_rank(0, layer, w.experts, w.slots)
    x = synth.activations(0, layer, 0, 1, w.hidden)
    while time.time() < start_at:
        time.sleep(0.001)
    t0 = time.time()
    oracle.moe_layer(x, Wr, b, ex, e2s, w.top_k, w.hidden, w.inter, fmt="nvfp4" if w.weight_format else "mxfp4")
    return t0, time.time()


def cpu_baseline_all_cores(w):
    """The oracle on every host core at once: one spawned process per core (at most one per layer), each
    running its own layer for the same token; throughput from the wall clock of the whole batch."""
    import multiprocessing as mp

    cores = max(1, min(os.cpu_count() or 1, w.layers))
    ctx = mp.get_context("spawn")  # the parent process holds a CUDA context: never fork it
    with ctx.Pool(cores) as pool:
        # data generation is not timed: every worker starts its oracle call at the same wall-clock time
        start_at = time.time() + 20.0 + 0.5 * cores
        spans = pool.map(_oracle_layer_worker, [(w.name, l, start_at) for l in range(cores)])
    wall = max(e for _, e in spans) - min(s for s, _ in spans)
    per_token = wall / cores * w.layers
    return {"value": 1.0 / per_token, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"1 token through {cores} of {w.layers} layers, one layer per process on {cores} host cores "
                      f"({wall:.2f} s wall), time scaled to the {w.layers}-layer stack"}


def run_reference(args, prefill=False):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from expert_offload_moe_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    total = 0.0
    n_tok = 2 if prefill else 1
    layers = 1 if prefill else args.ref_layers
    for i in range(args.warmup + args.steps):
        # the time actually measured for one step's sample: n_tok tokens through `layers` of the stack's layers
        t = oracle_prefill_seconds(w, n_tok) if prefill else oracle_token_seconds(w, layers)
        if i >= args.warmup:
            total += t
    # each step processes layers / L of the stack for n_tok tokens: that many whole-stack tokens per step
    token_equiv = n_tok * layers / w.layers
    val = args.steps * token_equiv / total
    what = f"{n_tok} {'prompt tokens' if prefill else 'token'} through {layers} of {w.layers} layers"
    line = {"impl": "reference", "metric": PREFILL_METRIC if prefill else METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.layers, "tokens_per_step": n_tok,
                       "step": f"{what} ({token_equiv:.4g} whole-stack tokens); ms_per_step is that sample's "
                               f"measured time, value = whole-stack tokens / measured time"},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: {what} on one core"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# committed ncu traffic summaries: (kernel, workload, tokens per step) -> file under profiles/
TRAFFIC_SUMMARIES = {
    ("ffn_tc_kernel", "gptoss20b_h2880_e32k4_resident_m1", 1): "ffn_tc_gptoss20b_traffic.txt",
    ("ffn_tc_kernel", "e512k10_h2048_i512_s256_m1", 1): "ffn_tc_e512k10_s256_traffic.txt",
    ("gateup_tc_kernel", "e512k10_h2048_i512_s384_m4m8", 8): "gateup_tc_e512k10_s384_m8_traffic.txt",
}


def traffic_for(kernel_src, kernel, workload, M):
    """DRAM bytes per launch from the committed ncu summary of this kernel on this workload, if it was taken
    on this kernel source."""
    summary = TRAFFIC_SUMMARIES.get((kernel, workload, M))
    if summary is None:
        return None
    summ = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(summ):
        return None
    sha = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()
    kv = {}
    for line in open(summ):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != sha:
        return None
    try:
        return float(kv["dram_bytes_per_launch_full_workload"])
    except (KeyError, ValueError):
        return None


def job_time(t_local, world, device):
    """The job's time: the largest of every rank's time for the same steps (an all-reduce MAX over the
    process group; the value on one rank is its own).  device: where the reduction tensor lives."""
    if world == 1:
        return float(t_local)
    import torch
    import torch.distributed as dist

    tt = torch.tensor([float(t_local)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_rate(units_per_rank, t_local_ms, world, device):
    """Whole-job throughput: the units every rank processed over the slowest rank's time (weak scaling,
    independent replicas)."""
    t_ms = job_time(t_local_ms, world, device)
    return units_per_rank * world / (t_ms / 1e3), t_ms


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from expert_offload_moe_gb300 import build as moe_build
    from expert_offload_moe_gb300 import moe, stack, synth

    moe_build.build()
    moe.lib()
    w = synth.WORKLOADS[args.workload]
    M = args.tokens or w.tokens[0]
    n_inputs = 64
    st = stack.DecodeStack(w, M=M, n_layers=args.layers, seed=rank, n_inputs=n_inputs,
                           cold_on_gpu=args.cold_on_gpu)
    L = st.L
    if args.two_launch:
        for lay in st.layers:
            lay.decode_fusion(False)
    st.capture()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return job_time(v, world, "cuda")

    # ---------------- timed region: graph replay, inputs resident in HBM -------
    for i in range(args.warmup):
        st.replay(i)
    barrier()
    clk = Clocks(local)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        st.replay(i)
    e1.record(stream)
    barrier()
    clocks = clk.stop()
    t_ms = max_over_ranks(e0.elapsed_time(e1))
    tokens = args.steps * M * world
    value = tokens / (t_ms / 1e3)

    # the timed region is short (a few tens of ms); the clocks are also sampled over >= 1.5 s of the same
    # graph replays right after it, so that the record has enough samples to show a throttle or a lock
    clk_long = Clocks(local)
    clk_long.start()
    n_long, t_long = 0, time.perf_counter()
    while time.perf_counter() - t_long < 1.5 or n_long < args.steps:
        st.replay(n_long)
        n_long += 1
        if n_long % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    window_s = time.perf_counter() - t_long
    clocks_sustained = clk_long.stop()
    clocks_sustained.update({"window_s": round(window_s, 3), "graph_replays": n_long,
                             "note": "same graph replays, right after the timed region"})

    # expert bytes actually read (the routing of every input is fixed, so one pass gives the mix)
    n_act, n_cold_e = [], []
    for i in range(n_inputs):
        st.step(i)
        torch.cuda.synchronize()
        for l in range(L):
            c = stack.host_counts(st.layers[l].res)
            n_act.append(int(c[2]))
            if args.cold_on_gpu:  # distinct cold experts (each streamed once from the host bank)
                cold = np.ctypeslib.as_array(ctypes.cast(st.layers[l].res.h_cold_expert,
                                                         ctypes.POINTER(ctypes.c_int32)), (int(c[1]),))
                n_cold_e.append(len(set(cold.tolist())))
    mean_act = float(np.mean(n_act))
    code_scale_bytes = 0.5 + 1.0 / synth.scale_block(w.weight_format)  # bytes per weight: code + its share of a scale
    gateup_bytes = mean_act * 2 * w.inter * w.hidden * code_scale_bytes
    expert_bytes_step = mean_act * w.expert_bytes * L
    router_bytes_step = w.experts * w.hidden * 4 * L

    # ---------------- kernel timing pass (events on the launching stream) -------
    # One step captured as its own CUDA graph with each kernel between two event-record nodes: replays run
    # the kernels back to back on the device (no host submission gaps), each one after the previous has
    # finished (an event node ends programmatic overlap), and the events time each kernel alone.
    kt_steps = min(args.steps, 128)
    for lay in st.layers:
        lay.profile(True)
    pg, ps = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    ps.wait_stream(stream)
    with torch.cuda.graph(pg, stream=ps):
        st._body(ps)
    torch.cuda.synchronize()
    prof = np.zeros(4)
    for i in range(kt_steps):
        st.load_inputs(i)
        pg.replay()
        torch.cuda.synchronize()
        for lay in st.layers:
            prof += lay.profile_read()
    for lay in st.layers:
        lay.profile(False)
    del pg
    launches = max(prof[3], 1)
    route_us, gateup_us, down_us = (1e3 * prof[i] / launches for i in range(3))
    pk, pk_src = peaks()
    hbm_peak = pk.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"])
    src = os.path.join(ROOT, "expert_offload_moe_gb300", "csrc", "moe_decode_tc.cu")
    if w.weight_format != 0 and M == 1 and not args.two_launch:  # NVFP4 one-token FFN on the tensor cores
        kernel, kbytes = "ffn_nv_kernel", mean_act * w.expert_bytes
        kernel_us = {"route": route_us, "ffn": gateup_us, "combine": down_us}
        traffic = None
    elif w.weight_format != 0:  # NVFP4 batches: CUDA-core decode kernels
        kernel, kbytes = "gateup_kernel", gateup_bytes
        kernel_us = {"route": route_us, "gateup": gateup_us, "down": down_us}
        traffic = None
    elif M == 1 and not args.two_launch:  # gate/up, SiLU and down in one launch (every expert byte), then combine
        kernel, kbytes = "ffn_tc_kernel", mean_act * w.expert_bytes
        kernel_us = {"route": route_us, "ffn": gateup_us, "combine": down_us}
        traffic = traffic_for(src, kernel, w.name, M)
    else:
        kernel, kbytes = "gateup_tc_kernel", gateup_bytes
        kernel_us = {"route": route_us, "gateup": gateup_us, "down": down_us}
        traffic = traffic_for(src, kernel, w.name, M)
    achieved = kbytes / (gateup_us * 1e-6) / 1e9

    # ---------------- floor: a plain read of the same bytes, timed the same way -----
    # one launch of the library's streaming-read probe per layer in turn, over that layer's slot bank (the
    # stack's banks together are far larger than L2), CUDA events around each launch on the same stream
    probe_bytes = int(kbytes) // 16 * 16
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    bank_ptrs = [lay.slot_ptr(0) for lay in st.layers]
    for l in range(min(L, 3)):
        moe.stream_read(bank_ptrs[l], probe_bytes, sink.data_ptr(), stream)
    try:  # event-record nodes in a graph, like the kernels above
        pev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(L)]
        probe_graph = True
    except TypeError:  # a torch without external events: eager launches
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
        probe_graph = False

    def probe_body(s):
        for l in range(L):
            pev[l][0].record(s)
            moe.stream_read(bank_ptrs[l], probe_bytes, sink.data_ptr(), s)
            pev[l][1].record(s)

    probe_t = []
    if probe_graph:
        pg = torch.cuda.CUDAGraph()
        ps.wait_stream(stream)
        with torch.cuda.graph(pg, stream=ps):
            probe_body(ps)
    for i in range(max(1, kt_steps // L)):
        if probe_graph:
            pg.replay()
        else:
            probe_body(stream)
        torch.cuda.synchronize()
        probe_t += [a.elapsed_time(b) for a, b in pev]
    probe_us = 1e3 * float(np.mean(probe_t))
    read_probe = {"bytes_per_launch": probe_bytes, "avg_launch_us": probe_us,
                  "achieved": probe_bytes / (probe_us * 1e-6) / 1e9, "frac": probe_bytes / (probe_us * 1e-6) / 1e9 / hbm_peak,
                  "note": "plain 128-bit streaming read of the same bytes, one event-timed launch per layer's bank"}
    timing_note = ("CUDA events around each kernel on its stream, recorded as event nodes of a captured step "
                   "graph: kernels back to back on the device, each after the previous one has finished; the "
                   "plain read %s" % ("likewise" if probe_graph else "by eager launches (no external events)"))

    # ---------------- e2e: host inputs in, outputs back, every step ------------
    x_host = torch.empty((n_inputs, L, M, w.hidden), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(st.x_all.cpu())
    out_host = torch.empty(st.out.shape, dtype=st.out.dtype, pin_memory=True)
    for i in range(args.warmup):
        st.x_cur.copy_(x_host[i % n_inputs], non_blocking=True)
        st.graph.replay()
        out_host.copy_(st.out, non_blocking=True)
    barrier()
    e0.record(stream)
    for i in range(args.steps):
        st.x_cur.copy_(x_host[i % n_inputs], non_blocking=True)
        st.graph.replay()
        out_host.copy_(st.out, non_blocking=True)
    e1.record(stream)
    barrier()
    t_e2e = max_over_ranks(e0.elapsed_time(e1))
    e2e = {"value": tokens / (t_e2e / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": L * M * w.hidden * 2,
           "d2h_bytes_per_step": int(st.out.numel() * st.out.element_size())}

    metric = METRIC
    if args.cold_on_gpu:
        metric = "MoE-layer decode tokens/s (M=1), cold routes computed on the GPU from the host bank in place"
    line = {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4*bf16->f32" if w.weight_format else "mxfp4*e4m3->f32", "data": "synthetic",
        "config": {"workload": w.name, "layers": L, "hidden": w.hidden, "inter": w.inter, "experts": w.experts,
                   "top_k": w.top_k, "slots": w.slots, "tokens_per_step": M, "parallelism": f"replicas{world}",
                   "weights": ("nvfp4" if w.weight_format else "mxfp4") + " experts, fp32 router, fp32 accumulation",
                   "l2": "inputs larger than L2: each step reads %.2f GB of distinct expert weights"
                         % (expert_bytes_step / 1e9),
                   "expert_gbs": expert_bytes_step / (t_ms / args.steps * 1e-3) / 1e9,
                   "router_gbs": router_bytes_step / (t_ms / args.steps * 1e-3) / 1e9,
                   "mean_active_experts": mean_act,
                   "kernel_us": kernel_us},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "bytes_per_launch": kbytes, "avg_launch_us": gateup_us, "plain_read_same_bytes": read_probe,
                     "timing": timing_note,
                     "peak_source": "measured hbm_gbs (MEASURED_PEAKS.json)" if pk_src == "measured"
                     else "fallback 6.8 TB/s"},
        "clocks": clocks,
        "clocks_sustained": clocks_sustained,
        "gpu_launches": int(args.steps * L * (3 + (4 if args.cold_on_gpu else 0))),
        "e2e": e2e,
    }
    if args.cold_on_gpu:
        host_bytes = float(np.mean(n_cold_e)) * w.expert_bytes * L
        line["config"]["cold_routes"] = {
            "mean_distinct_cold_experts_per_layer": float(np.mean(n_cold_e)),
            "host_bank_gbs": host_bytes / (t_ms / args.steps * 1e-3) / 1e9,
            "note": "hot experts from HBM slots on the tensor cores; cold experts streamed from page-locked "
                    "host memory by the CUDA-core kernels; every route of every token computed"}
    st.close()
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, 1)
        try:
            line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(w)
        except Exception as exc:  # the single-core figure stands on its own
            line["cpu_baseline_all_cores"] = {"unavailable": f"{type(exc).__name__}: {exc}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


PREFILL_METRIC = "MoE-layer prefill tokens/s (M=2048)"
FP8_OVER_BF16 = 2.0  # nominal dense ratio of the 8-bit block-scaled tensor rate to bf16 (4.5 / 2.25 PFLOP/s)


def run_prefill(args):
    """The prompt phase of the prefill-then-decode workload: every layer routes and runs a batch of
    M = prefill_tokens on the tensor cores over its staged expert bank.  A step = all layers, eager launches."""
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from expert_offload_moe_gb300 import build as moe_build
    from expert_offload_moe_gb300 import moe, stack, synth

    moe_build.build()
    moe.lib()
    w = synth.WORKLOADS[args.workload]
    st = stack.PrefillStack(w, n_layers=args.layers, seed=rank, n_inputs=2)
    L, M = st.L, st.M
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        st.step(i)
    torch.cuda.synchronize()
    clk = Clocks(local)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        st.step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    t_ms = e0.elapsed_time(e1)
    value = args.steps * M / (t_ms / 1e3)

    # per-GEMM device time (events on the launching stream, around each launch)
    for lay in st.layers:
        lay.profile(True)
    kt_steps = min(args.steps, 8)
    for i in range(kt_steps):
        st.step(i)
    torch.cuda.synchronize()
    prof = np.zeros(4)
    for lay in st.layers:
        prof += lay.profile_read()
        lay.profile(False)
    launches = max(prof[3], 1)
    route_us, gateup_us, down_us = (1e3 * prof[i] / launches for i in range(3))
    routes = M * w.top_k
    gateup_flop = 2.0 * routes * 2 * w.inter * w.hidden
    down_flop = 2.0 * routes * w.hidden * w.inter
    pk, pk_src = peaks()
    # the GEMMs are event-timed inside a step of a few ms: the burst figure is the denominator
    bf16 = pk.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"])
    bf16_sus = pk.get("bf16_tflops_sustained", bf16)
    peak = bf16 * FP8_OVER_BF16
    achieved = gateup_flop / (gateup_us * 1e-6) / 1e12
    mma_probe = mma_probe_tflops(moe, torch)

    # e2e: the step's activations copied in from pinned host memory and the outputs read back, every step
    x_host = torch.empty(st.x_all.shape[1:], dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(st.x_all[0].cpu())
    out_host = torch.empty(st.out.shape, dtype=st.out.dtype, pin_memory=True)
    for i in range(args.warmup):
        st.x_all[0].copy_(x_host, non_blocking=True)
        st.step(0)
        out_host.copy_(st.out, non_blocking=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        st.x_all[0].copy_(x_host, non_blocking=True)
        st.step(0)
        out_host.copy_(st.out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = e0.elapsed_time(e1)
    e2e = {"value": args.steps * M / (t_e2e / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": int(x_host.numel() * 2), "d2h_bytes_per_step": int(out_host.numel() * out_host.element_size())}
    step_s = t_ms / args.steps * 1e-3
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8*mxfp4->f32", "data": "synthetic",
        "config": {"workload": w.name, "phase": "prefill", "layers": L, "hidden": w.hidden, "inter": w.inter,
                   "experts": w.experts, "top_k": w.top_k, "tokens_per_step": M, "parallelism": f"replicas{world}",
                   "weights": "mxfp4 experts (whole bank staged on the device), fp32 router, fp32 accumulation",
                   "l2": "inputs larger than L2: each step reads %.2f GB of expert weights and %.2f GB of activations"
                         % (L * w.experts * w.expert_bytes / 1e9, L * M * w.hidden * 2 / 1e9),
                   "tensor_tflops_step": L * (gateup_flop + down_flop) / step_s / 1e12,
                   "kernel_us": {"route": route_us, "gateup_gemm": gateup_us, "down_gemm": down_us}},
        "roofline": {"bound": "tensor", "kernel": "prefill_gemm_kernel<1> (gate/up)", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "flop_per_launch": gateup_flop, "avg_launch_us": gateup_us,
                     "peak_source": ("measured bf16_tflops burst (MEASURED_PEAKS.json)" if pk_src == "measured"
                                     else "fallback 1.9 PFLOP/s bf16") + " x 2 (nominal 8-bit / bf16 ratio)",
                     "frac_of_sustained_x2": achieved / (bf16_sus * FP8_OVER_BF16),
                     "mma_probe_tflops": mma_probe, "frac_of_mma_probe": achieved / mma_probe,
                     "mma_probe": "moe_debug_mma_peak: one CTA per SM issuing the GEMM's M=128 N=256 K=32 "
                                  "block-scaled MMAs from operands resident in shared memory, event-timed",
                     "down": {"flop_per_launch": down_flop, "avg_launch_us": down_us,
                              "achieved": down_flop / (down_us * 1e-6) / 1e12,
                              "frac": down_flop / (down_us * 1e-6) / 1e12 / peak}},
        "clocks": clocks,
        "gpu_launches": int(args.steps * L * 6),
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_prefill_baseline(w)
    st.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def mma_probe_tflops(moe, torch, iters=4096, reps=5):
    """Median rate of the block-scaled MMA probe over `reps` event-timed launches (after one warm-up)."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    moe.mma_peak(iters, err.data_ptr(), stream)
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        moe.mma_peak(iters, err.data_ptr(), stream)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if int(err.item()) != 0:
        raise RuntimeError("the MMA probe's completion wait ran out")
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return moe.mma_peak_flops(iters, sms) / (sorted(times)[reps // 2] * 1e-3) / 1e12


def oracle_prefill_seconds(w, n_tokens, seed=0):
    """The oracle, as it stands, on one host core: seconds for n_tokens prompt tokens through one layer."""
    import oracle
    from expert_offload_moe_gb300 import synth

    oracle.build()
    Wr = synth.router_weights(seed, 0, w.experts, w.hidden)
    b = synth.router_bias(seed, 0, w.experts, w.bias_tau)
    ex = synth.expert_records(seed, 0, w.experts, w.hidden, w.inter)
    x = synth.activations(seed, 0, 0, n_tokens, w.hidden)
    t0 = time.perf_counter()
    ids, wt = oracle.topk_softmax(oracle.router_logits(x, Wr, b), w.top_k)
    for t in range(n_tokens):
        for j in range(w.top_k):
            oracle.expert_ffn_mxfp8(ex[ids[t][j]], w.hidden, w.inter, x[t])
    return time.perf_counter() - t0


def cpu_prefill_baseline(w, n_tokens=4):
    t = oracle_prefill_seconds(w, n_tokens)
    return {"value": n_tokens / (t * w.layers), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_tokens} prompt tokens through 1 of {w.layers} layers (single-threaded C oracle, "
                      f"{t:.1f} s), time scaled to the {w.layers}-layer stack"}


COLD_METRIC = "MoE-layer decode tokens/s (M=1), cold routes computed on the host cores"


def run_cold_host(args):
    """Decode where every route is computed: hot routes on the GPU, cold ones on the host cores meanwhile
    (route, forward_slots, forward_cold per layer; the host thread blocks in forward_cold)."""
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from expert_offload_moe_gb300 import build as moe_build
    from expert_offload_moe_gb300 import moe, stack, synth

    moe_build.build()
    moe.lib()
    w = synth.WORKLOADS[args.workload]
    M = w.tokens[0]
    n_inputs = 16
    st = stack.DecodeStack(w, M=M, n_layers=args.layers, seed=rank, n_inputs=n_inputs, out_f32=True)
    L = st.L
    stream = torch.cuda.current_stream()
    n_cold = []

    def step(i, record=False):
        st.load_inputs(i)
        for l, lay in enumerate(st.layers):
            res = lay.route(st.x_cur[l], M)
            lay.forward_slots(st.x_cur[l], st.out[l], M)
            lay.forward_cold(st.x_cur[l], st.out[l], M)
            if record:
                n_cold.append(int(stack.host_counts(res)[1]))

    for i in range(args.warmup):
        step(i, record=i == 0)
    torch.cuda.synchronize()
    clk = Clocks(local)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    t_ms = e0.elapsed_time(e1)
    value = args.steps * M / (t_ms / 1e3)
    cold_flop_step = float(np.mean(n_cold)) * 2 * 3 * w.hidden * w.inter * L
    line = {
        "metric": COLD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp4*e4m3->f32 (GPU), mxfp4*bf16->f32 (host)", "data": "synthetic",
        "config": {"workload": w.name, "layers": L, "hidden": w.hidden, "inter": w.inter, "experts": w.experts,
                   "top_k": w.top_k, "slots": w.slots, "tokens_per_step": M, "host_threads": os.cpu_count(),
                   "mean_cold_routes_per_layer": float(np.mean(n_cold)),
                   "host_gflops": cold_flop_step / (t_ms / args.steps * 1e-3) / 1e9,
                   "timing": "eager launches; the host thread computes each layer's cold routes between them"},
        "roofline": None,
        "clocks": clocks,
        "gpu_launches": int(args.steps * L * 4),
        "e2e": None,
    }
    st.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


SWEEP = [("LFU", "freq", 1.0), ("LFRU decay 0.9", "freq", 0.9), ("LFRU decay 0.7", "freq", 0.7),
         ("LRU", "lru", 1.0), ("FIFO", "fifo", 1.0), ("SLRU", "slru", 1.0)]


def run_policy_sweep(args):
    """The decode phase of the prefill-then-decode workload under each slot policy: every layer routes,
    computes its hot routes and updates its slots each step while the routing drifts between two
    popularity orders.  Reports the share of routes that found their expert in a slot, the refills and
    the decode rate with the cache updates (eager launches, one host decision per layer and step)."""
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from expert_offload_moe_gb300 import build as moe_build
    from expert_offload_moe_gb300 import moe, stack, synth

    moe_build.build()
    moe.lib()
    w = synth.WORKLOADS[args.workload]
    L = w.layers if args.layers is None else args.layers
    steps = w.steps
    inputs = [stack.LayerInputs(w, l) for l in range(L)]
    codes = {"freq": moe.MOE_POLICY_FREQ, "lru": moe.MOE_POLICY_LRU, "fifo": moe.MOE_POLICY_FIFO,
             "slru": moe.MOE_POLICY_SLRU}
    x = torch.empty((L, 1, w.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((L, 1, w.hidden), dtype=torch.bfloat16, device="cuda")
    biases = [[torch.from_numpy(synth.drifting_bias(0, l, w.experts, w.bias_tau, t, steps)).cuda()
               for t in range(steps)] for l in range(L)]
    xs = torch.from_numpy(np.stack([np.stack([synth.activations(0, l, 2000 + t, 1, w.hidden)[0] for l in range(L)])
                                    for t in range(steps)]).view(np.int16)).view(torch.bfloat16).cuda()
    rows = []
    for name, pol, decay in SWEEP:
        layers = [li.make_layer(max_tokens=8, max_refills=2, score_decay=decay) for li in inputs]
        for lay in layers:
            lay.set_policy(codes[pol])
        hot = cold = refills = 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for t in range(steps):
            x.copy_(xs[t].unsqueeze(1))
            for l, lay in enumerate(layers):
                lay.set_bias(biases[l][t])
                res = lay.route(x[l], 1)
                lay.forward_slots(x[l], out[l], 1)
                refills += lay.cache_update()
                c = stack.host_counts(res)  # cache_update waited for the route's mirror
                hot += int(c[0])
                cold += int(c[1])
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        for lay in layers:
            lay.close()
        rows.append({"policy": name, "hit_rate": hot / max(hot + cold, 1),
                     "refills_per_layer_step": refills / (L * steps),
                     "refill_gb": refills * w.expert_bytes / 1e9, "tokens_per_s": steps / dt})
    rows += device_table_rows(w, L, steps, inputs, xs, biases)
    fate = fate_rows(w, L, steps, inputs, biases)
    best = max(rows, key=lambda r: r["hit_rate"])
    line = {
        "metric": "slot-cache hot-route hit rate, decode with drifting routing (LFU)", "value": rows[0]["hit_rate"],
        "unit": "fraction of routes", "n_gpus": world, "steps": steps, "warmup": 0, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4*e4m3->f32", "data": "synthetic",
        "config": {"workload": w.name, "layers": L, "experts": w.experts, "top_k": w.top_k, "slots": w.slots,
                   "max_refills_per_step": 2, "drift": "bias from popularity order A to order B over the steps",
                   "sweep": rows, "best": best["policy"], "next_layer_prefetch": fate,
                   "timing": "wall clock, eager launches, one host policy decision per layer and step"},
        "roofline": None, "clocks": None, "gpu_launches": int(len(SWEEP) * steps * L * 3), "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


FATE_RHO = 0.9  # correlation of consecutive layers' inputs in the residual-stream stand-in


def fate_rows(w, L, steps, inputs, biases):
    """LFU with and without next-layer prefetch (tinyserve README "How it works" 4, FATE) on inputs whose layers
    are correlated like a residual stream (x_l = rho x_(l-1) + sqrt(1 - rho^2) e_l): after layer l's kernels are
    issued and its slots updated, layer l + 1 predicts its experts from x_l and copies the missing ones in."""
    import numpy as np
    import torch

    from expert_offload_moe_gb300 import stack, synth

    xs = torch.from_numpy(np.stack([synth.activations_residual(0, t, L, 1, w.hidden, FATE_RHO)
                                    for t in range(steps)]).view(np.int16)).view(torch.bfloat16).cuda()
    x = torch.empty((L, 1, w.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((L, 1, w.hidden), dtype=torch.bfloat16, device="cuda")
    rows = []
    for prefetch in (False, True):
        layers = [li.make_layer(max_tokens=8, max_refills=2) for li in inputs]
        hot = cold = refills = fetched = 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for t in range(steps):
            x.copy_(xs[t])
            for l, lay in enumerate(layers):
                lay.set_bias(biases[l][t])
                res = lay.route(x[l], 1)
                lay.forward_slots(x[l], out[l], 1)
                refills += lay.cache_update()
                c = stack.host_counts(res)
                hot += int(c[0])
                cold += int(c[1])
                if prefetch and l + 1 < L:
                    fetched += layers[l + 1].prefetch(x[l], 1)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        for lay in layers:
            lay.close()
        rows.append({"policy": "LFU + next-layer prefetch" if prefetch else "LFU", "inputs": f"residual rho={FATE_RHO}",
                     "hit_rate": hot / max(hot + cold, 1), "refills_per_layer_step": refills / (L * steps),
                     "prefetches_per_layer_step": fetched / (L * steps),
                     "copy_gb": (refills + fetched) * w.expert_bytes / 1e9, "tokens_per_s": steps / dt})
    return rows


def device_table_rows(w, L, steps, inputs, xs, biases):
    """The same decode phase with the slot table on the GPU (xinfer docs "How it works", Decode): every
    miss is filled in its own step, so every route is computed from a slot.  Timed twice: eager launches
    like the host policies, and as one CUDA graph per step (route with the table step, fill, gate/up and
    down of every layer; no host decision left)."""
    import numpy as np
    import torch

    from expert_offload_moe_gb300 import stack

    rows = []
    for mode in ("eager", "graph"):
        layers = [li.make_layer(max_tokens=8) for li in inputs]
        for lay in layers:
            lay.set_device_cache(True)
        x = torch.empty((L, 1, w.hidden), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((L, 1, w.hidden), dtype=torch.bfloat16, device="cuda")
        bias = torch.empty((L, w.experts), dtype=torch.float32, device="cuda")
        bias_all = torch.stack([torch.stack([biases[l][t] for l in range(L)]) for t in range(steps)])
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def body():
            for l, lay in enumerate(layers):
                lay.set_bias(bias[l], s)
                lay.route(x[l], 1, s)
                lay.forward_slots(x[l], out[l], 1, s)

        g = None
        if mode == "graph":
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                body()
            for lay in layers:  # capture ran nothing; start the counters from the same state as eager
                lay.set_device_cache(False)
                lay.set_device_cache(True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(s):
            for t in range(steps):
                x.copy_(xs[t].unsqueeze(1))
                bias.copy_(bias_all[t])
                if g is None:
                    body()
                else:
                    g.replay()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        st = np.sum([lay.device_cache_stats() for lay in layers], axis=0)
        for lay in layers:
            lay.close()
        routes = L * steps * w.top_k
        rows.append({"policy": f"device LRU, demand fill ({mode})", "hit_rate": float(st[2]) / routes,
                     "refills_per_layer_step": float(st[1]) / (L * steps),
                     "refill_gb": float(st[1]) * w.expert_bytes / 1e9, "tokens_per_s": steps / dt,
                     "routes_computed": "all (misses filled in the step)"})
    return rows


def main():
    args = parse()
    if args.policy_sweep:
        run_policy_sweep(args)
        return
    prefill = synth_workload(args.workload).prefill_tokens > 0
    if args.impl == "reference":
        run_reference(args, prefill)
    elif prefill:
        run_prefill(args)
    elif args.cold_on_host:
        run_cold_host(args)
    else:
        run_ours(args)


def synth_workload(name):
    from expert_offload_moe_gb300 import synth

    return synth.WORKLOADS[name]


if __name__ == "__main__":
    main()
