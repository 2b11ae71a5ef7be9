#!/usr/bin/env python3
"""Benchmark: one GLM-5.2-shaped MoE layer (Route -> Union -> int4 SwiGLU expert
FFN -> combine -> Learn) on GB300, tokens/s and int4 expert-weight GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode] [--impl ours|reference]

A step is one pass of the whole layer over one batch (T tokens) of synthetic
input.  The default workload is the T = 1 decode layer (E = 256 routed + 1
shared expert, k = 8, d = 6144, f = 2048, int4 group-32 weights with fp32
scales).  Every step reads its weights from one of R device-resident copies of
the layer, rotated, so the bytes of consecutive steps never share L2 (each
copy is 6.06 GB; the L2 is 129 MB).  Steps are captured into CUDA graphs with
CUDA events between the stages; the events of the last replay give the stage
durations used for the roofline line.

Multi-GPU: one process per GPU (torchrun); every rank runs the same layer on
its own tokens with no collective in the data path (tokens are independent:
weak scaling); the barrier and a MAX reduction of the elapsed time are the only
communication.  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (decode & prefill); int4 expert weight GB/s vs HBM peak"
UNIT = "tokens/s"


# ------------------------------------------------------------------ helpers --

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "batched_decode", "prefill", "stack", "tier", "tiny"],
                    help="tiny is the parity-size layer (fits in L2; for quick checks, not a bench line); "
                         "stack is 8 resident layers, the line's T from --tokens (default 64) plus a sweep "
                         "over T in {1, 4, 16, 64, 256}; tier is the decode layer with its experts in host "
                         "memory and a sweep over the fraction cached in HBM")
    ap.add_argument("--replicas", type=int, default=4, help="device copies of the layer rotated across steps")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the routed expert count (small-footprint profiling runs); 0 = workload's")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the tokens per step (small-footprint profiling runs); 0 = workload's")
    ap.add_argument("--mode", choices=["workload", "decode", "prefill", "hybrid"], default="workload",
                    help="FFN path: the workload's own (prefill for prefill, the library's automatic choice "
                         "for the stack, decode otherwise) or forced")
    ap.add_argument("--graph-steps", type=int, default=100, help="steps captured per CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="decode line only (by default it also carries the batched-decode layer on the decode "
                         "and on the hybrid path, the prefill layer, the stack and the expert tier under "
                         "\"workloads\")")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the CPU-baseline sample")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running (read-only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": float(max(power))}


def gpu_uuid(torch, dev: int) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# --------------------------------------------------------------- workloads --

def layer_bytes(sh, n_uniq: int) -> dict:
    """Algorithmic bytes of one layer step (each byte the definition must touch once)."""
    import workloads
    blk = workloads.expert_q_bytes(sh.d, sh.f) + 4 * workloads.expert_s_count(sh.d, sh.f, sh.G)
    ffn = (n_uniq + 1) * blk
    nib = (n_uniq + 1) * workloads.expert_q_bytes(sh.d, sh.f)
    router = sh.E * sh.d * 4 + sh.E * 4
    act = 2 * sh.T * sh.d * 4
    return {"ffn": ffn, "nibbles": nib, "layer": ffn + router + act, "expert_block": blk}


# ------------------------------------------------------------------ our arm --

def init_device(local, world):
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        try:
            dist.init_process_group("nccl", device_id=dev)
        except TypeError:
            dist.init_process_group("nccl")
    from int4_routed_expert_sigmoid_gb300 import build as libbuild
    libbuild.build()
    return dev


class LayerCopies:
    """R device copies of one seeded GLM-5.2-shaped layer (routed experts + shared expert, router
    weights), rotated across steps so that consecutive steps never find their weights in L2.  The
    decode, batched-decode and prefill workloads share layer 0's weights; only the selection bias
    (per workload) differs."""

    def __init__(self, sh, R, dev):
        import torch

        import int4_routed_expert_sigmoid_gb300 as moe
        import workloads
        E, d, f, G = sh.E, sh.d, sh.f, sh.G
        L = workloads.layer_inputs(sh, seed=0, threads=os.cpu_count() or 8)
        qb, sc = workloads.expert_q_bytes(d, f), workloads.expert_s_count(d, f, G)
        self.q_all = torch.empty((R, E * qb + qb), dtype=torch.uint8, device=dev)
        self.s_all = torch.empty((R, E * sc + sc), dtype=torch.float32, device=dev)
        self.q_all[0, :E * qb].copy_(torch.from_numpy(L.q_base.reshape(-1)))
        self.q_all[0, E * qb:].copy_(torch.from_numpy(L.shared_q))
        self.s_all[0, :E * sc].copy_(torch.from_numpy(L.s_base.reshape(-1)))
        self.s_all[0, E * sc:].copy_(torch.from_numpy(L.shared_s))
        wg0 = torch.from_numpy(L.wg).to(dev)
        for r in range(1, R):
            self.q_all[r].copy_(self.q_all[0])
            self.s_all[r].copy_(self.s_all[0])
        self.wgs = [wg0] + [wg0.clone() for _ in range(R - 1)]
        self.layers = [moe.LayerWeights(self.q_all[r, :E * qb], self.s_all[r, :E * sc], self.q_all[r, E * qb:],
                                        self.s_all[r, E * sc:], E=E, d=d, f=f, G=G) for r in range(R)]
        self.R, self.E, self.d, self.f, self.G = R, E, d, f, G
        self.block_bytes = qb + 4 * sc
        del L


def measure_layer(copies, sh, path, steps, warmup, graph_steps, e2e_steps, rank, world, dev):
    """One workload of the single-layer benchmark: `steps` timed steps of moe_layer_forward over T
    tokens (CUDA graphs of S steps), stage durations from a second graph with events between the
    stage calls, and an end-to-end run with host buffers.  Returns the workload's measurements."""
    import torch

    import int4_routed_expert_sigmoid_gb300 as moe
    import workloads
    T, E, k, d, f = sh.T, sh.E, sh.k, sh.d, sh.f
    mode = {"decode": moe.MOE_MODE_DECODE, "prefill": moe.MOE_MODE_PREFILL, "hybrid": moe.MOE_MODE_HYBRID}[path]
    prefill = path == "prefill"
    R = copies.R
    S = max(1, min(graph_steps, steps))
    bias0 = workloads.selection_bias(E, sh.bias, seed=0)
    biases = [None if bias0 is None else torch.from_numpy(bias0).to(dev) for _ in range(R)]
    wgs, layers = copies.wgs, copies.layers
    # distinct tokens per captured step position, seeded per rank
    xs = torch.from_numpy(workloads.activations(S * T, d, seed=1000 + rank)).to(dev).view(S, T, d)

    # ---- step buffers (serial on one stream: one set suffices)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    un = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
              offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
              perm=torch.empty(T * k, dtype=torch.int32, device=dev),
              sorted_pair=torch.empty(T * k, dtype=torch.int32, device=dev),
              uniq=torch.empty(E, dtype=torch.int32, device=dev),
              n_uniq=torch.empty(1, dtype=torch.int32, device=dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    hits = torch.zeros((R, E), dtype=torch.int64, device=dev)
    y_pair = torch.empty((T * k, d), dtype=torch.float32, device=dev)
    y_shared = torch.empty((T, d), dtype=torch.float32, device=dev)
    outs = torch.empty((S, T, d), dtype=torch.float32, device=dev)
    ws = moe.workspace(moe.ffn_workspace_bytes(T, k, d, f, mode), dev)
    lws_step = moe.workspace(moe.layer_workspace_bytes(T, k, E, d, f, mode), dev)

    def layer_step(i):
        """One step through the public fused entry point (the timed path)."""
        r = i % R
        moe.moe_layer_forward(xs[i % S], wgs[r], biases[r], layers[r], k, 1, 1.0, mode=mode,
                              out=outs[i % S], topk_idx=idx, topk_w=wts, hits=hits[r], ws=lws_step, err=err)

    def step(i, ev=None):
        """The same step through the separate stage calls, with events between stages."""
        r = i % R
        x = xs[i % S]
        if ev:
            ev[0].record()
        moe.moe_route(x, wgs[r], biases[r], k, 1, 1.0, topk_idx=idx, topk_w=wts, logits=logits)
        if ev:
            ev[1].record()
        moe.moe_union(idx, E, hits=hits[r], err=err, out=un)
        if ev:
            ev[2].record()
        moe.moe_expert_ffn_int4(x, layers[r], un, k, mode, y_pair=y_pair, y_shared=y_shared,
                                ws=ws, err=err)
        if ev:
            ev[3].record()
        moe.moe_combine(y_pair, y_shared, wts, un["perm"], out=outs[i % S])
        if ev:
            ev[4].record()

    # kernels per fused step: small batches logits(+x fragments), select+union, gate/up, down,
    # combine; otherwise logits, top-k, union, x fragments, gate/up, down, combine
    if prefill:   # logits, top-k, union, pair positions, token rows, gate/up, h conversion, down, combine
        launches_per_step = 9
    elif path == "hybrid":   # logits, top-k, union, split, x fragments, decode gate/up + down, the prefill
        launches_per_step = 13   # path's pair positions, token rows, gate/up, h conversion, down; combine
    else:
        launches_per_step = 5 if (T <= 8 and T * k <= 64) else 7

    # warm the code paths once outside capture, then capture
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(min(S, 2 * R)):
            step(i)
            layer_step(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    def capture(n, with_events):
        g = torch.cuda.CUDAGraph()
        # external events become event-record nodes of the graph (timestamps of each replay)
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)] for _ in range(n)] \
            if with_events else None
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            for i in range(n):
                if with_events:
                    step(i, evs[i])
                else:
                    layer_step(i)
        return g, evs

    g_main, _ = capture(S, False)
    g_stages, evs = capture(S, True)
    tail = steps % S
    g_tail = capture(tail, False)[0] if tail else None
    n_main = steps // S

    # ---- warm-up (untimed)
    for _ in range(max(1, -(-warmup // S))):
        g_main.replay()
    torch.cuda.synchronize()
    err.zero_()

    sampler = ClockSampler(gpu_uuid(torch, dev.index))
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(n_main):
        g_main.replay()
    if g_tail is not None:
        g_tail.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    elapsed_ms = t0.elapsed_time(t1)
    dev_err = int(err.item())

    # stage durations: the same S steps through the separate stage calls, replayed right after the
    # timed region (events between stages; the fused path has no stage boundaries to time)
    g_stages.replay()
    g_stages.replay()
    torch.cuda.synchronize()
    st = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(4)] for i in range(S)])
    stage_ms = st.mean(axis=0)
    n_uniq = int(un["n_uniq"].item())

    # the FFN call on its own, S calls back to back in one graph (the last step's routing, weights
    # rotated over the R copies), events only around the batch: the average is the FFN stage's
    # launch duration in a stream of FFN calls (the per-stage events above also hold each stage's
    # launch gap)
    g_ffn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ffn, capture_error_mode="thread_local"):
        for i in range(S):
            moe.moe_expert_ffn_int4(xs[i % S], layers[i % R], un, k, mode, y_pair=y_pair, y_shared=y_shared,
                                    ws=ws, err=err)
    g_ffn.replay()
    g_ffn.replay()
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record()
    for _ in range(3):
        g_ffn.replay()
    f1.record()
    torch.cuda.synchronize()
    ffn_call_ms = f0.elapsed_time(f1) / (3 * S)

    # ---- end to end through the C-ABI call with host buffers (moe_layer_forward_host: the step's
    # token rows copied in from page-locked memory, the layer, the result copied back; not
    # graph-captured, one call per step from the host)
    e2e_steps = max(1, min(e2e_steps, steps))
    x_host = torch.from_numpy(workloads.activations(e2e_steps * T, d, seed=5000 + rank)).view(e2e_steps, T, d)
    x_host = x_host.pin_memory()
    out_host = torch.empty((e2e_steps, T, d), dtype=torch.float32).pin_memory()
    hws = moe.workspace(moe.layer_host_workspace_bytes(T, k, E, d, f, mode), dev)
    for i in range(min(50, e2e_steps)):   # warm-up of the host path
        r = i % R
        moe.moe_layer_forward_host(x_host[i], wgs[r], biases[r], layers[r], k, mode=mode, out_host=out_host[i],
                                   ws=hws, err=err)
    torch.cuda.synchronize()
    barrier(world)
    w0 = time.perf_counter()
    for i in range(e2e_steps):
        r = i % R
        moe.moe_layer_forward_host(x_host[i], wgs[r], biases[r], layers[r], k, mode=mode, out_host=out_host[i],
                                   hits=hits[r], ws=hws, err=err)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - w0
    barrier(world)
    dev_err |= int(err.item())

    elapsed_max, e2e_max = reduce_max(world, [elapsed_ms, e2e_s], dev)
    peaks = load_peaks()
    byts = layer_bytes(sh, n_uniq)
    ffn_ms = ffn_call_ms
    if prefill:
        # dense work of the grouped GEMMs: 3 matrices of d x f per (token, expert) pair, 2 flops per MAC
        flops = 6.0 * d * f * (T * k + T)
        achieved = flops / (ffn_ms * 1e-3) / 1e12
        roof = {"kernel": "expert FFN call (pair positions + token rows, tcgen05 gate/up, h conversion, "
                          "tcgen05 down), timed over back-to-back calls",
                "bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": ncu_traffic(ROOT, "ffn_prefill"),
                "peak_source": peaks["source"] + " bf16 dense burst (fp16 operands run at the same tensor rate)",
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "flops_per_launch": flops, "ms_per_launch": round(ffn_ms, 5)}
    else:
        achieved = byts["ffn"] / (ffn_ms * 1e-3) / 1e9
        roof = {"kernel": ("expert FFN call (act fragments + gate/up + down kernels), timed over back-to-back calls"
                           if path == "decode" else
                           "hybrid expert FFN call (split, decode half, prefill half with the shared expert), timed "
                           "over back-to-back calls; bytes = the union's expert blocks"),
                "bound": "hbm",
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": ncu_traffic(ROOT, "ffn" if T == 1 else f"ffn_T{T}") if path == "decode" else None,
                "peak_source": peaks["source"], "bytes_per_launch": byts["ffn"], "ms_per_launch": round(ffn_ms, 5)}
    ms_per_step = elapsed_max / steps
    return {
        "value": round(job_throughput(T, steps, world, elapsed_max), 2), "unit": UNIT, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms_per_step, 6),
        "config": {"workload": f"{sh.name}: 1 MoE layer, E={E} routed + 1 shared, k={k}, d={d}, f={f}, "
                               f"int4 group-{sh.G} fp32 scales, T={T} token(s) per step, selection bias "
                               f"{sh.bias}, FFN path {path}",
                   "T": T, "E": E, "k": k, "d": d, "f": f, "G": sh.G, "weights": "int4",
                   "l2": (f"inputs larger than L2: {R} device copies of the layer "
                          f"({R * E * byts['expert_block'] / 1e9:.1f} GB) rotated across steps")
                   if R * E * byts["expert_block"] > 2 * 129e6 else "parity-size layer: fits in L2 (not a bench line)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "cuda_graph_steps": S},
        "roofline": roof,
        "stages_ms": {"route": round(float(stage_ms[0]), 5), "union": round(float(stage_ms[1]), 5),
                      "ffn": round(float(stage_ms[2]), 5), "combine": round(float(stage_ms[3]), 5),
                      "ffn_back_to_back": round(ffn_ms, 5)},
        "layer_gbs": round(byts["layer"] / (ms_per_step * 1e-3) / 1e9, 1),
        "nibble_gbs": round(byts["nibbles"] / (ms_per_step * 1e-3) / 1e9, 1),
        "n_uniq": n_uniq,
        "e2e": {"value": round(T * e2e_steps * world / e2e_max, 2), "unit": UNIT,
                "h2d_bytes_per_step": T * d * 4, "d2h_bytes_per_step": T * d * 4, "steps": e2e_steps,
                "call": "moe_layer_forward_host (page-locked host rows in and out, read and written by the "
                        "kernels over the host link; one call per step)"},
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks,
        "device_error": dev_err,
    }


def measure_tier(args, rank, world, dev, fractions=(1.0, 0.5, 0.25, 0.125), steps=200, warmup=200):
    """The decode T = 1 layer with its routed experts in page-locked host memory (Grace memory behind
    NVLink-C2C) and an HBM cache of a fraction of them (moe_layer_forward_tier: Place and Overlap).
    Per fraction: tokens/s, the share of union experts found resident, and the host -> device
    bytes copied per second.  Each call waits on the host for its routing, so the loop is host
    driven (no CUDA graph); the timed region is bracketed by synchronisations."""
    import torch

    import int4_routed_expert_sigmoid_gb300 as moe
    import workloads
    sh = workloads.WORKLOADS["decode"]
    E, k, d, f, G, T = sh.E, sh.k, sh.d, sh.f, sh.G, sh.T
    qb, sc = workloads.expert_q_bytes(d, f), workloads.expert_s_count(d, f, G)
    hq = torch.empty(E * qb, dtype=torch.uint8).pin_memory()
    hs = torch.empty(E * sc, dtype=torch.float32).pin_memory()
    L = workloads.layer_inputs(sh, seed=0, threads=os.cpu_count() or 8, q_base=hq.numpy(), s_base=hs.numpy())
    wg = torch.from_numpy(L.wg).to(dev)
    bias = torch.from_numpy(L.bias).to(dev)
    shq = torch.from_numpy(L.shared_q).to(dev)
    shs = torch.from_numpy(L.shared_s).to(dev)
    del L
    n_x = steps + warmup   # every call a new token: a repeated token would find its experts resident
    xs = torch.from_numpy(workloads.activations(n_x * T, d, seed=3000 + rank)).to(dev).view(n_x, T, d)
    out = torch.empty((T, d), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = moe.workspace(moe.tier_workspace_bytes(T, k, E, d, f, moe.MOE_MODE_DECODE), dev)
    copy = torch.cuda.Stream(device=dev)
    blk = qb + 4 * sc
    rows = []
    for frac in fractions:
        n_slots = max(k, int(round(frac * E)))
        tier = moe.ExpertTier(hq, hs, E=E, d=d, f=f, n_slots=n_slots, G=G, device=dev)
        if n_slots == E:
            tier.prefetch(np.arange(E), copy_stream=copy)   # every expert in HBM: the device-only path

        def call(i):
            moe.moe_layer_forward_tier(xs[i % n_x], wg, bias, tier, shq, shs, k, mode=moe.MOE_MODE_DECODE,
                                       out=out, ws=ws, err=err, copy_stream=copy)

        for i in range(warmup):
            call(i)
        torch.cuda.synchronize()
        err.zero_()
        st0 = tier.stats()
        barrier(world)
        t0 = time.perf_counter()
        for i in range(steps):
            call(warmup + i)
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
        el = reduce_max(world, [el], dev)[0]
        st1 = tier.stats()
        hits, miss = st1["hits"] - st0["hits"], st1["misses"] - st0["misses"]
        copied = st1["bytes_copied"] - st0["bytes_copied"]
        rows.append({"fraction_resident": frac, "n_slots": n_slots, "steps": steps,
                     "tokens_per_s": round(T * steps * world / el, 2), "ms_per_step": round(el / steps * 1e3, 4),
                     # every expert in HBM: the calls take the device-only path and count no hits
                     "hit_rate": round(hits / (hits + miss), 4) if hits + miss else None,
                     "path": "device-only (all experts resident)" if n_slots == E else "host-planned",
                     "c2c_gbs": round(copied / el / 1e9, 2), "copied_bytes_per_step": int(copied / steps),
                     "expert_block_bytes": blk, "device_error": int(err.item())})
        tier.close()
        del tier
        torch.cuda.synchronize()
    return {"config": {"workload": f"decode T={T} with routed experts in page-locked host memory (Grace, "
                                   f"NVLink-C2C) and an HBM cache of a fraction of them; E={E} + 1 shared, k={k}, "
                                   f"d={d}, f={f}, int4 group-{G}, N(0, 0.1) selection bias, LRU slots, no pins",
                       "T": T, "E": E, "k": k, "d": d, "f": f, "G": G},
            "fractions": rows}


def workload_shape(args, name):
    import dataclasses

    import workloads
    sh = workloads.WORKLOADS[name]
    if args.experts or args.tokens:
        sh = dataclasses.replace(sh, E=args.experts or sh.E, T=args.tokens or sh.T)
    return sh


def path_for(args, name):
    """FFN path of a single-layer workload: its own (prefill for prefill, decode otherwise) or forced."""
    if args.mode == "workload":
        return "prefill" if name == "prefill" else "decode"
    return args.mode


# steps of the secondary workloads carried in the default line (their own counts, a few seconds each)
EXTRA_STEPS = {"prefill": 40, "batched_decode": 200}


def run_ours(args, rank, world, local):
    """The single-layer workloads.  The default (decode T = 1) line also carries, under "workloads",
    the batched-decode T = 64 layer (on the decode path and on the opt-in hybrid path) and the prefill
    T = 4096 layer on the same weights, the 8-layer stack sweep and the expert tier, each with its own
    steps, roofline, stage times, union size and clocks."""
    import torch
    dev = init_device(local, world)
    sh = workload_shape(args, args.workload)
    path = path_for(args, args.workload)
    prefill = path == "prefill"
    R = max(1, min(args.replicas, 2) if prefill else args.replicas)
    copies = LayerCopies(sh, R, dev)
    res = measure_layer(copies, sh, path, args.steps, args.warmup,
                        args.graph_steps if not prefill else 4, 8 if prefill else args.e2e_steps, rank, world, dev)
    line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic"}
    for key in ("config", "roofline", "stages_ms", "layer_gbs", "nibble_gbs", "n_uniq", "e2e", "gpu_launches",
                "clocks", "device_error"):
        line[key] = res[key]
    extras = {}
    if args.workload == "decode" and not args.no_workloads and not (args.experts or args.tokens):
        # the other single-layer workloads on the same weights, then the stack on its own 8 layers
        # (batched_decode_hybrid: the same batch on the opt-in hybrid path, MOE_MODE_HYBRID, which gives
        # the tensor-core path's precision to the experts with more than 8 of its tokens)
        for name, wl, path_x in (("batched_decode", "batched_decode", path_for(args, "batched_decode")),
                                 ("batched_decode_hybrid", "batched_decode", "hybrid"),
                                 ("prefill", "prefill", path_for(args, "prefill"))):
            sh_x = workload_shape(args, wl)
            pf = path_x == "prefill"
            extras[name] = measure_layer(copies, sh_x, path_x, EXTRA_STEPS[wl], max(3, args.warmup),
                                         4 if pf else args.graph_steps, 8 if pf else 200, rank, world, dev)
            line["gpu_launches"] += extras[name]["gpu_launches"]
        del copies
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        extras["stack"] = measure_stack(args, rank, world, dev, T_line=64, steps=48, warmup=max(3, args.warmup),
                                        sweep_seconds=1.0)
        line["gpu_launches"] += extras["stack"]["gpu_launches"]
        extras["tier"] = measure_tier(args, rank, world, dev)
        line["workloads"] = extras
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sh, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------- layer stack --

def measure_stack(args, rank, world, dev, T_line, steps, warmup, sweep_seconds=2.0):
    """8 resident layers, out_l = x_l + MoE(RMSNorm(x_l)), each layer with its own seeded experts,
    router and Zipf selection bias (its own expert permutation).  A step is one pass of T tokens
    through all 8 layers; tokens/s = T / step time.  Times exactly `steps` steps at T_line and, under
    "sweep", every T of the stack's batch sweep, each for about `sweep_seconds`."""
    import torch

    import int4_routed_expert_sigmoid_gb300 as moe
    import workloads
    sh = workloads.WORKLOADS["stack"]
    E, k, d, f, G, NL = sh.E, sh.k, sh.d, sh.f, sh.G, sh.layers
    mode = {"workload": moe.MOE_MODE_AUTO, "decode": moe.MOE_MODE_DECODE, "prefill": moe.MOE_MODE_PREFILL,
            "hybrid": moe.MOE_MODE_HYBRID}[args.mode]   # automatic: the library picks the path by T
    eps = 1e-5

    # ---- the 8 layers, generated one at a time into one host buffer and copied to the device
    qb, sc = workloads.expert_q_bytes(d, f), workloads.expert_s_count(d, f, G)
    q_all = torch.empty((NL, E * qb + qb), dtype=torch.uint8, device=dev)
    s_all = torch.empty((NL, E * sc + sc), dtype=torch.float32, device=dev)
    q_host = np.empty((E, qb), dtype=np.uint8)
    s_host = np.empty((E, sc), dtype=np.float32)
    wgs, biases = [], []
    for l in range(NL):
        L = workloads.layer_inputs(sh, seed=0, layer=l, T=1, threads=os.cpu_count() or 8,
                                   q_base=q_host, s_base=s_host)
        q_all[l, :E * qb].copy_(torch.from_numpy(q_host.reshape(-1)))
        s_all[l, :E * sc].copy_(torch.from_numpy(s_host.reshape(-1)))
        q_all[l, E * qb:].copy_(torch.from_numpy(L.shared_q))
        s_all[l, E * sc:].copy_(torch.from_numpy(L.shared_s))
        wgs.append(torch.from_numpy(L.wg).to(dev))
        biases.append(torch.from_numpy(L.bias).to(dev))
        del L
    torch.cuda.synchronize()
    del q_host, s_host
    layers = [moe.LayerWeights(q_all[l, :E * qb], s_all[l, :E * sc], q_all[l, E * qb:], s_all[l, E * sc:],
                               E=E, d=d, f=f, G=G) for l in range(NL)]
    hits = torch.zeros((NL, E), dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    blk = workloads.expert_q_bytes(d, f) + 4 * workloads.expert_s_count(d, f, G)
    S = 8   # steps per captured graph (distinct inputs)

    def make(T):
        ctx = {"T": T}
        ctx["xs"] = torch.from_numpy(workloads.activations(S * T, d, seed=1000 + rank)).to(dev).view(S, T, d)
        ctx["acts"] = torch.empty((NL, T, d), dtype=torch.float32, device=dev)   # outputs of layers 0..6
        ctx["outs"] = torch.empty((S, T, d), dtype=torch.float32, device=dev)
        ctx["xn"] = torch.empty((2, T, d), dtype=torch.float32, device=dev)   # a layer's input, the next one's
        ctx["idx"] = torch.empty((NL, T, k), dtype=torch.int32, device=dev)
        ctx["wts"] = torch.empty((T, k), dtype=torch.float32, device=dev)
        ctx["ws"] = moe.workspace(moe.layer_workspace_bytes(T, k, E, d, f, mode), dev)
        return ctx

    def stack_step(ctx, x, out):
        # x_{l+1} = x_l + MoE(RMSNorm(x_l)): the first layer's input is normalised on its own; every
        # other layer's comes from the previous layer's combine (moe_layer_forward_norm)
        moe.moe_rms_norm(x, eps, out=ctx["xn"][0])
        for l in range(NL):
            xin = x if l == 0 else ctx["acts"][l - 1]
            xo = out if l == NL - 1 else ctx["acts"][l]
            cur, nxt = ctx["xn"][l % 2], ctx["xn"][(l + 1) % 2]
            if l < NL - 1:
                moe.moe_layer_forward_norm(cur, wgs[l], biases[l], layers[l], k, eps=eps, mode=mode, residual=xin,
                                           out=xo, out_normed=nxt, topk_idx=ctx["idx"][l], topk_w=ctx["wts"],
                                           hits=hits[l], ws=ctx["ws"], err=err)
            else:
                moe.moe_layer_forward(cur, wgs[l], biases[l], layers[l], k, 1, 1.0, mode=mode, residual=xin,
                                      out=xo, topk_idx=ctx["idx"][l], topk_w=ctx["wts"], hits=hits[l],
                                      ws=ctx["ws"], err=err)

    def graph(ctx, n):
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(S):
                stack_step(ctx, ctx["xs"][i], ctx["outs"][i])
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            for i in range(n):
                stack_step(ctx, ctx["xs"][i % S], ctx["outs"][i % S])
        return g

    def n_uniq_layers(ctx):
        idx = ctx["idx"].cpu().numpy()
        return [int(np.unique(idx[l]).size) for l in range(NL)]

    def timed(g, reps, tail_g=None):
        barrier(world)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            g.replay()
        if tail_g is not None:
            tail_g.replay()
        t1.record()
        torch.cuda.synchronize()
        barrier(world)
        return t0.elapsed_time(t1)

    peaks = load_peaks()

    def bytes_of(T, nu):
        # per layer: unique experts + shared, router weights and bias, x in, out, residual
        return sum((n + 1) * blk + E * d * 4 + E * 4 + 3 * T * d * 4 for n in nu)

    def path_of(T):
        # the FFN path and the layer's kernels (as counted in measure_layer); every layer but the last
        # also forms the next layer's normalised input, in its combine up to 64 tokens, else in one
        # more kernel
        if mode == moe.MOE_MODE_PREFILL:
            name, n = "prefill", 9
        elif mode == moe.MOE_MODE_HYBRID or (mode == moe.MOE_MODE_AUTO and T >= 128):
            name, n = "hybrid", 13
        else:
            name, n = "decode", 5 if (T <= 8 and T * k <= 64) else 7
        return name, n, (NL - 1) * (1 if T > 64 else 0)

    # ---- the batch sweep (each T timed for about sweep_seconds)
    sweep = []
    launches = 0
    for T in sh.batch_sweep:
        ctx = make(T)
        g = graph(ctx, S)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        probe = timed(g, 2) / (2 * S)
        reps = max(3, min(500, int(sweep_seconds * 1000.0 / max(probe * S, 1e-3))))
        err.zero_()
        smp = ClockSampler(gpu_uuid(torch, dev.index))
        smp.start()
        el = reduce_max(world, [timed(g, reps)], dev)[0]
        ck = smp.stop()
        nu = n_uniq_layers(ctx)
        ms = el / (reps * S)
        by = bytes_of(T, nu)
        launches += (1 + NL * path_of(T)[1] + path_of(T)[2]) * reps * S   # + the first layer's RMS norm
        sweep.append({"T": T, "steps": reps * S, "ms_per_step": round(ms, 5),
                      "tokens_per_s": round(job_throughput(T, reps * S, world, el), 2),
                      "stack_gbs": round(by / (ms * 1e-3) / 1e9, 1),
                      "frac": round(by / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                      "ffn_path": path_of(T)[0],
                      "n_uniq_per_layer": nu, "clocks": ck, "device_error": int(err.item())})
        del g, ctx
        torch.cuda.empty_cache()

    # ---- the line: exactly `steps` steps at T_line
    ctx = make(T_line)
    g_main = graph(ctx, S)
    n_main, tail = divmod(steps, S)
    g_tail = graph(ctx, tail) if tail else None
    for _ in range(max(1, -(-warmup // S))):
        g_main.replay()
    torch.cuda.synchronize()
    err.zero_()
    sampler = ClockSampler(gpu_uuid(torch, dev.index))
    sampler.start()
    time.sleep(0.3)
    elapsed = timed(g_main, n_main, g_tail)
    clocks = sampler.stop()
    dev_err = int(err.item())
    nu = n_uniq_layers(ctx)

    # ---- end to end with host buffers (not graph-captured)
    e2e_steps = max(1, min(args.e2e_steps, steps, 200))
    x_host = torch.from_numpy(workloads.activations(e2e_steps * T_line, d, seed=5000 + rank))
    x_host = x_host.view(e2e_steps, T_line, d).pin_memory()
    out_host = torch.empty((e2e_steps, T_line, d), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((T_line, d), dtype=torch.float32, device=dev)
    out_dev = torch.empty((T_line, d), dtype=torch.float32, device=dev)
    for _ in range(3):
        stack_step(ctx, x_dev, out_dev)
    torch.cuda.synchronize()
    barrier(world)
    w0 = time.perf_counter()
    for i in range(e2e_steps):
        x_dev.copy_(x_host[i], non_blocking=True)
        stack_step(ctx, x_dev, out_dev)
        out_host[i].copy_(out_dev, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - w0
    barrier(world)
    dev_err |= int(err.item())

    elapsed_max, e2e_max = reduce_max(world, [elapsed, e2e_s], dev)
    ms_per_step = elapsed_max / steps
    by = bytes_of(T_line, nu)
    achieved = by / (ms_per_step * 1e-3) / 1e9
    launches += (1 + NL * path_of(T_line)[1] + path_of(T_line)[2]) * steps
    del layers, q_all, s_all, ctx, g_main, g_tail
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {
        "value": round(job_throughput(T_line, steps, world, elapsed_max), 2), "unit": UNIT, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms_per_step, 6),
        "config": {"workload": f"stack: {NL} resident MoE layers (out = x + MoE(RMSNorm(x))), E={E} routed + 1 "
                               f"shared, k={k}, d={d}, f={f}, int4 group-{G} fp32 scales, Zipf(1.1) selection "
                               f"bias with a per-layer expert permutation, T={T_line} token(s) per step, "
                               f"FFN path {args.mode if args.mode != 'workload' else 'automatic'}",
                   "T": T_line, "E": E, "k": k, "d": d, "f": f, "G": G, "layers": NL, "weights": "int4",
                   "l2": f"inputs larger than L2: {NL} resident layers ({NL * (E + 1) * blk / 1e9:.1f} GB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU", "cuda_graph_steps": S},
        "roofline": {"kernel": "whole 8-layer step (all kernels; bytes = sum of the layers' algorithmic bytes)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "peak_source": peaks["source"], "bytes_per_step": by},
        "n_uniq_per_layer": nu,
        "sweep": sweep,
        "e2e": {"value": round(T_line * e2e_steps * world / e2e_max, 2), "unit": UNIT,
                "h2d_bytes_per_step": T_line * d * 4, "d2h_bytes_per_step": T_line * d * 4, "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clocks,
        "device_error": dev_err,
    }


def run_stack(args, rank, world, local):
    """The stack workload as its own line (T from --tokens, default 64)."""
    import workloads
    dev = init_device(local, world)
    sh = workloads.WORKLOADS["stack"]
    res = measure_stack(args, rank, world, dev, args.tokens or sh.T, args.steps, args.warmup)
    line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic"}
    for key in ("config", "roofline", "n_uniq_per_layer", "sweep", "e2e", "gpu_launches", "clocks",
                "device_error"):
        line[key] = res[key]
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sh, args.cpu_seconds, layers=sh.layers)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(T, steps, world, elapsed_ms):
    """Whole-job tokens/s: every rank processes T tokens per step; the slowest rank's time counts."""
    return T * steps * world / (elapsed_ms * 1e-3)


def reduce_max(world, vals, dev):
    if world == 1:
        return vals
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def ncu_traffic(root, key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernels."""
    p = os.path.join(root, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as fh:
            j = json.load(fh)
        ent = j.get(key)
        if not ent or ent.get("source_hash") != kernel_source_hash(root):
            return None
        return ent.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        return None


# the sources the captured FFN kernels (and their tensor maps) are built from
FFN_SOURCES = ("ffn_decode.cu", "ffn_prefill.cu", "moe_internal.h", "ptx.cuh", "tmap.cu")


def kernel_source_hash(root):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(root, "int4_routed_expert_sigmoid_gb300", "csrc")
    for n in FFN_SOURCES:
        with open(os.path.join(csrc, n), "rb") as fh:
            h.update(n.encode() + fh.read())
    return h.hexdigest()[:16]


# -------------------------------------------------------------- CPU oracle --

def _oracle_layer(sh, f_used, seed=0):
    """The workload's layer for the oracle; f_used < f keeps the first f_used
    intermediate rows of every expert (a bounded sample of the same work)."""
    import oracle
    import workloads
    L = workloads.layer_inputs(sh, seed=seed, threads=os.cpu_count() or 8)
    d, f, G = sh.d, sh.f, sh.G
    if f_used != f:
        def cut(q, s):
            q = q.reshape(-1)
            s = s.reshape(-1)
            qg = q[: f * d // 2].reshape(f, d // 2)[:f_used]
            qu = q[f * d // 2: f * d].reshape(f, d // 2)[:f_used]
            qd = q[f * d:].reshape(d, f // 2)[:, : f_used // 2]
            sg = s[: f * d // G].reshape(f, d // G)[:f_used]
            su = s[f * d // G: 2 * f * d // G].reshape(f, d // G)[:f_used]
            sd = s[2 * f * d // G:].reshape(d, f // G)[:, : f_used // G]
            return (np.concatenate([qg.ravel(), qu.ravel(), qd.ravel()]),
                    np.concatenate([sg.ravel(), su.ravel(), sd.ravel()]))
        qs, ss = zip(*[cut(L.q_base[e], L.s_base[e]) for e in range(sh.E)])
        q_base, s_base = np.stack(qs), np.stack(ss)
        shq, shs = cut(L.shared_q, L.shared_s)
    else:
        q_base, s_base, shq, shs = L.q_base, L.s_base, L.shared_q, L.shared_s
    return oracle, L, q_base, s_base, shq, shs


def host_cpu() -> dict:
    """The host's logical CPU count and model name (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            key, _, val = ln.partition(":")
            if key.strip() in ("Model name", "Vendor ID") and val.strip():
                model = val.strip() if model is None or key.strip() == "Model name" else model
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as fh:
                for ln in fh:
                    if ln.lower().startswith(("model name", "cpu part", "hardware")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown"}


def cpu_baseline(sh, seconds: float, layers: int = 1) -> dict:
    """The oracle, as it stands, on a bounded sample: full layers for a few tokens.
    With layers > 1 (a stack of equally shaped layers) the rate of one layer is
    divided by the layer count."""
    import workloads
    oracle, L, q_base, s_base, shq, shs = _oracle_layer(sh, sh.f)
    threads = oracle.threads()
    x = workloads.activations(4 * threads, sh.d, seed=9000)
    lay = oracle.Layer(x[:1], L.wg, L.bias, q_base, s_base, shq, shs, d=sh.d, f=sh.f, E=sh.E, k=sh.k, G=sh.G)
    t = time.perf_counter()
    lay.tokens(np.array([0], np.int32))
    t1 = time.perf_counter() - t
    n = int(min(4 * threads, max(threads, round(seconds * threads / max(t1, 1e-3)))))
    lay = oracle.Layer(x[:n], L.wg, L.bias, q_base, s_base, shq, shs, d=sh.d, f=sh.f, E=sh.E, k=sh.k, G=sh.G)
    t = time.perf_counter()
    lay.tokens(np.arange(n, dtype=np.int32))
    el = time.perf_counter() - t
    per = f"; rate / {layers} for the {layers}-layer stack" if layers > 1 else ""
    return {"value": round(n / el / layers, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} tokens of the {sh.name} layer (route + shared + {sh.k} routed int4 experts, full "
                      f"d={sh.d}, f={sh.f}), fp64 C oracle, OpenMP over tokens, {el:.1f} s{per}", **host_cpu()}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one token through the layer,
    with the experts cut to their first f' intermediate rows so that the whole
    run stays within about two minutes; the rate is scaled by f / f'."""
    if rank != 0:
        return
    import workloads
    sh = workloads.WORKLOADS[args.workload]
    total = max(1, args.steps + args.warmup)
    budget = 90.0
    # measure one full token to size the sample
    oracle, L, q_base, s_base, shq, shs = _oracle_layer(sh, sh.f)
    x = workloads.activations(1, sh.d, seed=9100)
    lay = oracle.Layer(x, L.wg, L.bias, q_base, s_base, shq, shs, d=sh.d, f=sh.f, E=sh.E, k=sh.k, G=sh.G)
    t = time.perf_counter()
    lay.tokens(np.array([0], np.int32))
    t_full = time.perf_counter() - t
    frac = min(1.0, budget / total / max(t_full, 1e-6))
    f_used = max(sh.G, int(sh.f * frac) // sh.G * sh.G)
    del L, q_base, s_base
    oracle, L, q_base, s_base, shq, shs = _oracle_layer(sh, f_used)
    xs = workloads.activations(total, sh.d, seed=9200)
    laid = [None]

    def one(i):
        lay = oracle.Layer(xs[i:i + 1], L.wg, L.bias, q_base, s_base, shq, shs, d=sh.d, f=f_used, E=sh.E,
                           k=sh.k, G=sh.G)
        lay.tokens(np.array([0], np.int32))
        laid[0] = lay

    for i in range(args.warmup):
        one(i)
    t = time.perf_counter()
    for i in range(args.steps):
        one(args.warmup + i)
    el = time.perf_counter() - t
    # each step carries one token of the workload's batch (tokens are independent);
    # a stack step passes it through every layer, here one layer standing for each
    value = args.steps * (f_used / sh.f) / el / sh.layers
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{sh.name}: {sh.layers} MoE layer(s), E={sh.E} routed + 1 shared, k={sh.k}, d={sh.d}, "
                                   f"f={sh.f}, int4 group-{sh.G}, T={sh.T}"},
            "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                             **host_cpu(),
                             "sample": f"each step: one token of the T={sh.T} batch through the layer (OpenMP over "
                                       f"the output rows of every expert matrix) with every "
                                       f"expert cut to its first {f_used} of {sh.f} intermediate rows; rate scaled "
                                       f"by {sh.f}/{f_used}" + (f" and divided by {sh.layers} layers"
                                                               if sh.layers > 1 else "")},
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload == "stack":
        run_stack(args, rank, world, local)
        return
    if args.workload == "tier":
        dev = init_device(local, world)
        res = measure_tier(args, rank, world, dev, steps=args.steps, warmup=args.warmup)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "n_gpus": world, **res}), flush=True)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
