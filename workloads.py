"""Seeded synthetic inputs for one GLM-5.2-shaped MoE layer.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It only draws random numbers and lays them out; it holds none of the
method's arithmetic (no routing, no dequantisation, no FFN).

Workloads (layer shapes from the colibri README, "The idea": 75 MoE layers of
256 routed experts, ~19 MB per expert at int4, ~11 GB of routed experts per
token, i.e. k = 8 with d = 6144, f = 2048):

  tiny            E=8   (+1 shared), k=2, d=256,  f=128,  T=16,   bias 0
  decode          E=256 (+1 shared), k=8, d=6144, f=2048, T=1,    bias ~ N(0, 0.1)
  batched_decode  same shape, T=64,   Zipf(1.1) selection bias
  prefill         same shape, T=4096, bias 0 (natural, near-uniform routing)
  stack           8 layers, T in {1, 4, 16, 64, 256}, Zipf bias whose expert
                  permutation changes per layer

Distributions: x ~ N(0, 1) fp32; router W_g ~ N(0, 0.02^2) fp32; packed int4
bytes uniform over 0..255 (each nibble uniform over [-8, 7]); scales
exp(-4 + 0.3 N(0, 1)) fp32, one per 32-element group.

Zipf selection bias: b_e = c * ln p_rank(e), p_r = r^-1.1 / sum_r r^-1.1, with
the rank order a seeded permutation of the experts.  c = 0.04 was calibrated
once by a seeded simulation of 20,000 tokens (sigmoid scores of N(0, 1.57^2)
logits plus b, top-8): the selection frequency then falls with rank with a
log-log slope of -1.13.

Every stream is a numpy PCG64 generator seeded by a SeedSequence of
(seed, layer, stream tag[, expert]), so one expert's weights can be regenerated
without the rest of the layer.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

ZIPF_S = 1.1
ZIPF_C = 0.04

_TAG_X, _TAG_WG, _TAG_BIAS, _TAG_PERM, _TAG_EXPERT, _TAG_SHARED = 11, 12, 13, 14, 15, 16


@dataclass(frozen=True)
class Shape:
    name: str
    E: int
    k: int
    d: int
    f: int
    T: int
    G: int = 32
    bias: str = "zero"          # "zero" | "normal" | "zipf"
    layers: int = 1
    batch_sweep: tuple = field(default=())


WORKLOADS = {
    "tiny": Shape("tiny", E=8, k=2, d=256, f=128, T=16),
    "decode": Shape("decode", E=256, k=8, d=6144, f=2048, T=1, bias="normal"),
    "batched_decode": Shape("batched_decode", E=256, k=8, d=6144, f=2048, T=64, bias="zipf"),
    "prefill": Shape("prefill", E=256, k=8, d=6144, f=2048, T=4096),
    "stack": Shape("stack", E=256, k=8, d=6144, f=2048, T=64, bias="zipf", layers=8,
                   batch_sweep=(1, 4, 16, 64, 256)),
}


def expert_q_bytes(d: int, f: int) -> int:
    """Packed bytes of one expert: gate [f][d], up [f][d], down [d][f] at 4 bits."""
    return 3 * d * f // 2


def expert_s_count(d: int, f: int, G: int) -> int:
    """fp32 scales of one expert: one per G elements of each of the three matrices."""
    return 3 * d * f // G


def _rng(seed: int, layer: int, tag: int, extra: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, tag, extra])))


def activations(T: int, d: int, seed: int, layer: int = 0) -> np.ndarray:
    return _rng(seed, layer, _TAG_X).standard_normal((T, d), dtype=np.float32)


def router_weights(E: int, d: int, seed: int, layer: int = 0) -> np.ndarray:
    w = _rng(seed, layer, _TAG_WG).standard_normal((E, d), dtype=np.float32)
    w *= np.float32(0.02)
    return w


def selection_bias(E: int, kind: str, seed: int, layer: int = 0) -> np.ndarray | None:
    if kind == "zero":
        return None
    if kind == "normal":
        b = _rng(seed, layer, _TAG_BIAS).standard_normal(E, dtype=np.float32)
        return b * np.float32(0.1)
    if kind == "zipf":
        order = _rng(seed, layer, _TAG_PERM).permutation(E)   # order[r-1] = expert of rank r
        rank = np.empty(E, dtype=np.float64)
        rank[order] = np.arange(1, E + 1, dtype=np.float64)
        lnp = -ZIPF_S * np.log(rank) - np.log(np.sum(np.arange(1, E + 1, dtype=np.float64) ** -ZIPF_S))
        return (ZIPF_C * lnp).astype(np.float32)
    raise ValueError(kind)


def expert_block(d: int, f: int, G: int, seed: int, layer: int, expert: int,
                 q_out: np.ndarray | None = None, s_out: np.ndarray | None = None):
    """One expert's packed bytes (gate|up|down) and fp32 scales (gate|up|down).

    expert = -1 gives the layer's shared expert.
    """
    tag = _TAG_SHARED if expert < 0 else _TAG_EXPERT
    r = _rng(seed, layer, tag, max(expert, 0))
    nq, ns = expert_q_bytes(d, f), expert_s_count(d, f, G)
    q = np.frombuffer(r.bytes(nq), dtype=np.uint8)
    z = r.standard_normal(ns, dtype=np.float32)
    z *= np.float32(0.3)
    z -= np.float32(4.0)
    s = np.exp(z)
    if q_out is not None:
        q_out[:] = q
        s_out[:] = s
        return q_out, s_out
    return q.copy(), s


@dataclass
class LayerInputs:
    shape: Shape
    layer: int
    x: np.ndarray          # [T][d] fp32 (layer 0's input; later layers take the previous output)
    wg: np.ndarray         # [E][d] fp32
    bias: np.ndarray | None
    q_base: np.ndarray     # [E][expert_q_bytes] uint8
    s_base: np.ndarray     # [E][expert_s_count] fp32
    shared_q: np.ndarray
    shared_s: np.ndarray


def layer_inputs(shape: Shape, seed: int = 0, layer: int = 0, T: int | None = None,
                 threads: int = 8, q_base: np.ndarray | None = None,
                 s_base: np.ndarray | None = None) -> LayerInputs:
    """All inputs of one layer.  q_base/s_base may be preallocated (e.g. pinned) buffers."""
    E, d, f, G = shape.E, shape.d, shape.f, shape.G
    T = shape.T if T is None else T
    nq, ns = expert_q_bytes(d, f), expert_s_count(d, f, G)
    if q_base is None:
        q_base = np.empty((E, nq), dtype=np.uint8)
    if s_base is None:
        s_base = np.empty((E, ns), dtype=np.float32)
    q_base = q_base.reshape(E, nq)
    s_base = s_base.reshape(E, ns)

    def one(e):
        expert_block(d, f, G, seed, layer, e, q_base[e], s_base[e])

    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(one, range(E)))
    sq, ss = expert_block(d, f, G, seed, layer, -1)
    return LayerInputs(shape, layer, activations(T, d, seed, layer), router_weights(E, d, seed, layer),
                       selection_bias(E, shape.bias, seed, layer), q_base, s_base, sq, ss)
