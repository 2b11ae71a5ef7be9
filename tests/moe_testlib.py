"""Shared helpers of the parity tests: move seeded inputs to the device, run the
CUDA path through the C ABI, and compare with the oracle.

Tolerances (fixed here, used by every parity test):
  * top-k indices, union arrays, hit counters: bit-exact.  A token whose oracle
    selection keys of two competing experts (adjacent in key order among the
    first k+1) differ by at most NEAR_TIE is flagged and reported; its routing
    is not required to match.
  * fp32-accurate (decode) path outputs: max |gpu - oracle| <= 1e-4 * RMS(oracle).
  * bf16 tensor-core (prefill) path outputs: max |gpu - oracle| <= 2e-2 * RMS(oracle).
  * combine weights: relative 1e-5 (fp32 sigmoid vs fp64).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

NEAR_TIE = 1e-6
TOL_DECODE = 1e-4
TOL_PREFILL = 2e-2
TOL_WEIGHT = 1e-5


def moe():
    import int4_routed_expert_sigmoid_gb300 as m
    return m


def device_layer(L: workloads.LayerInputs, device="cuda"):
    """Device copies of one layer's inputs and the C-ABI weight view."""
    m = moe()
    sh = L.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    lw = m.LayerWeights(t(L.q_base.reshape(-1)), t(L.s_base.reshape(-1)), t(L.shared_q), t(L.shared_s),
                        E=sh.E, d=sh.d, f=sh.f, G=sh.G)
    return dict(x=t(L.x), wg=t(L.wg), bias=None if L.bias is None else t(L.bias), layer=lw)


def oracle_layer(L: workloads.LayerInputs, *, k=None, normalize=1, route_scale=1.0, res=None, x=None,
                 top_p=1.0):
    sh = L.shape
    return oracle.Layer(L.x if x is None else x, L.wg, L.bias, L.q_base, L.s_base, L.shared_q, L.shared_s,
                        d=sh.d, f=sh.f, E=sh.E, k=sh.k if k is None else k, G=sh.G, normalize=normalize,
                        route_scale=route_scale, res=res, top_p=top_p)


def near_tie_tokens(keys: np.ndarray, k: int, tol: float = NEAR_TIE) -> np.ndarray:
    """Tokens whose key order among the first k+1 experts is decided by <= tol."""
    s = -np.sort(-keys, axis=1)[:, :min(k + 1, keys.shape[1])]
    gaps = s[:, :-1] - s[:, 1:]
    return (gaps <= tol).any(axis=1) if gaps.shape[1] else np.zeros(keys.shape[0], bool)


def topp_cut_ties(raw_w: np.ndarray, top_p: float, tol: float = NEAR_TIE) -> np.ndarray:
    """Tokens whose top-p cut is decided by <= tol: raw_w holds the oracle's unnormalised
    scores of the k chosen experts in selection order (top_p = 1), and a token is
    flagged when some prefix sum of them lies within tol * total of top_p * total."""
    if top_p >= 1.0:
        return np.zeros(raw_w.shape[0], bool)
    cum = np.cumsum(raw_w, axis=1)
    total = cum[:, -1:]
    return (np.abs(cum[:, :-1] - top_p * total) <= tol * total).any(axis=1)


def compare_routing(gpu_idx, gpu_w, o_idx, o_w, keys, k, extra_flags=None):
    """Asserts exact indices outside near-ties; returns (matched mask, flagged mask)."""
    flagged = near_tie_tokens(keys, k)
    if extra_flags is not None:
        flagged = flagged | extra_flags
    same = (gpu_idx == o_idx).all(axis=1)
    bad = ~same & ~flagged
    assert not bad.any(), f"routing differs on tokens {np.nonzero(bad)[0][:10]} (not near-ties)"
    if same.any():
        rel = np.abs(gpu_w[same] - o_w[same]) / np.maximum(np.abs(o_w[same]), 1e-30)
        assert rel.max() <= TOL_WEIGHT, f"combine weights off by {rel.max():.3e}"
    if flagged.any():
        print(f"[near-tie] {int(flagged.sum())} token(s) flagged; {int((~same & flagged).sum())} differ")
    return same, flagged


def rel_max_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(np.square(ref)))) if ref.size else 0.0
    return float(np.max(np.abs(gpu.astype(np.float64) - ref))) / max(rms, 1e-300)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def run_steps(dev: dict, k: int, *, normalize=1, route_scale=1.0, res=None, hits=None, mode=None,
              teacher_idx=None, teacher_w=None):
    """Route -> union(+hits) -> FFN -> combine through the separate entry points.

    teacher_idx/teacher_w (host arrays from the oracle) replace the GPU routing
    for the downstream stages when given."""
    m = moe()
    mode = m.MOE_MODE_AUTO if mode is None else mode
    lw = dev["layer"]
    idx, w, logits = m.moe_route(dev["x"], dev["wg"], dev["bias"], k, normalize, route_scale)
    use_idx, use_w = idx, w
    if teacher_idx is not None:
        use_idx = torch.from_numpy(np.ascontiguousarray(teacher_idx, np.int32)).cuda()
        use_w = torch.from_numpy(np.ascontiguousarray(teacher_w, np.float32)).cuda()
    un = m.moe_union(use_idx, lw.E, hits=hits)
    y_pair, y_shared, ferr = m.moe_expert_ffn_int4(dev["x"], lw, un, k, mode)
    out = m.moe_combine(y_pair, y_shared, use_w, un["perm"], residual=res)
    torch.cuda.synchronize()
    r = dict(idx=host(idx), w=host(w), logits=host(logits), out=host(out), y_pair=host(y_pair),
             y_shared=host(y_shared), err=int(host(un["err"])[0]) | int(host(ferr)[0]))
    for key in ("counts", "offsets", "perm", "sorted_pair", "uniq"):
        r[key] = host(un[key])
    r["n_uniq"] = int(host(un["n_uniq"])[0])
    return r


def check_union_equal(r: dict, u: dict, E: int):
    """Union arrays equal; sorted_pair only over its offsets[E] placed pairs (the rest is unspecified
    when slots are empty)."""
    assert r["n_uniq"] == u["n_uniq"]
    for key in ("counts", "offsets", "perm"):
        assert np.array_equal(r[key], u[key]), key
    n = int(u["offsets"][E])
    assert np.array_equal(r["sorted_pair"][:n], u["sorted_pair"][:n]), "sorted_pair"
    assert np.array_equal(r["uniq"][:u["n_uniq"]], u["uniq"][:u["n_uniq"]])
