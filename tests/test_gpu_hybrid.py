"""The hybrid FFN (MOE_MODE_HYBRID, and MOE_MODE_AUTO from 128 tokens): every expert of the union
with at most 8 pairs takes the decode path, the others and the shared expert the tcgen05 prefill
path.  Each expert's output rows must be bitwise those its path gives on its own, the cold experts
must keep the decode path's 1e-4 tolerance against the oracle, and the layer must match the oracle
within the prefill tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_testlib import TOL_DECODE, TOL_PREFILL, device_layer, host, moe, oracle_layer, rel_max_err, run_steps

pytestmark = pytest.mark.gpu

Shape = workloads.Shape
COLD_MAX = 8   # pairs of an expert up to which the hybrid takes the decode path

# mixed (Zipf: a few hot experts), T >= 128 (AUTO resolves to the hybrid), all cold (m <= T <= 8),
# all hot (two experts, ~20 tokens each), f = 384 (an f that is not a multiple of 256), one token
SHAPES = [
    Shape("hyb_mixed", E=16, k=4, d=512, f=256, T=24, bias="zipf"),
    Shape("hyb_t130", E=32, k=4, d=512, f=384, T=130, bias="zipf"),
    Shape("hyb_cold", E=64, k=2, d=256, f=128, T=8, bias="normal"),
    Shape("hyb_hot", E=2, k=1, d=256, f=128, T=40, bias="zero"),
    Shape("hyb_t1", E=16, k=4, d=512, f=256, T=1, bias="normal"),   # the decode half's one-token, fixed-order form
]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_sigmoid_gb300 import build
    build.build()


def _ffn(m, dev, un, k, mode):
    T, d = dev["x"].shape
    y_pair = torch.full((T * k, d), float("nan"), device="cuda")
    y_shared = torch.full((T, d), float("nan"), device="cuda")
    _, _, err = m.moe_expert_ffn_int4(dev["x"], dev["layer"], un, k, mode, y_pair=y_pair, y_shared=y_shared)
    torch.cuda.synchronize()
    assert int(host(err)[0]) == 0
    return host(y_pair), host(y_shared)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_hybrid_rows_are_their_paths_rows(shape):
    m = moe()
    L = workloads.layer_inputs(shape, seed=3, threads=4)
    dev = device_layer(L)
    k = shape.k
    idx, _, _ = m.moe_route(dev["x"], dev["wg"], dev["bias"], k)
    un = m.moe_union(idx, shape.E)
    torch.cuda.synchronize()
    n = int(host(un["n_uniq"])[0])
    uniq, off = host(un["uniq"])[:n], host(un["offsets"])
    yd, _ = _ffn(m, dev, un, k, m.MOE_MODE_DECODE)
    yp, sp = _ffn(m, dev, un, k, m.MOE_MODE_PREFILL)
    yh, sh_ = _ffn(m, dev, un, k, m.MOE_MODE_HYBRID)
    assert np.array_equal(sh_, sp), "the shared expert is the prefill path's"
    n_cold = 0
    for e in uniq:
        lo, hi = off[e], off[e + 1]
        cold = hi - lo <= COLD_MAX
        n_cold += cold
        ref = yd if cold else yp
        assert np.array_equal(yh[lo:hi], ref[lo:hi]), f"expert {e} ({hi - lo} pairs, {'cold' if cold else 'hot'})"
    print(f"{shape.name}: {n_cold} cold of {n} experts")


@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: s.name)
def test_hybrid_layer_against_the_oracle(shape):
    """Teacher-forced (the oracle's routing): the layer within the prefill tolerance, each cold
    expert's rows within the decode tolerance, each hot expert's and the shared rows within the
    prefill tolerance."""
    m = moe()
    L = workloads.layer_inputs(shape, seed=5, threads=4)
    dev = device_layer(L)
    k = shape.k
    res = workloads.activations(shape.T, shape.d, seed=78)
    o_idx, o_w, _, _ = oracle.route(L.x, L.wg, L.bias, k)
    o_union = oracle.union(o_idx, shape.E)
    _, _, o_out = oracle_layer(L, res=res).dense()
    t = run_steps(dev, k, res=torch.from_numpy(res).cuda(), teacher_idx=o_idx, teacher_w=o_w,
                  mode=m.MOE_MODE_HYBRID)
    assert t["err"] == 0
    assert rel_max_err(t["out"], o_out) <= TOL_PREFILL
    y_sh = oracle.expert_ffn_tokens(L.x, np.arange(shape.T), L.shared_q, L.shared_s, shape.d, shape.f, shape.G)
    assert rel_max_err(t["y_shared"], y_sh) <= TOL_PREFILL
    for e in o_union["uniq"][:o_union["n_uniq"]]:
        lo, hi = o_union["offsets"][e], o_union["offsets"][e + 1]
        toks = o_union["sorted_pair"][lo:hi] // k
        y = oracle.expert_ffn_tokens(L.x, toks, L.q_base[e], L.s_base[e], shape.d, shape.f, shape.G)
        tol = TOL_DECODE if hi - lo <= COLD_MAX else TOL_PREFILL
        assert rel_max_err(t["y_pair"][lo:hi], y) <= tol, f"expert {e} ({hi - lo} pairs)"


def test_auto_from_128_tokens_is_the_hybrid():
    m = moe()
    sh = Shape("hyb_auto", E=32, k=4, d=512, f=256, T=128, bias="zipf")
    L = workloads.layer_inputs(sh, seed=7, threads=4)
    dev = device_layer(L)
    outs = []
    for mode in (m.MOE_MODE_AUTO, m.MOE_MODE_HYBRID):
        out, err = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], sh.k, mode=mode)
        torch.cuda.synchronize()
        assert int(host(err)[0]) == 0
        outs.append(host(out))
    assert np.array_equal(outs[0], outs[1])
