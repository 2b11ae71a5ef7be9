"""GPU parity: the CUDA path through the C ABI vs the fp64 oracle on the same
seeded inputs (small shapes that span several tiles, k-chunks and ragged tails).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_testlib import (TOL_DECODE, TOL_PREFILL, check_union_equal, compare_routing, device_layer, host, moe,
                         near_tie_tokens, oracle_layer, rel_max_err, run_steps, topp_cut_ties)

pytestmark = pytest.mark.gpu

Shape = workloads.Shape
SMALL = [
    workloads.WORKLOADS["tiny"],                                            # 4 gate/up tiles, 1 k-chunk
    Shape("ragged_kc128", E=16, k=4, d=1024, f=384, T=37, bias="normal"),   # 4 k-chunks, 128-wide down chunks
    Shape("zipf_small", E=64, k=8, d=512, f=512, T=5, bias="zipf"),
    Shape("single_token", E=33, k=3, d=256, f=256, T=1, bias="normal"),
    Shape("multi_pass", E=8, k=2, d=256, f=128, T=300),                     # > 16 tokens per expert
    Shape("k1", E=4, k=1, d=256, f=128, T=9, bias="normal"),
    Shape("split4_t1", E=16, k=4, d=2048, f=256, T=1, bias="normal"),      # gate/up reduction in 4 parts
    Shape("split2_t1", E=12, k=2, d=1024, f=128, T=1, bias="normal"),      # ... in 2 parts
    Shape("k_eq_E", E=8, k=8, d=256, f=128, T=20, bias="normal"),         # every token takes every expert
    Shape("one_expert", E=1, k=1, d=256, f=128, T=7),                      # a single routed expert
]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_sigmoid_gb300 import build
    build.build()


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("normalize,route_scale,with_res", [(1, 1.0, False), (0, 1.0, True), (1, 2.5, True)])
def test_layer_parity_small(shape, normalize, route_scale, with_res):
    m = moe()
    L = workloads.layer_inputs(shape, seed=1, threads=4)
    res = workloads.activations(shape.T, shape.d, seed=77) if with_res else None
    dev = device_layer(L)
    res_d = torch.from_numpy(res).cuda() if res is not None else None
    k = shape.k

    o_idx, o_w, o_logits, keys = oracle.route(L.x, L.wg, L.bias, k, normalize, route_scale)
    o_union = oracle.union(o_idx, shape.E)
    _, _, o_out = oracle_layer(L, normalize=normalize, route_scale=route_scale, res=res).dense()

    # 1) the layer as the GPU routes it
    hits = torch.zeros(shape.E, dtype=torch.int64, device="cuda")
    dec = m.MOE_MODE_DECODE   # this test holds the decode path to its tolerance at every T
    r = run_steps(dev, k, normalize=normalize, route_scale=route_scale, res=res_d, hits=hits, mode=dec)
    assert r["err"] == 0
    assert np.max(np.abs(r["logits"] - o_logits)) <= 1e-5 * max(1.0, float(np.abs(o_logits).max()))
    same, flagged = compare_routing(r["idx"], r["w"], o_idx, o_w, keys, k)
    if same.all():
        check_union_equal(r, o_union, shape.E)
        assert np.array_equal(host(hits), o_union["counts"].astype(np.int64))
    assert int(host(hits).sum()) == shape.T * k
    assert rel_max_err(r["out"][same], o_out[same]) <= TOL_DECODE

    # 2) teacher-forced: downstream stages on the oracle's routing, all tokens
    t = run_steps(dev, k, res=res_d, teacher_idx=o_idx, teacher_w=o_w, mode=dec)
    assert t["err"] == 0
    check_union_equal(t, o_union, shape.E)
    assert rel_max_err(t["out"], o_out) <= TOL_DECODE
    y_sh = oracle.expert_ffn_tokens(L.x, np.arange(shape.T), L.shared_q, L.shared_s, shape.d, shape.f, shape.G)
    assert rel_max_err(t["y_shared"], y_sh) <= TOL_DECODE
    for e in o_union["uniq"][:o_union["n_uniq"]]:
        lo, hi = o_union["offsets"][e], o_union["offsets"][e + 1]
        toks = o_union["sorted_pair"][lo:hi] // k
        y = oracle.expert_ffn_tokens(L.x, toks, L.q_base[e], L.s_base[e], shape.d, shape.f, shape.G)
        assert rel_max_err(t["y_pair"][lo:hi], y) <= TOL_DECODE, f"expert {e}"

    # 3) the fused entry point gives the same bits as the separate calls
    out_f, err_f = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], k, normalize, route_scale,
                                       mode=dec, residual=res_d)
    torch.cuda.synchronize()
    assert int(host(err_f)[0]) == 0
    assert np.array_equal(host(out_f), r["out"])


def test_fused_layer_is_deterministic():
    m = moe()
    L = workloads.layer_inputs(SMALL[1], seed=3, threads=4)
    dev = device_layer(L)
    outs = []
    for _ in range(3):
        o, e = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], SMALL[1].k)
        torch.cuda.synchronize()
        assert int(host(e)[0]) == 0
        outs.append(host(o))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_union_flags_bad_expert_ids():
    m = moe()
    E, k = 8, 2
    idx = torch.tensor([[0, 3], [8, 3], [3, -2], [7, 0]], dtype=torch.int32, device="cuda")
    un = m.moe_union(idx, E)
    torch.cuda.synchronize()
    assert int(host(un["err"])[0]) & m.MOE_DEVERR_BAD_EXPERT
    perm = host(un["perm"])
    assert perm[2] == -1 and perm[5] == -1
    valid = [0, 1, 3, 4, 6, 7]
    sp = host(un["sorted_pair"])
    assert sorted(perm[valid].tolist()) == list(range(6))
    assert np.array_equal(sp[perm[valid]], np.array(valid))
    assert host(un["counts"]).tolist() == [2, 0, 0, 3, 0, 0, 0, 1]


def test_hits_accumulate_across_calls():
    m = moe()
    rng = np.random.default_rng(0)
    E, T, k = 256, 64, 8
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    hits = torch.zeros(E, dtype=torch.int64, device="cuda")
    d_idx = torch.from_numpy(idx).cuda()
    for _ in range(3):
        un = m.moe_union(d_idx, E, hits=hits)
    m.moe_hits(un["counts"], hits)
    torch.cuda.synchronize()
    expect = 4 * np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(host(hits), expect) and int(host(hits).sum()) == 4 * T * k


def test_abi_rejects_bad_arguments_on_device():
    m = moe()
    L = workloads.layer_inputs(workloads.WORKLOADS["tiny"], seed=0, threads=2)
    dev = device_layer(L)
    lw = dev["layer"]
    x = dev["x"]
    T, d = x.shape
    small_ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward(x, dev["wg"], None, lw, 2, ws=small_ws)
    assert ei.value.status == m.MOE_ERR_WORKSPACE
    bad = m.LayerWeights(lw.q_base, lw.s_base, lw.shared_q, lw.shared_s, E=lw.E, d=lw.d, f=lw.f, G=32)
    bad.c.G = 64
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward(x, dev["wg"], None, bad, 2)
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED
    with pytest.raises(m.MoeError) as ei:
        m.moe_route(x, dev["wg"], None, k=9)                # k > E
    assert ei.value.status == m.MOE_ERR_INVALID_ARG
    with pytest.raises(m.MoeError) as ei:
        m.moe_route(x[:, :255].contiguous(), dev["wg"], None, k=2)   # d not a multiple of 4
    assert ei.value.status == m.MOE_ERR_INVALID_ARG


PREFILL_SHAPES = [
    workloads.WORKLOADS["tiny"],                                            # 1 gate/up m-tile, 2 down m-tiles
    Shape("prefill_ragged", E=16, k=4, d=1024, f=384, T=37, bias="normal"),  # 3 and 8 m-tiles
    Shape("prefill_two_ntiles", E=8, k=2, d=256, f=128, T=300),              # shared expert: 256 + 44 tokens
    Shape("prefill_one_token", E=16, k=4, d=1024, f=384, T=1, bias="normal"),  # every unit a single token
    Shape("prefill_k_eq_E", E=8, k=8, d=256, f=128, T=130, bias="normal"),     # every expert takes every token
    Shape("prefill_one_expert", E=1, k=1, d=256, f=128, T=130),                # a single routed expert
]


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=lambda s: s.name)
def test_prefill_ffn_parity(shape):
    """tcgen05 prefill path (bf16 operands, fp32 accumulate) on the oracle's routing."""
    from moe_testlib import TOL_PREFILL
    m = moe()
    L = workloads.layer_inputs(shape, seed=2, threads=4)
    dev = device_layer(L)
    k = shape.k
    o_idx, o_w, _, _ = oracle.route(L.x, L.wg, L.bias, k, 1, 1.0)
    o_union = oracle.union(o_idx, shape.E)
    _, _, o_out = oracle_layer(L).dense()
    t = run_steps(dev, k, teacher_idx=o_idx, teacher_w=o_w, mode=m.MOE_MODE_PREFILL)
    assert t["err"] == 0
    check_union_equal(t, o_union, shape.E)
    y_sh = oracle.expert_ffn_tokens(L.x, np.arange(shape.T), L.shared_q, L.shared_s, shape.d, shape.f, shape.G)
    assert rel_max_err(t["y_shared"], y_sh) <= TOL_PREFILL
    for e in o_union["uniq"][:o_union["n_uniq"]]:
        lo, hi = o_union["offsets"][e], o_union["offsets"][e + 1]
        toks = o_union["sorted_pair"][lo:hi] // k
        y = oracle.expert_ffn_tokens(L.x, toks, L.q_base[e], L.s_base[e], shape.d, shape.f, shape.G)
        assert rel_max_err(t["y_pair"][lo:hi], y) <= TOL_PREFILL, f"expert {e}"
    assert rel_max_err(t["out"], o_out) <= TOL_PREFILL
    # the fused entry point in prefill mode routes itself; compare where the routing agrees
    out_f, err_f = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], k, mode=m.MOE_MODE_PREFILL)
    torch.cuda.synchronize()
    assert int(host(err_f)[0]) == 0
    r = run_steps(dev, k)
    same = (r["idx"] == o_idx).all(axis=1)
    assert rel_max_err(host(out_f)[same], o_out[same]) <= TOL_PREFILL
    # the automatic mode takes the hybrid path from 128 tokens on, the decode path below
    out_a, _ = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], k)
    want = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], k,
                               mode=m.MOE_MODE_HYBRID if shape.T >= 128 else m.MOE_MODE_DECODE)[0]
    assert np.array_equal(host(out_a), host(want))


@pytest.mark.parametrize("T,d,scale", [(1, 256, 1.0), (37, 1024, 1e-3), (5, 6144, 3e4)])
def test_rms_norm_parity(T, d, scale):
    """The stack's normalisation vs the oracle (fp32 vs fp64), in place and out of place."""
    m = moe()
    x = workloads.activations(T, d, seed=T) * np.float32(scale)
    ref = oracle.rms_norm(x, 1e-5)
    xd = torch.from_numpy(x).cuda()
    out = host(m.moe_rms_norm(xd, 1e-5))
    # <= ~40 roundings of 2^-24 relative on |x_n| <= ~4.5 (see the full-size test)
    assert rel_max_err(out, ref) <= 1.2e-5
    m.moe_rms_norm(xd, 1e-5, out=xd)
    torch.cuda.synchronize()
    assert np.array_equal(host(xd), out)


ROUTE_TC = [
    # (T, E, d, bias, x scale): token counts that take the tensor-core logits kernel, a ragged last
    # token tile, several expert tiles, and inputs far from unit scale (the split keeps fp32's range)
    (512, 64, 1024, "normal", 1.0),
    (777, 128, 2048, "zipf", 1.0),
    (640, 256, 512, "normal", 1e3),
    (520, 64, 256, "zero", 1e-3),
    (130, 256, 6144, "normal", 1.0),   # the GLM-5.2 router width, a ragged second token tile
]


@pytest.mark.parametrize("T,E,d,bias,xs", ROUTE_TC, ids=lambda v: str(v))
def test_route_tensor_core_logits(T, E, d, bias, xs):
    """Large-T routing (split-tf32 logits on the tensor cores) against the fp64 oracle."""
    m = moe()
    k = 8
    x = workloads.activations(T, d, seed=11) * np.float32(xs)
    wg = workloads.router_weights(E, d, seed=12)
    b = workloads.selection_bias(E, bias, seed=13)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    idx, w, logits = m.moe_route(t(x), t(wg), None if b is None else t(b), k)
    torch.cuda.synchronize()
    o_idx, o_w, o_logits, keys = oracle.route(x, wg, b, k, 1, 1.0)
    lg = host(logits)
    assert np.isfinite(lg).all()
    assert np.max(np.abs(lg - o_logits)) <= 1e-5 * max(1.0, float(np.abs(o_logits).max()))
    compare_routing(host(idx), host(w), o_idx, o_w, keys, k)


UNION_CASES = [
    # (T, k, E, duplicates): more than 1024 pairs with distinct experts per token take the bitmap
    # path (sizes up to the prefill batch), fewer the chunked path; an expert named twice by one
    # token sends a bitmap call to the chunked path; a bitmap too large for shared memory
    # (E = 1024, T = 2048) takes the chunked path directly
    (1, 8, 256, False), (37, 4, 16, False), (4096, 8, 256, False), (300, 8, 1024, False),
    (2048, 8, 1024, False), (64, 8, 256, True), (5000, 2, 8, True), (700, 8, 64, True),
]


@pytest.mark.parametrize("T,k,E,dups", UNION_CASES, ids=lambda v: str(v))
def test_union_paths_bit_exact(T, k, E, dups):
    """The union kernel's paths against the oracle's stable counting sort, bit for bit."""
    m = moe()
    rng = np.random.default_rng(T * 7 + E)
    if dups:
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
        idx[:, 1] = idx[:, 0]   # every token names its first expert twice
    else:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    hits = torch.zeros(E, dtype=torch.int64, device="cuda")
    un = m.moe_union(torch.from_numpy(idx).cuda(), E, hits=hits)
    torch.cuda.synchronize()
    r = {key: host(v) for key, v in un.items()}
    r["n_uniq"] = int(r["n_uniq"][0])
    assert int(r["err"][0]) == 0
    o = oracle.union(idx, E)
    check_union_equal(r, o, E)
    assert np.array_equal(host(hits), o["counts"].astype(np.int64))


# ------------------------------------------------------------ wide routing ----
# Selection widths and expert counts the ABI accepts beyond the GLM-5.2 shape, up to both maxima: k up to 32
# (every candidate slot of a 32-expert block is used), E up to 1024 (32 blocks of 32).
WIDE = [(64, 16), (256, 16), (64, 32), (256, 32), (512, 8), (1024, 8), (1024, 32)]


@pytest.mark.parametrize("E,k", WIDE, ids=lambda v: str(v))
def test_route_wide_selection_block_topk(E, k):
    """The stand-alone top-k kernel (T > 8) against the oracle's brute-force order."""
    m = moe()
    T, d = 37, 256
    x = workloads.activations(T, d, seed=E + k)
    wg = workloads.router_weights(E, d, seed=E * k) * np.float32(20.0)   # logits ~ N(0, 0.8)
    b = workloads.selection_bias(E, "normal", seed=k)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    idx, w, logits = m.moe_route(t(x), t(wg), t(b), k)
    torch.cuda.synchronize()
    o_idx, o_w, o_logits, keys = oracle.route(x, wg, b, k)
    assert np.max(np.abs(host(logits) - o_logits)) <= 1e-5 * max(1.0, float(np.abs(o_logits).max()))
    same, _ = compare_routing(host(idx), host(w), o_idx, o_w, keys, k)
    assert same.sum() >= T - 2


@pytest.mark.parametrize("E,k", WIDE, ids=lambda v: str(v))
def test_layer_wide_selection_small_batch(E, k):
    """The fused small-batch path (select + union in one block, T <= 8 and T*k <= 64) and the
    general decode path at the same widths: routing, union, hits and outputs against the oracle."""
    m = moe()
    T_small = min(8, 64 // k)
    for T in (T_small, 11):
        sh = Shape(f"wide_{E}_{k}_{T}", E=E, k=k, d=256, f=128, T=T, bias="normal")
        L = workloads.layer_inputs(sh, seed=E + T, threads=8)
        dev = device_layer(L)
        hits = torch.zeros(E, dtype=torch.int64, device="cuda")
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        out, err = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], k, mode=m.MOE_MODE_DECODE,
                                       topk_idx=idx, hits=hits)
        torch.cuda.synchronize()
        assert int(host(err)[0]) == 0
        o_idx, o_w, _, keys = oracle.route(L.x, L.wg, L.bias, k)
        gi = host(idx)
        flagged = near_tie_tokens(keys, k)
        assert np.array_equal(gi[~flagged], o_idx[~flagged]), f"T={T}"
        assert np.array_equal(host(hits), oracle.union(gi, E)["counts"].astype(np.int64))
        same = (gi == o_idx).all(axis=1)
        _, _, o_out = oracle_layer(L).dense()
        assert rel_max_err(host(out)[same], o_out[same]) <= TOL_DECODE, f"T={T}"


# ------------------------------------------------------------------ top-p ----

def _topp_flags(L_or_x, wg, bias, k, top_p):
    x = L_or_x
    _, raw, _, keys = oracle.route(x, wg, bias, k, normalize=0, top_p=1.0)
    return near_tie_tokens(keys, k) | topp_cut_ties(raw, top_p)


@pytest.mark.parametrize("top_p", [0.3, 0.6, 0.85, 0.999])
def test_route_topp_parity(top_p):
    """moe_route_topp against the oracle's cut (bit-exact outside flagged ties), on the
    stand-alone top-k kernel; top_p = 1 gives moe_route's bits."""
    m = moe()
    T, d, E, k = 300, 512, 256, 8
    x = workloads.activations(T, d, seed=7)
    wg = workloads.router_weights(E, d, seed=8) * np.float32(30.0)
    b = workloads.selection_bias(E, "normal", seed=9)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    idx, w, _ = m.moe_route(t(x), t(wg), t(b), k, top_p=top_p)
    torch.cuda.synchronize()
    o_idx, o_w, _, keys = oracle.route(x, wg, b, k, top_p=top_p)
    flags = _topp_flags(x, wg, b, k, top_p)
    same, _ = compare_routing(host(idx), host(w), o_idx, o_w, keys, k, extra_flags=flags)
    gi = host(idx)
    assert same.sum() >= T - 5
    assert np.all(gi[:, 0] >= 0) and ((gi == -1).any() or top_p > 0.99)
    # the kept slots are a prefix of plain top-k's slots
    i1, w1, _ = m.moe_route(t(x), t(wg), t(b), k, top_p=1.0)
    i0, w0, _ = m.moe_route(t(x), t(wg), t(b), k)
    torch.cuda.synchronize()
    assert np.array_equal(host(i1), host(i0)) and np.array_equal(host(w1), host(w0))
    kept = gi >= 0
    assert np.array_equal(gi[kept], host(i0)[kept])


@pytest.mark.parametrize("T,mode_name", [(5, "MOE_MODE_DECODE"), (37, "MOE_MODE_DECODE"), (37, "MOE_MODE_PREFILL"),
                                         (37, "MOE_MODE_HYBRID"), (130, "MOE_MODE_HYBRID")])
def test_layer_topp_parity(T, mode_name):
    """The fused layer with top-p pruning (small-batch select+union path at T = 5, stage kernels at
    T = 37, both FFN paths and the hybrid): routing, union with empty slots, hits and outputs against the
    oracle."""
    m = moe()
    mode = getattr(m, mode_name)
    tol = TOL_DECODE if mode == m.MOE_MODE_DECODE else TOL_PREFILL
    top_p = 0.7
    sh = Shape(f"topp_{T}", E=32, k=8, d=512, f=256, T=T, bias="normal")
    L = workloads.layer_inputs(sh, seed=T, threads=8)
    dev = device_layer(L)
    res = workloads.activations(T, sh.d, seed=5)
    hits = torch.zeros(sh.E, dtype=torch.int64, device="cuda")
    idx = torch.empty((T, sh.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, sh.k), dtype=torch.float32, device="cuda")
    out, err = m.moe_layer_forward(dev["x"], dev["wg"], dev["bias"], dev["layer"], sh.k, 1, 1.0, mode=mode,
                                   residual=torch.from_numpy(res).cuda(), topk_idx=idx, topk_w=w, hits=hits,
                                   top_p=top_p)
    torch.cuda.synchronize()
    assert int(host(err)[0]) == 0
    o_idx, o_w, _, keys = oracle.route(L.x, L.wg, L.bias, sh.k, top_p=top_p)
    same, _ = compare_routing(host(idx), host(w), o_idx, o_w, keys, sh.k,
                              extra_flags=_topp_flags(L.x, L.wg, L.bias, sh.k, top_p))
    gi = host(idx)
    assert (gi == -1).any()
    assert np.array_equal(host(hits), oracle.union(gi, sh.E)["counts"].astype(np.int64))
    assert int(host(hits).sum()) == int((gi >= 0).sum())
    _, _, o_out = oracle_layer(L, res=res, top_p=top_p).dense()
    assert rel_max_err(host(out)[same], o_out[same]) <= tol


def test_union_empty_slots():
    """-1 marks an empty slot: no group, perm -1, no hit, no error (bitmap and chunked paths)."""
    m = moe()
    rng = np.random.default_rng(3)
    for T, k, E in ((5, 4, 16), (600, 8, 64)):
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        cut = rng.integers(1, k + 1, size=T)
        for t in range(T):
            idx[t, cut[t]:] = -1
        hits = torch.zeros(E, dtype=torch.int64, device="cuda")
        un = m.moe_union(torch.from_numpy(idx).cuda(), E, hits=hits)
        torch.cuda.synchronize()
        r = {key: host(v) for key, v in un.items()}
        r["n_uniq"] = int(r["n_uniq"][0])
        assert int(r["err"][0]) == 0
        o = oracle.union(idx, E)
        check_union_equal(r, o, E)
        assert np.all(r["perm"][idx.reshape(-1) == -1] == -1)
        assert np.array_equal(host(hits), o["counts"].astype(np.int64))


# -------------------------------------------------- prefill scale range ----

@pytest.mark.parametrize("mu", [-12.0, 5.0, -25.0, 12.0])
def test_prefill_weight_scale_range(mu):
    """Group scales lognormal(mu, 0.3) far from the workloads' mu = -4: the prefill path scales each
    weight row by a power of two, so its fp16 weights keep their precision at any magnitude
    (2e-2 of the RMS); the decode path applies fp32 scales after the MMA (1e-4)."""
    from moe_testlib import TOL_PREFILL
    m = moe()
    sh = Shape("scale_range", E=16, k=4, d=1024, f=384, T=37, bias="normal")
    L = workloads.layer_inputs(sh, seed=4, threads=8)
    fac = np.float32(np.exp(mu + 4.0))
    L.s_base[:] *= fac
    L.shared_s[:] *= fac
    dev = device_layer(L)
    o_idx, o_w, _, _ = oracle.route(L.x, L.wg, L.bias, sh.k)
    o_union = oracle.union(o_idx, sh.E)
    for mode, tol in ((m.MOE_MODE_PREFILL, TOL_PREFILL), (m.MOE_MODE_DECODE, TOL_DECODE)):
        t = run_steps(dev, sh.k, teacher_idx=o_idx, teacher_w=o_w, mode=mode)
        assert t["err"] == 0, f"mode {mode}: device error {t['err']}"
        assert np.isfinite(t["y_pair"]).all() and np.isfinite(t["y_shared"]).all()
        y_sh = oracle.expert_ffn_tokens(L.x, np.arange(sh.T), L.shared_q, L.shared_s, sh.d, sh.f, sh.G)
        assert rel_max_err(t["y_shared"], y_sh) <= tol, f"mode {mode} shared"
        for e in o_union["uniq"][:o_union["n_uniq"]]:
            lo, hi = o_union["offsets"][e], o_union["offsets"][e + 1]
            toks = o_union["sorted_pair"][lo:hi] // sh.k
            y = oracle.expert_ffn_tokens(L.x, toks, L.q_base[e], L.s_base[e], sh.d, sh.f, sh.G)
            assert rel_max_err(t["y_pair"][lo:hi], y) <= tol, f"mode {mode} expert {e}"


def test_prefill_flags_scales_beyond_its_row_range():
    """A group scale 2^20 times its row's first group scale is beyond the prefill path's fp16
    weights: the device error word says so (MOE_DEVERR_SCALE_RANGE)."""
    m = moe()
    sh = Shape("scale_spread", E=8, k=2, d=256, f=128, T=16)
    L = workloads.layer_inputs(sh, seed=6, threads=4)
    G, d = sh.G, sh.d
    L.s_base[3, 5 * (d // G) + 2] *= np.float32(2.0 ** 20)   # gate row 5 of expert 3, group 2
    dev = device_layer(L)
    idx = np.tile(np.array([[3, 0]], np.int32), (sh.T, 1))
    t = run_steps(dev, sh.k, teacher_idx=idx, teacher_w=np.full((sh.T, 2), 0.5), mode=m.MOE_MODE_PREFILL)
    assert t["err"] & m.MOE_DEVERR_SCALE_RANGE
    assert m.device_error(m.MOE_DEVERR_SCALE_RANGE) == m.MOE_ERR_UNSUPPORTED


# ---------------------------------------------------------- group size 64 ----
G64 = [
    Shape("g64_ragged", E=16, k=4, d=1024, f=512, T=37, G=64, bias="normal"),
    Shape("g64_t1", E=12, k=3, d=2048, f=256, T=1, G=64, bias="normal"),
    Shape("g64_multi_pass", E=8, k=2, d=256, f=256, T=300, G=64),
]


@pytest.mark.parametrize("shape", G64, ids=lambda s: s.name)
def test_group_size_64_parity(shape):
    """One scale per 64 elements (the gs64 container) on both FFN paths and the hybrid, against the oracle on its
    routing; and bit for bit equal to the same layer stated with G = 32 and paired scales."""
    from moe_testlib import TOL_PREFILL
    m = moe()
    L = workloads.layer_inputs(shape, seed=5, threads=4)
    dev = device_layer(L)
    k = shape.k
    o_idx, o_w, _, _ = oracle.route(L.x, L.wg, L.bias, k)
    o_union = oracle.union(o_idx, shape.E)
    _, _, o_out = oracle_layer(L).dense()
    # the same layer with G = 32: each scale repeated for both halves of its group
    n32 = workloads.expert_s_count(shape.d, shape.f, 32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    s32 = np.repeat(L.s_base.reshape(shape.E, -1), 2, axis=1).reshape(-1)
    lw32 = m.LayerWeights(dev["layer"].q_base, t(s32), dev["layer"].shared_q, t(np.repeat(L.shared_s, 2)),
                          E=shape.E, d=shape.d, f=shape.f, G=32)
    assert s32.size == shape.E * n32
    for mode, tol in ((m.MOE_MODE_DECODE, TOL_DECODE), (m.MOE_MODE_PREFILL, TOL_PREFILL),
                      (m.MOE_MODE_HYBRID, TOL_PREFILL)):
        r = run_steps(dev, k, teacher_idx=o_idx, teacher_w=o_w, mode=mode)
        assert r["err"] == 0
        check_union_equal(r, o_union, shape.E)
        assert rel_max_err(r["out"], o_out) <= tol, f"mode {mode}"
        y_sh = oracle.expert_ffn_tokens(L.x, np.arange(shape.T), L.shared_q, L.shared_s, shape.d, shape.f, 64)
        assert rel_max_err(r["y_shared"], y_sh) <= tol
        for e in o_union["uniq"][:o_union["n_uniq"]]:
            lo, hi = o_union["offsets"][e], o_union["offsets"][e + 1]
            y = oracle.expert_ffn_tokens(L.x, o_union["sorted_pair"][lo:hi] // k, L.q_base[e], L.s_base[e],
                                         shape.d, shape.f, 64)
            assert rel_max_err(r["y_pair"][lo:hi], y) <= tol, f"mode {mode} expert {e}"
        r32 = run_steps(dict(dev, layer=lw32), k, teacher_idx=o_idx, teacher_w=o_w, mode=mode)
        assert r32["err"] == 0
        assert np.array_equal(r["y_pair"][:o_union["offsets"][shape.E]], r32["y_pair"][:o_union["offsets"][shape.E]])
        assert np.array_equal(r["y_shared"], r32["y_shared"]) and np.array_equal(r["out"], r32["out"])


def test_group_size_64_needs_f_multiple_of_256():
    m = moe()
    sh = Shape("g64_bad", E=4, k=2, d=256, f=384, T=3, G=64)
    L = workloads.layer_inputs(sh, seed=1, threads=2)
    dev = device_layer(L)
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward(dev["x"], dev["wg"], None, dev["layer"], sh.k)
    assert ei.value.status == m.MOE_ERR_UNSUPPORTED
