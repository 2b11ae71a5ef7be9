"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a closed form, an invariant, an exhaustive
enumeration, brute force on tiny inputs, or sizes the pages print -- chosen so
that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from conftest import read_golden

LN3 = math.log(3.0)          # sigmoid(ln 3) = 3/4 exactly in real arithmetic


# ------------------------------------------------------------------ int4 ----

def test_unpack_golden_bytes():
    for hexbyte, lo, hi in read_golden("int4_nibbles.txt"):
        v = oracle.int4_unpack(np.array([int(hexbyte, 16)], np.uint8), 2)
        assert (int(v[0]), int(v[1])) == (int(lo), int(hi)), hexbyte


def test_pack_unpack_exhaustive():
    # all 256 bytes round-trip through unpack -> pack
    q = np.arange(256, dtype=np.uint8)
    v = oracle.int4_unpack(q, 512)
    assert v.min() == -8 and v.max() == 7
    q2, bad = oracle.int4_pack(v)
    assert bad == 0 and np.array_equal(q, q2)
    # all 16 x 16 value pairs round-trip through pack -> unpack
    lo, hi = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    pairs = np.stack([lo.ravel(), hi.ravel()], axis=1).astype(np.int8).ravel()
    q3, bad = oracle.int4_pack(pairs)
    assert bad == 0 and np.array_equal(oracle.int4_unpack(q3, pairs.size), pairs)
    # each nibble position takes each of the 16 values exactly 16 times
    assert all(np.sum(v[0::2] == x) == 16 and np.sum(v[1::2] == x) == 16 for x in range(-8, 8))


def test_pack_flags_out_of_range():
    _, bad = oracle.int4_pack(np.array([8, -9, 7, -8], np.int8))
    assert bad == 2


def test_random_round_trip():
    rng = np.random.default_rng(5)
    v = rng.integers(-8, 8, size=10_000).astype(np.int8)
    q, bad = oracle.int4_pack(v)
    assert bad == 0 and np.array_equal(oracle.int4_unpack(q, v.size), v)


def test_dequant_group_boundaries():
    """deq[r, i] uses scale s[r, i // G]: elements 31 and 32 use different groups."""
    rows, cols, G = 3, 128, 32
    q, _ = oracle.int4_pack(np.ones(rows * cols, np.int8))
    s = (np.arange(rows * cols // G, dtype=np.float32) + 1.0) * np.float32(0.5)
    w = oracle.dequant(q, s, rows, cols, G)
    for r in range(rows):
        for i in (0, 31, 32, 63, 64, 127):
            assert w[r, i] == s[r * (cols // G) + i // G]
    # value -8 at the last element of a row, scale 2^-3 -> -1 exactly
    v = np.zeros(rows * cols, np.int8)
    v[cols - 1] = -8
    q, _ = oracle.int4_pack(v)
    w = oracle.dequant(q, np.full(rows * cols // G, 0.125, np.float32), rows, cols, G)
    assert w[0, cols - 1] == -1.0 and np.count_nonzero(w) == 1


def test_expert_bytes_match_page_sizes():
    g = {row[0]: (float(row[1]), float(row[2])) for row in read_golden("page_sizes.txt")}
    d, f = 6144, 2048
    qb = oracle.expert_q_bytes(d, f)
    assert qb == workloads.expert_q_bytes(d, f)
    val, tol = g["expert_bytes_mb"]
    assert abs(qb / 1e6 - val) <= tol
    layers, E = int(g["layers"][0]), int(g["experts_per_layer"][0])
    assert layers * E + E == int(g["experts_total"][0])          # 75 x 256 + MTP head
    val, tol = g["experts_on_disk_gb"]
    assert abs(int(g["experts_total"][0]) * qb / 1e9 - val) <= tol
    # ~11 GB of routed experts per token across 75 layers fixes k = 8 at this size
    val, tol = g["routed_gb_per_token"]
    k = workloads.WORKLOADS["decode"].k
    assert abs(layers * k * qb / 1e9 - val) <= tol
    assert all(abs(layers * kk * qb / 1e9 - val) > tol for kk in (1, 2, 4, 6, 7, 9, 10))


# ---------------------------------------------------------------- route ----

def test_logits_one_hot_and_linearity():
    rng = np.random.default_rng(1)
    E, d = 16, 64
    wg = rng.standard_normal((E, d)).astype(np.float32)
    x = np.zeros((3, d), np.float32)
    x[0, 5] = 1.0
    x[1, 63] = 1.0
    x[2, 0] = -2.0
    l = oracle.router_logits(x, wg)
    assert np.array_equal(l[0], wg[:, 5].astype(np.float64))
    assert np.array_equal(l[1], wg[:, 63].astype(np.float64))
    assert np.array_equal(l[2], -2.0 * wg[:, 0].astype(np.float64))


def test_sigmoid_scores_closed_forms():
    # logit 0 -> score 1/2; logit ln 3 -> score 3/4 (one-hot x picks the logit)
    E, d = 4, 8
    wg = np.zeros((E, d), np.float32)
    wg[1, 2] = np.float32(LN3)
    x = np.zeros((1, d), np.float32)
    x[0, 2] = 1.0
    idx, w, logits, keys = oracle.route(x, wg, None, k=E, normalize=0)
    assert idx[0, 0] == 1 and abs(w[0, 0] - 0.75) < 1e-7   # ln 3 rounded to fp32
    assert list(idx[0, 1:]) == [0, 2, 3] and np.all(w[0, 1:] == 0.5)


def brute_force_topk(keys_row, k):
    order = sorted(range(len(keys_row)), key=lambda e: (-keys_row[e], e))
    return order[:k]


@pytest.mark.parametrize("E,k,bias_kind", [(8, 2, "zero"), (16, 4, "normal"), (64, 8, "zipf"),
                                           (256, 8, "normal"), (9, 9, "normal")])
def test_topk_equals_brute_force_sort(E, k, bias_kind):
    rng = np.random.default_rng(E * 10 + k)
    T, d = 40, 48
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (rng.standard_normal((E, d)) * 0.3).astype(np.float32)
    bias = workloads.selection_bias(E, bias_kind, seed=3) if bias_kind != "zipf" else \
        workloads.selection_bias(E, "zipf", seed=3)
    idx, w, logits, keys = oracle.route(x, wg, bias, k=k, normalize=0)
    for t in range(T):
        assert list(idx[t]) == brute_force_topk(list(keys[t]), k)
        # combine weights are the unbiased sigmoid scores of the chosen experts
        for j in range(k):
            assert w[t, j] == pytest.approx(1.0 / (1.0 + math.exp(-logits[t, idx[t, j]])), rel=1e-15)


def test_topk_without_bias_is_topk_of_logits():
    rng = np.random.default_rng(2)
    T, d, E, k = 50, 32, 32, 5
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = rng.standard_normal((E, d)).astype(np.float32)
    idx, _, logits, _ = oracle.route(x, wg, None, k=k)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    assert np.array_equal(np.sort(idx, axis=1), np.sort(ref, axis=1))


def test_ties_go_to_lower_expert_id():
    d, E = 8, 6
    wg = np.zeros((E, d), np.float32)
    wg[[1, 3, 4], 0] = 1.0          # experts 1, 3, 4 tie on the highest score
    x = np.zeros((1, d), np.float32)
    x[0, 0] = 1.0
    idx, _, _, _ = oracle.route(x, wg, None, k=4)
    assert list(idx[0]) == [1, 3, 4, 0]


def test_bias_selects_but_does_not_weight():
    d, E = 4, 4
    wg = np.zeros((E, d), np.float32)
    wg[:, 0] = np.array([2.0, 1.0, 0.0, -1.0], np.float32)
    x = np.zeros((1, d), np.float32)
    x[0, 0] = 1.0
    bias = np.array([0.0, 0.0, 0.0, 1.0], np.float32)   # lifts the weakest expert to the top
    idx, w, _, _ = oracle.route(x, wg, bias, k=2, normalize=0)
    assert list(idx[0]) == [3, 0]
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.e), rel=1e-15)     # sigmoid(-1)


@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_normalized_weights_sum_to_route_scale(scale):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((20, 16)).astype(np.float32)
    wg = rng.standard_normal((10, 16)).astype(np.float32)
    _, w, _, _ = oracle.route(x, wg, None, k=3, normalize=1, route_scale=scale)
    assert np.allclose(w.sum(axis=1), scale, rtol=0, atol=4e-16 * scale)
    _, w1, _, _ = oracle.route(x, wg, None, k=1, normalize=1, route_scale=scale)
    assert np.all(np.abs(w1 - scale) <= np.spacing(scale))    # within 1 ulp


def test_k_equals_E_returns_all_in_key_order():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 12)).astype(np.float32)
    wg = rng.standard_normal((7, 12)).astype(np.float32)
    idx, _, _, keys = oracle.route(x, wg, None, k=7)
    for t in range(5):
        assert sorted(idx[t]) == list(range(7))
        assert all(keys[t, idx[t, j]] >= keys[t, idx[t, j + 1]] for j in range(6))


# ---------------------------------------------------------------- union ----

def check_union_invariants(idx, E, u):
    T, k = idx.shape
    P = T * k
    flat = idx.reshape(-1)
    assert u["n_uniq"] == len(set(flat.tolist()))
    assert int(u["counts"].sum()) == P and u["offsets"][0] == 0 and u["offsets"][E] == P
    assert np.array_equal(np.diff(u["offsets"]), u["counts"])
    assert sorted(u["perm"].tolist()) == list(range(P))                  # bijection
    assert np.array_equal(u["sorted_pair"][u["perm"]], np.arange(P))    # inverse
    assert list(u["uniq"][:u["n_uniq"]]) == sorted(set(flat.tolist()))
    # brute force: Python's stable sort of pair ids by expert
    assert u["sorted_pair"].tolist() == sorted(range(P), key=lambda p: flat[p])
    for e in range(E):
        grp = u["sorted_pair"][u["offsets"][e]:u["offsets"][e + 1]]
        assert np.all(flat[grp] == e) and np.all(np.diff(grp) > 0)


@pytest.mark.parametrize("T,k,E", [(1, 8, 256), (16, 2, 8), (64, 8, 256), (333, 3, 17)])
def test_union_invariants(T, k, E):
    rng = np.random.default_rng(T + k + E)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    u = oracle.union(idx, E)
    check_union_invariants(idx, E, u)
    if T == 1:
        assert u["n_uniq"] == k


def test_union_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.union(np.array([[0, 8]], np.int32), 8)


def test_hits_accumulate():
    rng = np.random.default_rng(8)
    E, T, k = 32, 10, 4
    h = np.zeros(E, np.uint64)
    for _ in range(3):
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        u = oracle.union(idx, E)
        before = h.copy()
        oracle.hits(u["counts"], h)
        assert int((h - before).sum()) == T * k
        assert np.array_equal(h - before, np.bincount(idx.ravel(), minlength=E).astype(np.uint64))


# ------------------------------------------------------------------ FFN ----

def pack_matrix(v):
    q, bad = oracle.int4_pack(np.asarray(v, np.int8).ravel())
    assert bad == 0
    return q


def expert_from_values(vg, vu, vd, sg, su, sd):
    """Expert block from int values gate [f][d], up [f][d], down [d][f] and scale arrays."""
    q = np.concatenate([pack_matrix(vg), pack_matrix(vu), pack_matrix(vd)])
    s = np.concatenate([np.ravel(sg), np.ravel(su), np.ravel(sd)]).astype(np.float32)
    return q, s


def test_ffn_one_hot_expert_reproduces_input_slice():
    """Gate row r one-hot at a, up row r one-hot at b, down column r one-hot at c:
    y_c = silu(x_a) * x_b and every other output is 0."""
    d, f, G = 64, 32, 32
    a, b, c, r = 7, 40, 19, 11
    vg = np.zeros((f, d)); vg[r, a] = 1
    vu = np.zeros((f, d)); vu[r, b] = 1
    vd = np.zeros((d, f)); vd[c, r] = 1
    ones = lambda rows, cols: np.ones(rows * cols // G)
    q, s = expert_from_values(vg, vu, vd, ones(f, d), ones(f, d), ones(d, f))
    x = np.zeros(d, np.float32)
    x[a] = np.float32(LN3)
    x[b] = 3.0
    y = oracle.expert_ffn(x, q, s, d, f, G)
    expect = float(np.float32(LN3)) * (1.0 / (1.0 + 1.0 / 3.0 * math.exp(LN3 - float(np.float32(LN3))))) * 3.0
    assert y[c] == pytest.approx(expect, rel=1e-15)
    assert np.count_nonzero(y) == 1
    # powers of two in the up and down scales scale the output exactly
    su = np.ones(f * d // G); su[r * (d // G) + b // G] = 0.25
    sd = np.ones(d * f // G); sd[c * (f // G) + r // G] = 8.0
    q2, s2 = expert_from_values(vg, vu, vd, ones(f, d), su, sd)
    assert oracle.expert_ffn(x, q2, s2, d, f, G)[c] == y[c] * 2.0
    # all-zero weights give zero
    z = np.zeros_like(q)
    assert not np.any(oracle.expert_ffn(x, z, s, d, f, G))


def test_ffn_permutation_experts_closed_form():
    """Gate, up and down as distinct permutation matrices (d = f): each output is
    silu(x[p_g[r]]) * x[p_u[r]] routed through the down permutation.  A transposed
    operand or a swapped index breaks the equality."""
    d = f = 64
    G = 32
    rng = np.random.default_rng(9)
    pg, pu, pd = rng.permutation(d), rng.permutation(d), rng.permutation(d)
    vg = np.zeros((f, d)); vg[np.arange(f), pg] = 1          # g_r = x[pg[r]]
    vu = np.zeros((f, d)); vu[np.arange(f), pu] = -1         # u_r = -x[pu[r]]
    vd = np.zeros((d, f)); vd[np.arange(d), pd] = 1          # y_c = h[pd[c]]
    ones = np.ones(d * f // G)
    q, s = expert_from_values(vg, vu, vd, ones, ones * 2.0, ones)   # up scale 2: u_r = -2 x[pu[r]]
    x = rng.standard_normal(d).astype(np.float32)
    y = oracle.expert_ffn(x, q, s, d, f, G)
    xd = x.astype(np.float64)
    for c in range(d):
        r = pd[c]
        g = xd[pg[r]]
        assert y[c] == pytest.approx(g / (1.0 + math.exp(-g)) * (-2.0 * xd[pu[r]]), rel=1e-14, abs=1e-300)


def test_ffn_row_permutation_invariance():
    """Permuting the f rows of gate and up together with the columns of down
    leaves the expert's output unchanged (up to fp64 summation order)."""
    d, f, G = 64, 96, 32
    rng = np.random.default_rng(10)
    vg = rng.integers(-8, 8, (f, d)); vu = rng.integers(-8, 8, (f, d)); vd = rng.integers(-8, 8, (d, f))
    sg = rng.uniform(0.01, 0.02, (f, d // G)); su = rng.uniform(0.01, 0.02, (f, d // G))
    sd = np.full((d, f // G), 0.03)                           # uniform down scales survive a column permutation
    q, s = expert_from_values(vg, vu, vd, sg, su, sd)
    x = rng.standard_normal(d).astype(np.float32)
    y = oracle.expert_ffn(x, q, s, d, f, G)
    p = rng.permutation(f)
    q2, s2 = expert_from_values(vg[p], vu[p], vd[:, p], sg[p], su[p], sd)
    y2 = oracle.expert_ffn(x, q2, s2, d, f, G)
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-14)
    assert np.max(np.abs(y)) > 1e-3


# ---------------------------------------------------------------- layer ----

def tiny_layer(seed=0, normalize=1, route_scale=1.0, res=False, **kw):
    sh = workloads.WORKLOADS["tiny"]
    L = workloads.layer_inputs(sh, seed=seed, threads=1)
    r = workloads.activations(sh.T, sh.d, seed + 99) if res else None
    return oracle.Layer(L.x, L.wg, L.bias, L.q_base, L.s_base, L.shared_q, L.shared_s,
                        d=sh.d, f=sh.f, E=sh.E, k=sh.k, G=sh.G, normalize=normalize,
                        route_scale=route_scale, res=r, **kw), L


@pytest.mark.parametrize("normalize,res", [(1, False), (0, True)])
def test_dense_path_equals_union_path_bitwise(normalize, res):
    lay, _ = tiny_layer(normalize=normalize, res=res)
    idx, w, out = lay.dense()
    u = lay.union_path()
    assert np.array_equal(idx, u["idx"]) and np.array_equal(w, u["w"])
    assert np.array_equal(out, u["out"])
    check_union_invariants(idx, lay.E, u)


def test_brute_force_tiny_layer():
    """Every expert evaluated densely; mask and weights from a Python sort."""
    lay, L = tiny_layer(res=True)
    sh = workloads.WORKLOADS["tiny"]
    qb, sc = workloads.expert_q_bytes(sh.d, sh.f), workloads.expert_s_count(sh.d, sh.f, sh.G)
    logits = lay.x.astype(np.float64) @ lay.wg.astype(np.float64).T
    idx, w, out = lay.dense()
    for t in range(sh.T):
        scores = [1.0 / (1.0 + math.exp(-v)) for v in logits[t]]
        chosen = brute_force_topk(scores, sh.k)             # bias is 0 in this workload
        assert list(idx[t]) == chosen
        tot = sum(scores[e] for e in chosen)
        ys = [oracle.expert_ffn(lay.x[t], L.q_base[e], L.s_base[e], sh.d, sh.f, sh.G) for e in range(sh.E)]
        expect = lay.res[t].astype(np.float64) + oracle.expert_ffn(lay.x[t], L.shared_q, L.shared_s, sh.d, sh.f, sh.G)
        for e in range(sh.E):
            m = scores[e] / tot if e in chosen else 0.0
            expect = expect + m * ys[e]
        assert np.allclose(out[t], expect, rtol=1e-12, atol=1e-12)
    assert qb * sh.E == L.q_base.size and sc * sh.E == L.s_base.size


def test_identical_experts_make_routing_irrelevant():
    lay, L = tiny_layer(res=True)
    sh = workloads.WORKLOADS["tiny"]
    q_same = np.tile(L.q_base[3], (sh.E, 1))
    s_same = np.tile(L.s_base[3], (sh.E, 1))
    lay2 = oracle.Layer(L.x, L.wg, L.bias, q_same, s_same, L.shared_q, L.shared_s, d=sh.d, f=sh.f,
                        E=sh.E, k=sh.k, G=sh.G, normalize=1, res=lay.res)
    _, _, out = lay2.dense()
    for t in range(sh.T):
        y = oracle.expert_ffn(L.x[t], L.q_base[3], L.s_base[3], sh.d, sh.f, sh.G)
        ys = oracle.expert_ffn(L.x[t], L.shared_q, L.shared_s, sh.d, sh.f, sh.G)
        assert np.allclose(out[t], lay.res[t] + ys + y, rtol=1e-13, atol=1e-13)


def test_zero_route_scale_leaves_residual_plus_shared():
    lay, L = tiny_layer(route_scale=0.0, res=True)
    sh = workloads.WORKLOADS["tiny"]
    _, _, out = lay.dense()
    for t in range(sh.T):
        ys = oracle.expert_ffn(L.x[t], L.shared_q, L.shared_s, sh.d, sh.f, sh.G)
        assert np.array_equal(out[t], lay.res[t].astype(np.float64) + ys)


def test_k1_normalized_adds_scaled_expert():
    sh = workloads.WORKLOADS["tiny"]
    L = workloads.layer_inputs(sh, seed=4, threads=1)
    lay = oracle.Layer(L.x, L.wg, L.bias, L.q_base, L.s_base, L.shared_q, L.shared_s, d=sh.d, f=sh.f,
                       E=sh.E, k=1, G=sh.G, normalize=1, route_scale=2.0)
    idx, w, out = lay.dense()
    assert np.all(w == 2.0)
    for t in range(sh.T):
        e = idx[t, 0]
        y = oracle.expert_ffn(L.x[t], L.q_base[e], L.s_base[e], sh.d, sh.f, sh.G)
        ys = oracle.expert_ffn(L.x[t], L.shared_q, L.shared_s, sh.d, sh.f, sh.G)
        assert np.allclose(out[t], ys + 2.0 * y, rtol=1e-14, atol=1e-14)


def test_token_subset_matches_full_layer():
    lay, _ = tiny_layer(res=True)
    idx, w, out = lay.dense()
    sel = np.array([15, 0, 7], np.int32)
    i2, w2, o2 = lay.tokens(sel)
    assert np.array_equal(i2, idx[sel]) and np.array_equal(w2, w[sel]) and np.array_equal(o2, out[sel])


def test_workload_generator_is_seeded_and_layer_independent():
    sh = workloads.WORKLOADS["tiny"]
    a = workloads.layer_inputs(sh, seed=0, threads=2)
    b = workloads.layer_inputs(sh, seed=0, threads=3)
    c = workloads.layer_inputs(sh, seed=0, layer=1, threads=2)
    assert np.array_equal(a.q_base, b.q_base) and np.array_equal(a.s_base, b.s_base)
    assert np.array_equal(a.x, b.x) and not np.array_equal(a.q_base, c.q_base)
    q5, s5 = workloads.expert_block(sh.d, sh.f, sh.G, 0, 0, 5)
    assert np.array_equal(q5, a.q_base[5]) and np.array_equal(s5, a.s_base[5])
    # each nibble is uniform over [-8, 7]; scales are lognormal around e^-4
    v = oracle.int4_unpack(a.q_base, a.q_base.size * 2)
    assert v.min() == -8 and v.max() == 7 and abs(v.mean() + 0.5) < 0.02
    assert abs(np.log(a.s_base).mean() + 4.0) < 0.01 and abs(np.log(a.s_base).std() - 0.3) < 0.01


# ------------------------------------------------------------- stack norm ----

def test_rms_norm_closed_forms():
    """Rows worked by hand: a constant row maps to +-1; (3, -4, 0, 0) has RMS 2.5."""
    x = np.array([[2, 2, 2, 2], [-0.5, -0.5, -0.5, -0.5], [3, -4, 0, 0], [0, 0, 0, 0]], np.float32)
    n = oracle.rms_norm(x, eps=0.0)[:3]
    assert np.array_equal(n[:2], np.array([[1, 1, 1, 1], [-1, -1, -1, -1]]))
    assert np.allclose(n[2], [1.2, -1.6, 0, 0], rtol=0, atol=1e-15)
    # with eps: c / sqrt(c^2 + eps); an all-zero row stays zero
    e = oracle.rms_norm(x, eps=0.25)
    assert np.allclose(e[0], 2 / np.sqrt(4.25), rtol=0, atol=1e-15)
    assert np.allclose(e[2], np.array([3, -4, 0, 0]) / np.sqrt(6.25 + 0.25), rtol=0, atol=1e-15)
    assert not e[3].any()


def test_rms_norm_invariants():
    """Unit mean square, scale invariance (exact for powers of two) and row independence."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((6, 384)) * rng.uniform(0.1, 100, (6, 1))).astype(np.float32)
    n = oracle.rms_norm(x, eps=0.0)
    assert np.allclose(np.mean(n * n, axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.array_equal(oracle.rms_norm(x * np.float32(64.0), eps=0.0), n)
    assert np.array_equal(oracle.rms_norm(x[3:4], eps=0.0), n[3:4])
    assert np.all(np.sign(n) == np.sign(x))


# ---------------------------------------------------- routing from logits ----

def test_route_from_logits_matches_route_and_brute_force():
    """Routing given the logits equals routing from x (bit for bit) and a full sort of the keys."""
    rng = np.random.default_rng(21)
    T, d, E, k = 30, 40, 24, 5
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (rng.standard_normal((E, d)) * 0.4).astype(np.float32)
    bias = workloads.selection_bias(E, "normal", seed=5)
    i1, w1, logits, keys = oracle.route(x, wg, bias, k, normalize=1, route_scale=1.5)
    i2, w2, keys2 = oracle.route_from_logits(logits, bias, k, normalize=1, route_scale=1.5)
    assert np.array_equal(i1, i2) and np.array_equal(w1, w2) and np.array_equal(keys, keys2)
    for t in range(T):
        assert list(i2[t]) == brute_force_topk(list(keys2[t]), k)


def test_route_from_logits_hand_worked():
    # sigmoid is monotone: without bias the order is the logits' order, ties to the lower id
    logits = np.array([[0.0, 3.0, -3.0, 1.0, 1.0]])
    idx, w, _ = oracle.route_from_logits(logits, None, 3, normalize=0)
    assert list(idx[0]) == [1, 3, 4]
    # a zero bias array and no bias agree; a bias of +1 on expert 2 lifts it to the top
    idx0, _, _ = oracle.route_from_logits(logits, np.zeros(5, np.float32), 3, normalize=0)
    assert list(idx0[0]) == [1, 3, 4]
    idxb, wb, _ = oracle.route_from_logits(logits, np.array([0, 0, 1, 0, 0], np.float32), 3, normalize=0)
    assert list(idxb[0]) == [2, 1, 3]
    assert wb[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(3.0)), rel=1e-15)   # unbiased score


# ------------------------------------------------------------ top-p cut ----
# Scores sigmoid(ln 3) = 3/4, sigmoid(0) = 1/2, sigmoid(-ln 3) = 1/4 (sum 3/2) give
# hand-worked cut points: p = 0.3 -> 0.45 of mass, reached by the first score;
# p = 0.6 -> 0.9, reached by 3/4 + 1/2 = 5/4; p = 0.9 -> 1.35, only by all three.

HAND_LOGITS = np.array([[math.log(3.0), 0.0, -math.log(3.0), -5.0]])


@pytest.mark.parametrize("p,kept,w_norm", [
    (0.3, [0], [1.0, 0.0, 0.0]),
    (0.6, [0, 1], [0.6, 0.4, 0.0]),
    (0.9, [0, 1, 2], [0.5, 1.0 / 3.0, 1.0 / 6.0]),
    (1.0, [0, 1, 2], [0.5, 1.0 / 3.0, 1.0 / 6.0]),
])
def test_topp_hand_worked(p, kept, w_norm):
    idx, w, _ = oracle.route_from_logits(HAND_LOGITS, None, 3, normalize=1, top_p=p)
    expect_idx = [e if j < len(kept) else -1 for j, e in enumerate([0, 1, 2])]
    assert list(idx[0]) == expect_idx
    assert np.allclose(w[0], w_norm, rtol=1e-14, atol=0)
    idx0, w0, _ = oracle.route_from_logits(HAND_LOGITS, None, 3, normalize=0, top_p=p)
    raw = [0.75, 0.5, 0.25]
    assert np.allclose(w0[0], [raw[j] if j < len(kept) else 0.0 for j in range(3)], rtol=1e-14, atol=0)


def test_topp_one_is_plain_topk_and_tiny_p_keeps_one():
    rng = np.random.default_rng(31)
    T, d, E, k = 25, 32, 40, 8
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (rng.standard_normal((E, d)) * 0.5).astype(np.float32)
    bias = workloads.selection_bias(E, "normal", seed=2)
    i1, w1, _, _ = oracle.route(x, wg, bias, k, normalize=1, route_scale=2.5)
    ip, wp, _, _ = oracle.route(x, wg, bias, k, normalize=1, route_scale=2.5, top_p=1.0)
    assert np.array_equal(i1, ip) and np.array_equal(w1, wp)
    it, wt, _, _ = oracle.route(x, wg, bias, k, normalize=1, route_scale=2.5, top_p=1e-9)
    assert np.array_equal(it[:, 0], i1[:, 0]) and np.all(it[:, 1:] == -1)
    assert np.all(np.abs(wt[:, 0] - 2.5) <= np.spacing(2.5)) and np.all(wt[:, 1:] == 0.0)   # within 1 ulp


def test_topp_keeps_a_prefix_growing_with_p():
    """The kept experts are always a prefix of the top-k list, never fewer as p grows,
    and their normalised weights add up to route_scale."""
    rng = np.random.default_rng(41)
    T, d, E, k = 40, 24, 32, 8
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = rng.standard_normal((E, d)).astype(np.float32)
    full, _, _, _ = oracle.route(x, wg, None, k)
    prev = np.ones(T, np.int64)
    for p in (0.05, 0.2, 0.4, 0.55, 0.7, 0.85, 0.95, 0.999):
        idx, w, _, _ = oracle.route(x, wg, None, k, normalize=1, route_scale=1.0, top_p=p)
        m = (idx >= 0).sum(axis=1)
        assert np.all(m >= 1) and np.all(m >= prev)
        for t in range(T):
            assert list(idx[t, :m[t]]) == list(full[t, :m[t]]) and np.all(idx[t, m[t]:] == -1)
        assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
        prev = m


def test_union_skips_empty_slots():
    idx = np.array([[3, -1, -1], [0, 3, -1], [2, 0, 1]], np.int32)
    u = oracle.union(idx, 4)
    assert u["counts"].tolist() == [2, 1, 1, 2] and u["offsets"][4] == 6
    perm = u["perm"]
    assert perm[1] == -1 and perm[2] == -1 and perm[5] == -1
    valid = [p for p in range(9) if idx.reshape(-1)[p] != -1]
    assert sorted(perm[valid].tolist()) == list(range(6))
    assert np.array_equal(u["sorted_pair"][perm[valid]], np.array(valid))
    with pytest.raises(ValueError):
        oracle.union(np.array([[0, -2]], np.int32), 4)   # only -1 marks an empty slot


@pytest.mark.parametrize("p", [0.3, 0.5])
def test_topp_layer_closed_forms(p):
    """With identical routed experts and normalised weights, the pruned layer is still
    res + shared + route_scale * FFN(x); the dense and union-path evaluations agree bit for bit."""
    lay, L = tiny_layer(res=True)
    sh = workloads.WORKLOADS["tiny"]
    q_same = np.tile(L.q_base[5], (sh.E, 1))
    s_same = np.tile(L.s_base[5], (sh.E, 1))
    lay2 = oracle.Layer(L.x, L.wg, L.bias, q_same, s_same, L.shared_q, L.shared_s, d=sh.d, f=sh.f,
                        E=sh.E, k=sh.k, G=sh.G, normalize=1, route_scale=1.5, res=lay.res, top_p=p)
    idx, _, out = lay2.dense()
    assert (idx == -1).any()          # the cut removes some slots at this p
    for t in range(sh.T):
        y = oracle.expert_ffn(L.x[t], L.q_base[5], L.s_base[5], sh.d, sh.f, sh.G)
        ys = oracle.expert_ffn(L.x[t], L.shared_q, L.shared_s, sh.d, sh.f, sh.G)
        assert np.allclose(out[t], lay.res[t] + ys + 1.5 * y, rtol=1e-13, atol=1e-13)
    lay3 = oracle.Layer(L.x, L.wg, L.bias, L.q_base, L.s_base, L.shared_q, L.shared_s, d=sh.d, f=sh.f,
                        E=sh.E, k=sh.k, G=sh.G, normalize=1, res=lay.res, top_p=p)
    i3, w3, o3 = lay3.dense()
    u = lay3.union_path()
    assert np.array_equal(i3, u["idx"]) and np.array_equal(w3, u["w"]) and np.array_equal(o3, u["out"])
    assert int(u["counts"].sum()) == int((i3 >= 0).sum())


# --------------------------------------------------------- thread count ----

def test_results_do_not_depend_on_thread_count():
    lay, L = tiny_layer(res=True)
    sh = workloads.WORKLOADS["tiny"]
    n0 = oracle.threads()
    try:
        oracle.set_threads(1)
        a = lay.dense()
        ya = oracle.expert_ffn(L.x[3], L.q_base[2], L.s_base[2], sh.d, sh.f, sh.G)
        oracle.set_threads(max(2, n0))
        b = lay.dense()
        yb = oracle.expert_ffn(L.x[3], L.q_base[2], L.s_base[2], sh.d, sh.f, sh.G)
        c = lay.tokens(np.array([4], np.int32))   # one token: rows split over the threads
    finally:
        oracle.set_threads(n0)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
    assert np.array_equal(ya, yb)
    assert np.array_equal(c[2][0], a[2][4])


# ---------------------------------------------------------- group size 64 ----

def test_dequant_group_size_64_boundaries():
    """With G = 64, elements 63 and 64 of a row use different scales, 31 and 32 the same."""
    rows, cols, G = 2, 256, 64
    q, _ = oracle.int4_pack(np.ones(rows * cols, np.int8))
    s = (np.arange(rows * cols // G, dtype=np.float32) + 1.0) * np.float32(0.25)
    w = oracle.dequant(q, s, rows, cols, G)
    for r in range(rows):
        assert w[r, 31] == w[r, 32] == s[r * (cols // G)]
        assert w[r, 63] == s[r * (cols // G)] and w[r, 64] == s[r * (cols // G) + 1]
        assert w[r, 255] == s[r * (cols // G) + 3]


def test_group_64_layer_equals_group_32_with_paired_scales():
    """A layer with one scale per 64 elements is the layer with one scale per 32 elements whose
    two halves of each 64-group share that scale: the same fp64 bits, expert by expert."""
    sh64 = workloads.Shape("g64", E=6, k=2, d=256, f=256, T=5, G=64, bias="normal")
    L = workloads.layer_inputs(sh64, seed=3, threads=2)
    d, f = sh64.d, sh64.f
    n32 = workloads.expert_s_count(d, f, 32)
    s32 = np.repeat(L.s_base.reshape(sh64.E, -1), 2, axis=1).reshape(sh64.E, n32)
    sh32 = np.repeat(L.shared_s, 2)
    a = oracle.Layer(L.x, L.wg, L.bias, L.q_base, L.s_base, L.shared_q, L.shared_s, d=d, f=f, E=sh64.E,
                     k=sh64.k, G=64).dense()
    b = oracle.Layer(L.x, L.wg, L.bias, L.q_base, s32, L.shared_q, sh32, d=d, f=f, E=sh64.E, k=sh64.k,
                     G=32).dense()
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
    # the group size is read: the G = 64 scales taken as G = 32 scales (half of the expert's scale
    # array, each used for 32 elements) give another result
    e = oracle.expert_ffn(L.x[0], L.q_base[1], L.s_base[1], d, f, 64)
    wrong = oracle.expert_ffn(L.x[0], L.q_base[1], np.concatenate([L.s_base[1], L.s_base[1]]), d, f, 32)
    assert not np.array_equal(wrong, e)
