"""The expert tier (Place and Overlap): routed experts in page-locked host
memory, a cache of them in device memory.  Placement decides speed only, so
every call must give the same bits as the layer with all experts resident, at
any residency, on both FFN paths; the tier's counts must match the unions."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_testlib import TOL_DECODE, TOL_PREFILL, device_layer, host, moe, oracle_layer, rel_max_err

pytestmark = pytest.mark.gpu

Shape = workloads.Shape


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_sigmoid_gb300 import build
    build.build()


def _tier(m, L, n_slots):
    sh = L.shape
    hq = torch.from_numpy(np.ascontiguousarray(L.q_base.reshape(-1))).pin_memory()
    hs = torch.from_numpy(np.ascontiguousarray(L.s_base.reshape(-1))).pin_memory()
    return m.ExpertTier(hq, hs, E=sh.E, d=sh.d, f=sh.f, n_slots=n_slots, G=sh.G)


@pytest.mark.parametrize("mode_name", ["MOE_MODE_DECODE", "MOE_MODE_PREFILL"])
@pytest.mark.parametrize("T,n_slots", [(1, 4), (1, 9), (5, 16), (37, 16)])
def test_tier_matches_resident_layer(mode_name, T, n_slots):
    m = moe()
    mode = getattr(m, mode_name)
    sh = Shape("tier", E=16, k=4, d=1024, f=256, T=T, bias="normal")
    L = workloads.layer_inputs(sh, seed=T + n_slots, threads=4)
    dev = device_layer(L)
    tier = _tier(m, L, n_slots)
    copy = torch.cuda.Stream()
    hits_t = torch.zeros(sh.E, dtype=torch.int64, device="cuda")
    hits_r = torch.zeros(sh.E, dtype=torch.int64, device="cuda")
    uniq_total = 0
    res = torch.from_numpy(workloads.activations(T, sh.d, seed=9)).cuda()
    for call in range(6):   # consecutive calls: hits, misses and evictions in between
        x = torch.from_numpy(workloads.activations(T, sh.d, seed=100 + call)).cuda()
        idx = torch.empty((T, sh.k), dtype=torch.int32, device="cuda")
        out_t, err_t = m.moe_layer_forward_tier(x, dev["wg"], dev["bias"], tier, dev["layer"].shared_q,
                                                dev["layer"].shared_s, sh.k, mode=mode, residual=res,
                                                topk_idx=idx, hits=hits_t, copy_stream=copy)
        out_r, err_r = m.moe_layer_forward(x, dev["wg"], dev["bias"], dev["layer"], sh.k, mode=mode, residual=res,
                                           hits=hits_r)
        torch.cuda.synchronize()
        assert int(host(err_t)[0]) == 0 and int(host(err_r)[0]) == 0
        assert np.array_equal(host(out_t), host(out_r)), f"call {call}"
        uniq_total += int(np.unique(host(idx)).size)
        if call == 0:
            # and the layer itself against the oracle (decode tolerance or prefill tolerance)
            o_idx, _, _, _ = oracle.route(host(x), L.wg, L.bias, sh.k)
            same = (host(idx) == o_idx).all(axis=1)
            _, _, o_out = oracle_layer(L, x=host(x), res=host(res)).dense()
            tol = TOL_DECODE if mode == m.MOE_MODE_DECODE else TOL_PREFILL
            assert rel_max_err(host(out_t)[same], o_out[same]) <= tol
    assert np.array_equal(host(hits_t), host(hits_r))
    st = tier.stats()
    blk = m.expert_q_bytes(sh.d, sh.f) + 4 * m.expert_s_count(sh.d, sh.f)
    assert st["calls"] == 6 and st["bytes_copied"] == st["misses"] * blk
    if n_slots < sh.E:
        assert st["hits"] + st["misses"] == uniq_total
    else:
        # every expert copied at most once; once all have slots, calls skip the host round trip and
        # count no hits
        assert st["misses"] <= sh.E and st["hits"] + st["misses"] <= uniq_total
    tier.close()


def test_tier_pins_the_learned_hot_set_and_refuses_overfull_batches():
    m = moe()
    sh = Shape("tier_pin", E=16, k=4, d=1024, f=256, T=1, bias="zipf")
    L = workloads.layer_inputs(sh, seed=4, threads=4)
    dev = device_layer(L)
    tier = _tier(m, L, 8)
    copy = torch.cuda.Stream()
    hits = torch.zeros(sh.E, dtype=torch.int64, device="cuda")
    xs = [torch.from_numpy(workloads.activations(1, sh.d, seed=200 + i)).cuda() for i in range(12)]
    for x in xs[:6]:   # learn
        m.moe_layer_forward_tier(x, dev["wg"], dev["bias"], tier, dev["layer"].shared_q, dev["layer"].shared_s,
                                 sh.k, hits=hits, copy_stream=copy)
    torch.cuda.synchronize()
    hot = m.usage_top(host(hits).astype(np.uint64), 3)
    tier.pin(hot, copy_stream=copy)
    ex, pn = tier.slots()
    assert set(ex[pn].tolist()) == set(hot.tolist())
    before = tier.stats()
    for x in xs[6:]:
        idx = torch.empty((1, sh.k), dtype=torch.int32, device="cuda")
        out_t, err = m.moe_layer_forward_tier(x, dev["wg"], dev["bias"], tier, dev["layer"].shared_q,
                                              dev["layer"].shared_s, sh.k, topk_idx=idx, copy_stream=copy)
        out_r, _ = m.moe_layer_forward(x, dev["wg"], dev["bias"], dev["layer"], sh.k)
        torch.cuda.synchronize()
        assert int(host(err)[0]) == 0 and np.array_equal(host(out_t), host(out_r))
        ex, pn = tier.slots()
        assert set(ex[pn].tolist()) == set(hot.tolist())   # pinned experts never leave
    after = tier.stats()
    assert after["calls"] - before["calls"] == 6
    # a batch needing more experts than the unpinned slots is refused, nothing copied
    big = torch.from_numpy(workloads.activations(8, sh.d, seed=7)).cuda()
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward_tier(big, dev["wg"], dev["bias"], tier, dev["layer"].shared_q, dev["layer"].shared_s,
                                 sh.k, copy_stream=copy)
    assert ei.value.status == m.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    tier.unpin_all()
    _, pn = tier.slots()
    assert not pn.any()
    tier.close()


def test_tier_prefetch_all_takes_the_device_only_path():
    """With every expert prefetched into the slots no call can miss: calls skip the host round trip
    (no hits counted, nothing copied) and still give the resident layer's bits."""
    m = moe()
    sh = Shape("tier_all", E=16, k=4, d=1024, f=256, T=5, bias="normal")
    L = workloads.layer_inputs(sh, seed=8, threads=4)
    dev = device_layer(L)
    tier = _tier(m, L, sh.E)
    copy = torch.cuda.Stream()
    tier.prefetch(np.arange(sh.E)[::-1], copy_stream=copy)
    ex, pn = tier.slots()
    assert sorted(ex.tolist()) == list(range(sh.E)) and not pn.any()
    before = tier.stats()
    for i in range(4):
        x = torch.from_numpy(workloads.activations(sh.T, sh.d, seed=300 + i)).cuda()
        for mode in (m.MOE_MODE_DECODE, m.MOE_MODE_PREFILL):
            out_t, err = m.moe_layer_forward_tier(x, dev["wg"], dev["bias"], tier, dev["layer"].shared_q,
                                                  dev["layer"].shared_s, sh.k, mode=mode, copy_stream=copy)
            out_r, _ = m.moe_layer_forward(x, dev["wg"], dev["bias"], dev["layer"], sh.k, mode=mode)
            torch.cuda.synchronize()
            assert int(host(err)[0]) == 0 and np.array_equal(host(out_t), host(out_r))
    after = tier.stats()
    assert after["calls"] - before["calls"] == 8
    assert after["hits"] == before["hits"] and after["misses"] == before["misses"]
    assert after["bytes_copied"] == before["bytes_copied"]
    # the tier has no hybrid path: the mode is refused before anything is enqueued
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward_tier(x, dev["wg"], dev["bias"], tier, dev["layer"].shared_q, dev["layer"].shared_s,
                                 sh.k, mode=m.MOE_MODE_HYBRID, copy_stream=copy)
    assert ei.value.status == m.MOE_ERR_INVALID_ARG
    assert tier.stats()["calls"] == after["calls"]
    tier.close()
