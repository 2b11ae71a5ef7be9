"""moe_expert_ffn_int4_noalloc: the expert FFN for callers that cannot allocate
device memory (a host framework that owns all device memory, or a
latency-critical caller that cannot afford cudaMalloc/cudaFree).  Its scratch
is the library's static 8 MiB device array instead of a caller workspace.

Checked through the C ABI against the existing workspace entry point, on two
calls in a row (the second call finds the first call's leftovers in the shared
array), on the decode path and with the prefill path forced.  Both entry points
run the same kernels on the same inputs, so their outputs must be bit-identical:
a scratch-aliasing error cannot hide under a tolerance.  This file is collected
last so that a failure here stops a -x run only after every other test has run.
"""
import numpy as np
import pytest
import torch

import workloads
from moe_testlib import device_layer, host, moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_sigmoid_gb300 import build
    build.build()
    return moe()


def _routed(m, shape, seed):
    L = workloads.layer_inputs(shape, seed=seed, threads=4)
    dev = device_layer(L)
    idx, _, _ = m.moe_route(dev["x"], dev["wg"], dev["bias"], shape.k)
    un = m.moe_union(idx, shape.E)
    return dev, un


@pytest.mark.parametrize("mode_name", ["MOE_MODE_AUTO", "MOE_MODE_PREFILL"])
def test_noalloc_ffn_matches_workspace_ffn_on_two_calls(m, mode_name):
    mode = getattr(m, mode_name)
    shapes = [workloads.Shape("na_a", E=16, k=4, d=1024, f=384, T=37, bias="normal"),
              workloads.Shape("na_b", E=8, k=2, d=256, f=128, T=5)]
    for i, sh in enumerate(shapes):            # two different calls in a row
        dev, un = _routed(m, sh, seed=10 + i)
        ref_pair, ref_sh, ref_err = m.moe_expert_ffn_int4(dev["x"], dev["layer"], un, sh.k, mode)
        got_pair, got_sh, got_err = m.moe_expert_ffn_int4_noalloc(dev["x"], dev["layer"], un, sh.k, mode)
        torch.cuda.synchronize()
        assert int(host(ref_err)[0]) == 0 and int(host(got_err)[0]) == 0
        assert np.array_equal(host(got_pair), host(ref_pair)), f"{sh.name}: routed outputs differ"
        assert np.array_equal(host(got_sh), host(ref_sh)), f"{sh.name}: shared outputs differ"


def _zero_layer(m, E, d, f, T, k):
    qb, sc = m.expert_q_bytes(d, f), m.expert_s_count(d, f)
    q = torch.zeros(E * qb, dtype=torch.uint8, device="cuda")
    s = torch.zeros(E * sc, dtype=torch.float32, device="cuda")
    lw = m.LayerWeights(q, s, q[:qb], s[:sc], E=E, d=d, f=f)
    idx = (torch.arange(T * k, dtype=torch.int32, device="cuda") % E).view(T, k)   # distinct per token
    un = m.moe_union(idx, E)
    return lw, un


def test_noalloc_scratch_boundary_at_the_layer_shape(m):
    """At d = 6144, f = 2048, k = 8 the automatic mode's scratch fits the reserved array up to
    T = 73 and not at T = 74: the library's own limit, checked through the entry point."""
    d, f, E, k = 6144, 2048, 8, 8
    for T, fits in ((73, True), (74, False)):
        assert (m.ffn_workspace_bytes(T, k, d, f) <= m._binding.NOALLOC_SCRATCH_BYTES) == fits
        lw, un = _zero_layer(m, E, d, f, T, k)
        x = torch.zeros((T, d), dtype=torch.float32, device="cuda")
        if fits:
            y_pair, y_sh, err = m.moe_expert_ffn_int4_noalloc(x, lw, un, k)
            torch.cuda.synchronize()
            assert int(host(err)[0]) == 0
            assert not host(y_pair).any() and not host(y_sh).any()   # zero weights give zero outputs
        else:
            with pytest.raises(m.MoeError) as ei:
                m.moe_expert_ffn_int4_noalloc(x, lw, un, k)
            assert ei.value.status == m.MOE_ERR_WORKSPACE
        del lw, un
    torch.cuda.empty_cache()


def test_noalloc_rejects_batches_beyond_the_reserved_scratch(m):
    d, f, E, T, k = 6144, 2048, 8, 512, 8
    assert m.ffn_workspace_bytes(T, k, d, f) > m._binding.NOALLOC_SCRATCH_BYTES
    x = torch.zeros((T, d), dtype=torch.float32, device="cuda")
    lw, un = _zero_layer(m, E, d, f, T, k)
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_ffn_int4_noalloc(x, lw, un, k)
    assert ei.value.status == m.MOE_ERR_WORKSPACE
