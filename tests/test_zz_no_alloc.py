"""moe_expert_ffn_int4_noalloc: the expert FFN for callers that cannot allocate
device memory (a host framework that owns all device memory, or a
latency-critical caller that cannot afford cudaMalloc/cudaFree).  Its scratch
is the library's static 8 MiB device array instead of a caller workspace.

Checked through the C ABI against the existing workspace entry point, on two
calls in a row (the second call finds the first call's leftovers in the shared
array), within the decode-path tolerance the parity tests use.  This file is
collected last so that a failure here stops a -x run only after every other
test has run.
"""
import numpy as np
import pytest
import torch

import workloads
from moe_testlib import TOL_DECODE, device_layer, host, moe, rel_max_err

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


def test_noalloc_ffn_matches_workspace_ffn_on_two_calls(m):
    shapes = [workloads.Shape("na_a", E=16, k=4, d=1024, f=384, T=37, bias="normal"),
              workloads.Shape("na_b", E=8, k=2, d=256, f=128, T=5)]
    for i, sh in enumerate(shapes):            # two different calls in a row
        dev, un = _routed(m, sh, seed=10 + i)
        ref_pair, ref_sh, ref_err = m.moe_expert_ffn_int4(dev["x"], dev["layer"], un, sh.k)
        got_pair, got_sh, got_err = m.moe_expert_ffn_int4_noalloc(dev["x"], dev["layer"], un, sh.k)
        torch.cuda.synchronize()
        assert int(host(ref_err)[0]) == 0 and int(host(got_err)[0]) == 0
        assert rel_max_err(host(got_pair), host(ref_pair).astype(np.float64)) <= TOL_DECODE
        assert rel_max_err(host(got_sh), host(ref_sh).astype(np.float64)) <= TOL_DECODE


def test_noalloc_rejects_batches_beyond_the_reserved_scratch(m):
    d, f, E, T, k = 6144, 2048, 8, 512, 8
    assert m.ffn_workspace_bytes(T, k, d, f) > m._binding.NOALLOC_SCRATCH_BYTES
    x = torch.zeros((T, d), dtype=torch.float32, device="cuda")
    qb, sc = m.expert_q_bytes(d, f), m.expert_s_count(d, f)
    q = torch.zeros(E * qb, dtype=torch.uint8, device="cuda")
    s = torch.zeros(E * sc, dtype=torch.float32, device="cuda")
    lw = m.LayerWeights(q, s, q[:qb], s[:sc], E=E, d=d, f=f)
    un = {key: torch.zeros(n, dtype=torch.int32, device="cuda")
          for key, n in (("offsets", E + 1), ("sorted_pair", T * k), ("uniq", E), ("n_uniq", 1))}
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_ffn_int4_noalloc(x, lw, un, k)
    assert ei.value.status == m.MOE_ERR_WORKSPACE
