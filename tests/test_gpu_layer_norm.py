"""moe_layer_forward_norm (the layer plus RMSNorm of its output, for a pre-norm
stack) gives bitwise the outputs of moe_layer_forward followed by moe_rms_norm,
on both FFN paths, for rows the fused combine takes and for a wider row (the
two kernels one after the other)."""
import numpy as np
import pytest
import torch

import workloads
from moe_testlib import device_layer, host, moe

pytestmark = pytest.mark.gpu

Shape = workloads.Shape


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_sigmoid_gb300 import build
    build.build()


@pytest.mark.parametrize("mode_name", ["MOE_MODE_DECODE", "MOE_MODE_PREFILL", "MOE_MODE_HYBRID"])
@pytest.mark.parametrize("T,d", [(1, 1024), (5, 512), (37, 1024), (64, 768), (65, 768), (3, 8448)])
def test_layer_norm_matches_layer_then_rms_norm(mode_name, T, d):
    m = moe()
    mode = getattr(m, mode_name)
    sh = Shape("layer_norm", E=16, k=4, d=d, f=256, T=T, bias="normal")
    L = workloads.layer_inputs(sh, seed=T + d, threads=4)
    dev = device_layer(L)
    x = torch.from_numpy(workloads.activations(T, d, seed=11)).cuda()
    res = torch.from_numpy(workloads.activations(T, d, seed=12)).cuda()
    eps = 1e-5
    out_f, xn_f, err_f = m.moe_layer_forward_norm(x, dev["wg"], dev["bias"], dev["layer"], sh.k, eps=eps, mode=mode,
                                                  residual=res)
    out_s, err_s = m.moe_layer_forward(x, dev["wg"], dev["bias"], dev["layer"], sh.k, mode=mode, residual=res)
    xn_s = m.moe_rms_norm(out_s, eps)
    torch.cuda.synchronize()
    assert int(host(err_f)[0]) == 0 and int(host(err_s)[0]) == 0
    assert np.array_equal(host(out_f), host(out_s))
    assert np.array_equal(host(xn_f), host(xn_s))


def test_layer_norm_rejects_aliasing_and_bad_eps():
    m = moe()
    sh = Shape("layer_norm_args", E=8, k=2, d=256, f=128, T=2, bias="normal")
    L = workloads.layer_inputs(sh, seed=1, threads=2)
    dev = device_layer(L)
    x = torch.from_numpy(workloads.activations(sh.T, sh.d, seed=2)).cuda()
    out = torch.empty_like(x)
    for kw in (dict(out=out, out_normed=out), dict(out_normed=x), dict(eps=-1.0), dict(eps=float("nan"))):
        with pytest.raises(m.MoeError) as ei:
            m.moe_layer_forward_norm(x, dev["wg"], dev["bias"], dev["layer"], sh.k, **kw)
        assert ei.value.status == m.MOE_ERR_INVALID_ARG
