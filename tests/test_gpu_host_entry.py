"""moe_layer_forward_host: the layer with its token rows and result in
page-locked host memory gives the bits of moe_layer_forward on the same rows
(both FFN paths, with a residual and the hit counters), and refuses a
workspace without room for the row copies."""
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
@pytest.mark.parametrize("T", [1, 9])
def test_host_entry_matches_device_entry(mode_name, T):
    m = moe()
    mode = getattr(m, mode_name)
    sh = Shape("host_entry", E=16, k=4, d=1024, f=256, T=T, bias="normal")
    L = workloads.layer_inputs(sh, seed=T, threads=4)
    dev = device_layer(L)
    res = torch.from_numpy(workloads.activations(T, sh.d, seed=3)).cuda()
    hits_h = torch.zeros(sh.E, dtype=torch.int64, device="cuda")
    hits_d = torch.zeros(sh.E, dtype=torch.int64, device="cuda")
    for call in range(2):   # the second call reuses the workspace and the host buffers
        x_host = torch.from_numpy(workloads.activations(T, sh.d, seed=40 + call)).pin_memory()
        out_h, err_h = m.moe_layer_forward_host(x_host, dev["wg"], dev["bias"], dev["layer"], sh.k, mode=mode,
                                                residual=res, hits=hits_h)
        out_d, err_d = m.moe_layer_forward(x_host.cuda(), dev["wg"], dev["bias"], dev["layer"], sh.k, mode=mode,
                                           residual=res, hits=hits_d)
        torch.cuda.synchronize()
        assert int(host(err_h)[0]) == 0 and int(host(err_d)[0]) == 0
        assert np.array_equal(out_h.numpy(), host(out_d)), f"call {call}"
    assert np.array_equal(host(hits_h), host(hits_d))


@pytest.mark.parametrize("pinned", [True, False])
def test_host_entry_pageable_and_pinned_buffers(pinned):
    """Page-locked buffers take the direct route (a kernel reads the rows, the combine writes the
    result into host memory), pageable ones the copy route; both give the device entry's bits, and
    a direct-route call that follows another in the stream sees its own rows."""
    m = moe()
    sh = Shape("host_entry_route", E=16, k=4, d=512, f=256, T=5, bias="normal")
    L = workloads.layer_inputs(sh, seed=8, threads=4)
    dev = device_layer(L)
    ws = m.workspace(m.layer_host_workspace_bytes(sh.T, sh.k, sh.E, sh.d, sh.f), "cuda")
    outs, refs = [], []
    for call in range(3):   # back to back on one stream, one synchronisation at the end
        x = torch.from_numpy(workloads.activations(sh.T, sh.d, seed=60 + call))
        out_host = torch.empty((sh.T, sh.d), dtype=torch.float32)
        if pinned:
            x, out_host = x.pin_memory(), out_host.pin_memory()
        m.moe_layer_forward_host(x, dev["wg"], dev["bias"], dev["layer"], sh.k, out_host=out_host, ws=ws)
        outs.append(out_host)
        refs.append(m.moe_layer_forward(x.cuda(), dev["wg"], dev["bias"], dev["layer"], sh.k)[0])
    torch.cuda.synchronize()
    for call in range(3):
        assert np.array_equal(outs[call].numpy(), host(refs[call])), f"call {call}"


def test_host_entry_workspace_and_pointers():
    m = moe()
    sh = Shape("host_entry_ws", E=8, k=2, d=256, f=128, T=3, bias="normal")
    L = workloads.layer_inputs(sh, seed=1, threads=2)
    dev = device_layer(L)
    need = m.layer_host_workspace_bytes(sh.T, sh.k, sh.E, sh.d, sh.f)
    assert need >= m.layer_workspace_bytes(sh.T, sh.k, sh.E, sh.d, sh.f) + 2 * sh.T * sh.d * 4
    x_host = torch.from_numpy(workloads.activations(sh.T, sh.d, seed=2)).pin_memory()
    small = torch.empty(need - 1024, dtype=torch.uint8, device="cuda")   # short even after the 256-byte alignment
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer_forward_host(x_host, dev["wg"], dev["bias"], dev["layer"], sh.k, ws=small)
    assert ei.value.status == m.MOE_ERR_WORKSPACE
