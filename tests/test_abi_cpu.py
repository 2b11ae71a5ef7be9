"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/moe.h declares, and rejects bad arguments on the host before any CUDA
call.  No compute call is made here."""
import ctypes

import pytest

import oracle
import workloads


@pytest.fixture(scope="module")
def m():
    from int4_routed_expert_sigmoid_gb300 import build
    build.build()
    import int4_routed_expert_sigmoid_gb300 as pkg
    return pkg


def test_exports_every_header_symbol(m):
    names = m.header_functions()
    assert len(names) >= 12
    L = m.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings_and_device_error_decoding(m):
    assert m.status_str(m.MOE_OK) == "ok"
    assert "workspace" in m.status_str(m.MOE_ERR_WORKSPACE)
    assert m.device_error(0) == m.MOE_OK
    assert m.device_error(m.MOE_DEVERR_BAD_EXPERT) == m.MOE_ERR_INVALID_ARG
    assert m.device_error(m.MOE_DEVERR_TIMEOUT) == m.MOE_ERR_CUDA
    assert m.device_error(m.MOE_DEVERR_BOUNDS) == m.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("d,f", [(256, 128), (6144, 2048), (1024, 384)])
def test_expert_sizes_agree_with_oracle_layout(m, d, f):
    assert m.expert_q_bytes(d, f) == oracle.expert_q_bytes(d, f) == workloads.expert_q_bytes(d, f)
    assert m.expert_s_count(d, f, 32) == oracle.expert_s_count(d, f, 32) == workloads.expert_s_count(d, f, 32)


def test_workspace_queries(m):
    assert m.ffn_workspace_bytes(0, 8, 6144, 2048) == 0
    a = m.layer_workspace_bytes(1, 8, 256, 6144, 2048)
    b = m.layer_workspace_bytes(64, 8, 256, 6144, 2048)
    assert 0 < a < b and a % 256 == 0
    # y_pair alone is T*k*d floats
    assert b >= 64 * 8 * 6144 * 4


def test_mode_constants_and_workspace_by_path(m):
    """The binding's FFN modes are the header's enum; the workspace follows the path a mode resolves to:
    AUTO is the decode path below 128 tokens and the hybrid from 128 (decode + prefill scratch + lists)."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")).read()
    modes = dict(re.findall(r"(MOE_MODE_\w+) = (\d+)", hdr))
    assert set(modes) == {"MOE_MODE_AUTO", "MOE_MODE_DECODE", "MOE_MODE_PREFILL", "MOE_MODE_HYBRID"}
    for name, val in modes.items():
        assert getattr(m, name) == int(val), name
    d, f, k = 6144, 2048, 8
    for T in (1, 127, 128, 256):
        dec = m.ffn_workspace_bytes(T, k, d, f, m.MOE_MODE_DECODE)
        pre = m.ffn_workspace_bytes(T, k, d, f, m.MOE_MODE_PREFILL)
        hyb = m.ffn_workspace_bytes(T, k, d, f, m.MOE_MODE_HYBRID)
        assert hyb >= dec + pre and hyb % 256 == 0
        assert m.ffn_workspace_bytes(T, k, d, f, m.MOE_MODE_AUTO) == (dec if T < 128 else hyb)
    assert m.ffn_workspace_bytes(4, k, d, f, 4) == 0   # not a mode


def test_host_validation_rejects_without_launching(m):
    L = m.lib()
    P = None
    assert L.moe_route(P, P, P, 1, 256, 8, 2, 1, 1.0, P, P, P, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_union(P, 1, 2, 8, P, P, P, P, P, P, P, P, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_hits(P, 8, P, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_combine(P, P, P, P, P, 1, 2, 256, P, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_rms_norm(P, 1, 256, 1e-5, P, P) == m.MOE_ERR_INVALID_ARG
    ok = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: the sizes are refused first
    assert L.moe_rms_norm(ok, 1, 6, 1e-5, ok, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_rms_norm(ok, 0, 256, 1e-5, ok, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_rms_norm(ok, 1, 256, -1.0, ok, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_rms_norm(ok, 1, 256, float("nan"), ok, P) == m.MOE_ERR_INVALID_ARG
    assert L.moe_layer_forward(P, P, P, None, P, 1, 2, 1, 1.0, 0, P, P, P, P, P, 0, P, P) == m.MOE_ERR_INVALID_ARG
    # a layer with an unsupported group size is refused before its pointers are used: G = 48, and
    # G = 64 with f not a multiple of 256
    for G, f in ((48, 256), (64, 128)):
        fake = m._binding.moe_layer_int4(16, 16, 16, 16, 8, 256, f, G)
        assert L.moe_expert_ffn_int4(P, ctypes.byref(fake), P, P, P, P, 1, 2, 0, P, P, P, 0, P, P) == \
            m.MOE_ERR_UNSUPPORTED
    # misaligned pointers are refused
    bad = ctypes.c_void_p(0x1004)
    assert L.moe_hits(bad, 8, bad, P) == m.MOE_ERR_INVALID_ARG


def test_binding_error_bits_match_the_header(m):
    """The binding's device error bits are the header's values."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")).read()
    bits = dict(re.findall(r"#define (MOE_DEVERR_\w+) (0x[0-9a-fA-F]+)", hdr))
    assert len(bits) == 4
    for name, val in bits.items():
        assert getattr(m, name) == int(val, 16), name


def test_debug_bounds_build_exports_every_header_symbol(m):
    """The bounds-checked build (MOE_DEBUG_BOUNDS) compiles and exports the same symbols."""
    from int4_routed_expert_sigmoid_gb300 import build
    path = build.build(debug_bounds=True)
    assert path != build.LIB
    L = ctypes.CDLL(path)
    missing = [n for n in m.header_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_empty_batch_is_refused_before_launching(m):
    """T = 0 (an empty batch) is an argument error on every entry point, found before anything is
    launched (there is no GPU here: a launch would come back as MOE_ERR_CUDA), and the workspace size
    queries give 0 for it."""
    L = m.lib()
    ok = ctypes.c_void_p(0x10000)   # aligned and never dereferenced: the batch size is refused first
    lay = ctypes.byref(m._binding.moe_layer_int4(0x10000, 0x10000, 0x10000, 0x10000, 16, 256, 128, 32))
    big = 1 << 40
    inv = m.MOE_ERR_INVALID_ARG
    assert L.moe_route(ok, ok, None, 0, 256, 16, 2, 1, 1.0, ok, ok, ok, None) == inv
    assert L.moe_route_topp(ok, ok, None, 0, 256, 16, 2, 1, 1.0, 0.7, ok, ok, ok, None) == inv
    assert L.moe_union(ok, 0, 2, 16, ok, ok, ok, ok, ok, ok, None, ok, None) == inv
    for mode in (0, 1, 2, 3):
        assert L.moe_expert_ffn_int4(ok, lay, ok, ok, ok, ok, 0, 2, mode, ok, ok, ok, big, ok, None) == inv
        assert L.moe_layer_forward(ok, ok, None, lay, None, 0, 2, 1, 1.0, mode, ok, None, None, None, ok, big, ok,
                                   None) == inv
        assert L.moe_layer_forward_topp(ok, ok, None, lay, None, 0, 2, 1, 1.0, 0.7, mode, ok, None, None, None, ok,
                                        big, ok, None) == inv
        assert L.moe_layer_forward_norm(ok, ok, None, lay, None, 0, 2, 1, 1.0, 1.0, mode, ok, ok, 1e-5, None, None,
                                        None, ok, big, ok, None) == inv
        assert m.layer_workspace_bytes(0, 2, 16, 256, 128, mode) == 0
        assert m.ffn_workspace_bytes(0, 2, 256, 128, mode) == 0
    assert L.moe_combine(ok, ok, ok, ok, None, 0, 2, 256, ok, None) == inv
