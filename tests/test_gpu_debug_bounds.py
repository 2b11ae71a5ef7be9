"""The bounds-checked build (MOE_DEBUG_BOUNDS).  On valid inputs no index is
flagged and every output is bit-identical to the normal build's, on every FFN path
and through the host-buffer entry; given a union list with an expert id outside
the layer, it flags and skips that entry and leaves the other experts' rows as
they were.  Each library runs in its own child process (tests/debug_bounds_child.py)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_sigmoid_gb300 import build
    return build.build(), build.build(debug_bounds=True)


def _run(lib, path, *extra):
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_child.py"), lib, path, *extra],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return np.load(path)


def test_debug_bounds_build_matches_and_flags_nothing(libs, tmp_path):
    normal = _run(libs[0], str(tmp_path / "normal.npz"))
    checked = _run(libs[1], str(tmp_path / "checked.npz"))
    assert sorted(normal.files) == sorted(checked.files) and len(normal.files) == 4 * (3 * 3 + 2)
    for key in normal.files:
        if key.endswith("_err"):
            assert int(checked[key][0]) == 0 and int(normal[key][0]) == 0, key
        else:
            assert np.array_equal(normal[key], checked[key]), key


def test_debug_bounds_build_skips_a_bad_expert_in_the_union(libs, tmp_path):
    """The bounds-checked build given union arrays that name an expert outside the layer (the FFN call on
    every path): the entry is flagged (MOE_DEVERR_BOUNDS, or MOE_DEVERR_BAD_EXPERT from the hybrid's split)
    and skipped, the other experts' rows and the shared expert's come out as with the intact list.  Run
    with the checked library only: the normal build trusts the union arrays."""
    import int4_routed_expert_sigmoid_gb300 as m
    r = _run(libs[1], str(tmp_path / "bad.npz"), "bad")
    for T in (4, 130):
        name = f"dbg_bad_t{T}"
        n = int(r[f"{name}_n_uniq"][0])
        uniq, off = r[f"{name}_uniq"][:n], r[f"{name}_offsets"]
        for mode_name in ("MOE_MODE_DECODE", "MOE_MODE_PREFILL", "MOE_MODE_HYBRID"):
            key = f"{name}_{mode_name}"
            assert int(r[f"{key}_ok_err"][0]) == 0, key
            assert int(r[f"{key}_bad_err"][0]) & (m.MOE_DEVERR_BOUNDS | m.MOE_DEVERR_BAD_EXPERT), key
            yo, yb = r[f"{key}_ok_y"], r[f"{key}_bad_y"]
            for e in uniq[1:]:
                assert np.array_equal(yb[off[e]:off[e + 1]], yo[off[e]:off[e + 1]]), (key, e)
            assert np.array_equal(r[f"{key}_bad_ys"], r[f"{key}_ok_ys"]), key
