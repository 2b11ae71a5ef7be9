"""The bounds-checked build (MOE_DEBUG_BOUNDS) on valid inputs: no index is
flagged and every output is bit-identical to the normal build's, on every FFN path
and through the host-buffer entry.  Each library runs in its own child process
(tests/debug_bounds_child.py)."""
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


def _run(lib, path):
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_child.py"), lib, path],
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
