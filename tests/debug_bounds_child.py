"""Child process of tests/test_gpu_debug_bounds.py: runs the layer through one
libmoe build (argv[1]) on the small parity shapes and saves the outputs and
error words to argv[2] (npz).  A separate process, so that the normal and the
bounds-checked library are never loaded together."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from int4_routed_expert_sigmoid_gb300 import _binding  # noqa: E402

_binding.LIB_PATH = os.path.abspath(sys.argv[1])
import torch  # noqa: E402

import int4_routed_expert_sigmoid_gb300 as moe  # noqa: E402
import workloads  # noqa: E402
from moe_testlib import device_layer  # noqa: E402

Shape = workloads.Shape
SHAPES = [Shape("dbg_t1", E=16, k=4, d=1024, f=256, T=1, bias="normal"),
          Shape("dbg_t5", E=64, k=8, d=512, f=512, T=5, bias="zipf"),
          Shape("dbg_t37", E=16, k=4, d=1024, f=384, T=37, bias="normal"),
          Shape("dbg_t130", E=32, k=4, d=512, f=256, T=130, bias="zipf")]
out = {}
if len(sys.argv) > 3 and sys.argv[3] == "bad":
    # union arrays naming an expert outside the layer, handed to the FFN call: only ever run with the
    # bounds-checked library, whose checks turn the bad entry into an error bit and skip it
    for T in (4, 130):
        sh = Shape(f"dbg_bad_t{T}", E=8, k=2, d=256, f=128, T=T, bias="normal")
        L = workloads.layer_inputs(sh, seed=4, threads=2)
        dev = device_layer(L)
        idx, _, _ = moe.moe_route(dev["x"], dev["wg"], dev["bias"], sh.k)
        un = moe.moe_union(idx, sh.E)
        bad = dict(un)
        bad["uniq"] = un["uniq"].clone()
        bad["uniq"][0] = sh.E + 3
        torch.cuda.synchronize()
        out[f"{sh.name}_n_uniq"] = un["n_uniq"].cpu().numpy()
        out[f"{sh.name}_uniq"] = un["uniq"].cpu().numpy()
        out[f"{sh.name}_offsets"] = un["offsets"].cpu().numpy()
        for mode_name in ("MOE_MODE_DECODE", "MOE_MODE_PREFILL", "MOE_MODE_HYBRID"):
            for tag, u in (("ok", un), ("bad", bad)):
                y, ys, err = moe.moe_expert_ffn_int4(dev["x"], dev["layer"], u, sh.k, getattr(moe, mode_name))
                torch.cuda.synchronize()
                out[f"{sh.name}_{mode_name}_{tag}_y"] = y.cpu().numpy()
                out[f"{sh.name}_{mode_name}_{tag}_ys"] = ys.cpu().numpy()
                out[f"{sh.name}_{mode_name}_{tag}_err"] = err.cpu().numpy()
    np.savez(sys.argv[2], **out)
    sys.exit(0)
for sh in SHAPES:
    L = workloads.layer_inputs(sh, seed=5, threads=4)
    dev = device_layer(L)
    x = torch.from_numpy(workloads.activations(sh.T, sh.d, seed=6)).cuda()
    res = torch.from_numpy(workloads.activations(sh.T, sh.d, seed=7)).cuda()
    for mode_name in ("MOE_MODE_DECODE", "MOE_MODE_PREFILL", "MOE_MODE_HYBRID"):
        hits = torch.zeros(sh.E, dtype=torch.int64, device="cuda")
        y, err = moe.moe_layer_forward(x, dev["wg"], dev["bias"], dev["layer"], sh.k, mode=getattr(moe, mode_name),
                                       residual=res, hits=hits)
        torch.cuda.synchronize()
        out[f"{sh.name}_{mode_name}_y"] = y.cpu().numpy()
        out[f"{sh.name}_{mode_name}_err"] = err.cpu().numpy()
        out[f"{sh.name}_{mode_name}_hits"] = hits.cpu().numpy()
    # the host-buffer entry on page-locked rows (the copy kernel, the combine writing into host memory)
    y_h, err_h = moe.moe_layer_forward_host(x.cpu().pin_memory(), dev["wg"], dev["bias"], dev["layer"], sh.k,
                                            residual=res)
    torch.cuda.synchronize()
    out[f"{sh.name}_host_y"] = y_h.numpy()
    out[f"{sh.name}_host_err"] = err_h.cpu().numpy()
np.savez(sys.argv[2], **out)
