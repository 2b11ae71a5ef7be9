"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here takes torch CUDA tensors, checks dtypes/shapes enough to
build the C call, and calls the entry point of the same name.  All arithmetic
runs in the CUDA kernels behind the C ABI.  There is no CPU fallback: if the
library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmoe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_STALE = 0, -1, -2, -3, -4, -5
MOE_DEVERR_BAD_EXPERT, MOE_DEVERR_TIMEOUT, MOE_DEVERR_SCALE_RANGE, MOE_DEVERR_BOUNDS = 0x1, 0x2, 0x4, 0x8
MOE_MODE_AUTO, MOE_MODE_DECODE, MOE_MODE_PREFILL, MOE_MODE_HYBRID = 0, 1, 2, 3

_HITS_DTYPES = tuple(getattr(torch, n) for n in ("int64", "uint64") if hasattr(torch, n))
_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


class moe_layer_int4(ctypes.Structure):
    _fields_ = [("q_base", ctypes.c_void_p), ("s_base", ctypes.c_void_p),
                ("shared_q", ctypes.c_void_p), ("shared_s", ctypes.c_void_p),
                ("E", ctypes.c_int), ("d", ctypes.c_int), ("f", ctypes.c_int), ("G", ctypes.c_int)]


_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "moe_status_str": ([_I], ctypes.c_char_p),
    "moe_device_error": ([ctypes.c_int32], _I),
    "moe_expert_q_bytes": ([_I, _I], _SZ),
    "moe_expert_s_count": ([_I, _I, _I], _SZ),
    "moe_route": ([_P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P], _I),
    "moe_route_topp": ([_P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _P, _P, _P, _P], _I),
    "moe_union": ([_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_hits": ([_P, _I, _P, _P], _I),
    "moe_expert_ffn_int4": ([_P, ctypes.POINTER(moe_layer_int4), _P, _P, _P, _P, _I, _I, _I, _P, _P,
                             _P, _SZ, _P, _P], _I),
    "moe_ffn_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "moe_expert_ffn_int4_noalloc": ([_P, ctypes.POINTER(moe_layer_int4), _P, _P, _P, _P, _I, _I, _I, _P, _P,
                                     _P, _P], _I),
    "moe_combine": ([_P, _P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_rms_norm": ([_P, _I, _I, _F, _P, _P], _I),
    "moe_layer_forward": ([_P, _P, _P, ctypes.POINTER(moe_layer_int4), _P, _I, _I, _I, _F, _I, _P, _P,
                           _P, _P, _P, _SZ, _P, _P], _I),
    "moe_layer_forward_topp": ([_P, _P, _P, ctypes.POINTER(moe_layer_int4), _P, _I, _I, _I, _F, _F, _I, _P,
                                _P, _P, _P, _P, _SZ, _P, _P], _I),
    "moe_layer_workspace_bytes": ([_I, _I, _I, _I, _I, _I], _SZ),
    "moe_layer_forward_norm": ([_P, _P, _P, ctypes.POINTER(moe_layer_int4), _P, _I, _I, _I, _F, _F, _I, _P, _P, _F,
                                _P, _P, _P, _P, _SZ, _P, _P], _I),
    "moe_layer_forward_host": ([_P, _P, _P, ctypes.POINTER(moe_layer_int4), _P, _I, _I, _I, _F, _F, _I, _P,
                                _P, _P, _P, _P, _SZ, _P, _P], _I),
    "moe_layer_host_workspace_bytes": ([_I, _I, _I, _I, _I, _I], _SZ),
    "moe_usage_save": ([ctypes.c_char_p, _P, _I, _I, ctypes.c_uint64], _I),
    "moe_usage_load": ([ctypes.c_char_p, _P, _I, _I, ctypes.c_uint64], _I),
    "moe_usage_top": ([_P, _I, _I, _P], _I),
    "moe_tier_create": ([_I, _I, _I, _I, _P, _P, _P, _P, _I, ctypes.POINTER(ctypes.c_void_p)], _I),
    "moe_tier_destroy": ([_P], None),
    "moe_tier_pin": ([_P, _P, _I, _P], _I),
    "moe_tier_prefetch": ([_P, _P, _I, _P], _I),
    "moe_tier_unpin_all": ([_P], _I),
    "moe_tier_stats": ([_P, _P], _I),
    "moe_tier_slots": ([_P, _P, _P], _I),
    "moe_tier_workspace_bytes": ([_I, _I, _I, _I, _I, _I], _SZ),
    "moe_layer_forward_tier": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _F, _F, _I, _P, _P, _P, _P, _P, _SZ, _P,
                                _P, _P], _I),
}


def lib() -> ctypes.CDLL:
    """Load libmoe.so (built by ``int4_routed_expert_sigmoid_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libmoe.so is not built ({LIB_PATH}); run "
                    "`python -m int4_routed_expert_sigmoid_gb300.build` -- there is no fallback path")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
        return _lib


def status_str(status: int) -> str:
    return lib().moe_status_str(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, dtype, what: str) -> torch.Tensor:
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{what} must be a contiguous CUDA tensor of {dtype}")
    return t


def expert_q_bytes(d: int, f: int) -> int:
    return int(lib().moe_expert_q_bytes(d, f))


def expert_s_count(d: int, f: int, G: int = 32) -> int:
    return int(lib().moe_expert_s_count(d, f, G))


def device_error(err_word: int) -> int:
    return int(lib().moe_device_error(int(err_word)))


class LayerWeights:
    """Device-resident int4 experts of one layer plus the moe_layer_int4 view."""

    def __init__(self, q_base: torch.Tensor, s_base: torch.Tensor, shared_q: torch.Tensor,
                 shared_s: torch.Tensor, E: int, d: int, f: int, G: int = 32):
        self.q_base = _need(q_base, torch.uint8, "q_base")
        self.s_base = _need(s_base, torch.float32, "s_base")
        self.shared_q = _need(shared_q, torch.uint8, "shared_q")
        self.shared_s = _need(shared_s, torch.float32, "shared_s")
        if self.q_base.numel() < E * expert_q_bytes(d, f) or self.s_base.numel() < E * expert_s_count(d, f, G):
            raise ValueError("expert arrays smaller than E expert blocks")
        self.E, self.d, self.f, self.G = E, d, f, G
        self.c = moe_layer_int4(q_base.data_ptr(), s_base.data_ptr(), shared_q.data_ptr(),
                                shared_s.data_ptr(), E, d, f, G)


def moe_route(x, w_gate, bias, k: int, normalize: int = 1, route_scale: float = 1.0,
              topk_idx=None, topk_w=None, logits=None, stream=None, top_p: float | None = None):
    """moe_route, or moe_route_topp when top_p is given."""
    _need(x, torch.float32, "x")
    _need(w_gate, torch.float32, "w_gate")
    T, d = x.shape
    E = w_gate.shape[0]
    if bias is not None:
        _need(bias, torch.float32, "bias")
    dev = x.device
    topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_w = torch.empty((T, k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if logits is None else logits
    if top_p is None:
        _check(lib().moe_route(_p(x), _p(w_gate), _p(bias), T, d, E, k, int(normalize), float(route_scale),
                               _p(topk_idx), _p(topk_w), _p(logits), _stream(stream)), "moe_route")
    else:
        _check(lib().moe_route_topp(_p(x), _p(w_gate), _p(bias), T, d, E, k, int(normalize), float(route_scale),
                                    float(top_p), _p(topk_idx), _p(topk_w), _p(logits), _stream(stream)),
               "moe_route_topp")
    return topk_idx, topk_w, logits


def moe_union(topk_idx, E: int, hits=None, err=None, out=None, stream=None):
    """Returns dict(counts, offsets, perm, sorted_pair, uniq, n_uniq, err) of device tensors."""
    _need(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    dev = topk_idx.device
    if out is None:
        out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   perm=torch.empty(T * k, dtype=torch.int32, device=dev),
                   sorted_pair=torch.empty(T * k, dtype=torch.int32, device=dev),
                   uniq=torch.empty(E, dtype=torch.int32, device=dev),
                   n_uniq=torch.empty(1, dtype=torch.int32, device=dev))
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    out["err"] = err
    if hits is not None and not (hits.is_cuda and hits.dtype in _HITS_DTYPES and hits.numel() >= E):
        raise ValueError("hits must be a CUDA int64/uint64 tensor of E counters")
    _check(lib().moe_union(_p(topk_idx), T, k, E, _p(out["counts"]), _p(out["offsets"]), _p(out["perm"]),
                           _p(out["sorted_pair"]), _p(out["uniq"]), _p(out["n_uniq"]), _p(hits), _p(err),
                           _stream(stream)), "moe_union")
    return out


def moe_hits(counts, hits, stream=None):
    _need(counts, torch.int32, "counts")
    if not (hits.is_cuda and hits.dtype in _HITS_DTYPES and hits.numel() >= counts.numel()):
        raise ValueError("hits must be a CUDA int64/uint64 tensor of E counters")
    _check(lib().moe_hits(_p(counts), counts.numel(), _p(hits), _stream(stream)), "moe_hits")


def ffn_workspace_bytes(T: int, k: int, d: int, f: int, mode: int = MOE_MODE_AUTO) -> int:
    return int(lib().moe_ffn_workspace_bytes(T, k, d, f, mode))


def layer_workspace_bytes(T: int, k: int, E: int, d: int, f: int, mode: int = MOE_MODE_AUTO) -> int:
    return int(lib().moe_layer_workspace_bytes(T, k, E, d, f, mode))


def workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned device scratch buffer of at least nbytes."""
    return torch.empty(max(int(nbytes), 1) + 256, dtype=torch.uint8, device=device)


def _ws_ptr(ws: torch.Tensor) -> tuple[ctypes.c_void_p, int]:
    base = ws.data_ptr()
    aligned = (base + 255) & ~255
    return ctypes.c_void_p(aligned), ws.numel() - (aligned - base)


def moe_expert_ffn_int4(x, layer: LayerWeights, un: dict, k: int, mode: int = MOE_MODE_AUTO,
                        y_pair=None, y_shared=None, ws=None, err=None, stream=None):
    _need(x, torch.float32, "x")
    T, d = x.shape
    dev = x.device
    y_pair = torch.empty((T * k, d), dtype=torch.float32, device=dev) if y_pair is None else y_pair
    y_shared = torch.empty((T, d), dtype=torch.float32, device=dev) if y_shared is None else y_shared
    if ws is None:
        ws = workspace(ffn_workspace_bytes(T, k, d, layer.f, mode), dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    wp, wn = _ws_ptr(ws)
    _check(lib().moe_expert_ffn_int4(_p(x), ctypes.byref(layer.c), _p(un["offsets"]), _p(un["sorted_pair"]),
                                     _p(un["uniq"]), _p(un["n_uniq"]), T, k, mode, _p(y_pair), _p(y_shared),
                                     wp, wn, _p(err), _stream(stream)), "moe_expert_ffn_int4")
    return y_pair, y_shared, err


def _header_scratch_bytes() -> int:
    """MOE_NOALLOC_SCRATCH_BYTES as include/moe.h defines it (one source for the limit)."""
    import re
    m = re.search(r"#define\s+MOE_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", open(HEADER).read())
    if not m:
        raise RuntimeError("MOE_NOALLOC_SCRATCH_BYTES not found in include/moe.h")
    return int(m.group(1)) << int(m.group(2))


NOALLOC_SCRATCH_BYTES = _header_scratch_bytes()


def moe_expert_ffn_int4_noalloc(x, layer: LayerWeights, un: dict, k: int, mode: int = MOE_MODE_AUTO,
                                y_pair=None, y_shared=None, err=None, stream=None):
    """moe_expert_ffn_int4 with its scratch in the library's static device array
    (for callers that cannot allocate device memory); outputs as for
    moe_expert_ffn_int4.  Calls on one device share that array: keep them on one
    stream."""
    _need(x, torch.float32, "x")
    T, d = x.shape
    dev = x.device
    y_pair = torch.empty((T * k, d), dtype=torch.float32, device=dev) if y_pair is None else y_pair
    y_shared = torch.empty((T, d), dtype=torch.float32, device=dev) if y_shared is None else y_shared
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().moe_expert_ffn_int4_noalloc(_p(x), ctypes.byref(layer.c), _p(un["offsets"]),
                                             _p(un["sorted_pair"]), _p(un["uniq"]), _p(un["n_uniq"]), T, k,
                                             mode, _p(y_pair), _p(y_shared), _p(err), _stream(stream)),
           "moe_expert_ffn_int4_noalloc")
    return y_pair, y_shared, err


def moe_combine(y_pair, y_shared, topk_w, perm, residual=None, out=None, stream=None):
    T, k = topk_w.shape
    d = y_shared.shape[1]
    out = torch.empty((T, d), dtype=torch.float32, device=y_shared.device) if out is None else out
    _check(lib().moe_combine(_p(y_pair), _p(y_shared), _p(topk_w), _p(perm), _p(residual), T, k, d, _p(out),
                             _stream(stream)), "moe_combine")
    return out


def moe_rms_norm(x, eps: float = 1e-5, out=None, stream=None):
    _need(x, torch.float32, "x")
    T, d = x.shape
    out = torch.empty_like(x) if out is None else out
    _check(lib().moe_rms_norm(_p(x), T, d, float(eps), _p(out), _stream(stream)), "moe_rms_norm")
    return out


def moe_layer_forward(x, w_gate, bias, layer: LayerWeights, k: int, normalize: int = 1,
                      route_scale: float = 1.0, mode: int = MOE_MODE_AUTO, residual=None, out=None,
                      topk_idx=None, topk_w=None, hits=None, ws=None, err=None, stream=None,
                      top_p: float | None = None):
    """moe_layer_forward, or moe_layer_forward_topp when top_p is given."""
    _need(x, torch.float32, "x")
    T, d = x.shape
    dev = x.device
    out = torch.empty((T, d), dtype=torch.float32, device=dev) if out is None else out
    if ws is None:
        ws = workspace(layer_workspace_bytes(T, k, layer.E, d, layer.f, mode), dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    wp, wn = _ws_ptr(ws)
    if top_p is None:
        _check(lib().moe_layer_forward(_p(x), _p(w_gate), _p(bias), ctypes.byref(layer.c), _p(residual), T, k,
                                       int(normalize), float(route_scale), mode, _p(out), _p(topk_idx),
                                       _p(topk_w), _p(hits), wp, wn, _p(err), _stream(stream)), "moe_layer_forward")
    else:
        _check(lib().moe_layer_forward_topp(_p(x), _p(w_gate), _p(bias), ctypes.byref(layer.c), _p(residual), T,
                                            k, int(normalize), float(route_scale), float(top_p), mode, _p(out),
                                            _p(topk_idx), _p(topk_w), _p(hits), wp, wn, _p(err),
                                            _stream(stream)), "moe_layer_forward_topp")
    return out, err


def moe_layer_forward_norm(x, w_gate, bias, layer: LayerWeights, k: int, eps: float = 1e-5, normalize: int = 1,
                           route_scale: float = 1.0, mode: int = MOE_MODE_AUTO, residual=None, out=None,
                           out_normed=None, topk_idx=None, topk_w=None, hits=None, ws=None, err=None, stream=None,
                           top_p: float = 1.0):
    """moe_layer_forward_norm: the layer's out and RMSNorm(out) (the next layer's input)."""
    _need(x, torch.float32, "x")
    T, d = x.shape
    dev = x.device
    out = torch.empty((T, d), dtype=torch.float32, device=dev) if out is None else out
    out_normed = torch.empty((T, d), dtype=torch.float32, device=dev) if out_normed is None else out_normed
    if ws is None:
        ws = workspace(layer_workspace_bytes(T, k, layer.E, d, layer.f, mode), dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    wp, wn = _ws_ptr(ws)
    _check(lib().moe_layer_forward_norm(_p(x), _p(w_gate), _p(bias), ctypes.byref(layer.c), _p(residual), T, k,
                                        int(normalize), float(route_scale), float(top_p), mode, _p(out),
                                        _p(out_normed), float(eps), _p(topk_idx), _p(topk_w), _p(hits), wp, wn,
                                        _p(err), _stream(stream)), "moe_layer_forward_norm")
    return out, out_normed, err


def layer_host_workspace_bytes(T: int, k: int, E: int, d: int, f: int, mode: int = MOE_MODE_AUTO) -> int:
    return int(lib().moe_layer_host_workspace_bytes(T, k, E, d, f, mode))


def moe_layer_forward_host(x_host, w_gate, bias, layer: LayerWeights, k: int, normalize: int = 1,
                           route_scale: float = 1.0, mode: int = MOE_MODE_AUTO, residual=None, out_host=None,
                           topk_idx=None, topk_w=None, hits=None, ws=None, err=None, stream=None,
                           top_p: float = 1.0):
    """moe_layer_forward_host: x_host and out_host are CPU float32 tensors [T][d] (page-locked for
    asynchronous copies); the device tensors as in moe_layer_forward."""
    if x_host.device.type != "cpu" or x_host.dtype != torch.float32 or not x_host.is_contiguous():
        raise TypeError("x_host must be a contiguous float32 CPU tensor")
    T, d = x_host.shape
    dev = w_gate.device
    out_host = torch.empty((T, d), dtype=torch.float32).pin_memory() if out_host is None else out_host
    if out_host.device.type != "cpu" or out_host.dtype != torch.float32 or not out_host.is_contiguous():
        raise TypeError("out_host must be a contiguous float32 CPU tensor")
    if ws is None:
        ws = workspace(layer_host_workspace_bytes(T, k, layer.E, d, layer.f, mode), dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    wp, wn = _ws_ptr(ws)
    _check(lib().moe_layer_forward_host(ctypes.c_void_p(x_host.data_ptr()), _p(w_gate), _p(bias),
                                        ctypes.byref(layer.c), _p(residual), T, k, int(normalize),
                                        float(route_scale), float(top_p), mode,
                                        ctypes.c_void_p(out_host.data_ptr()), _p(topk_idx), _p(topk_w), _p(hits),
                                        wp, wn, _p(err), _stream(stream)), "moe_layer_forward_host")
    return out_host, err


def header_functions() -> list[str]:
    """Names of the functions include/moe.h declares (for export checks)."""
    import re
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*MOE_API\s+(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)))


class ExpertTier:
    """A layer's routed experts in page-locked host memory with n_slots of them cached in device
    memory (moe_tier_*).  host_q/host_s: pinned CPU tensors [E * q_bytes] uint8 / [E * s_count]
    float32; the slot arrays are allocated here as torch device tensors (the library allocates no
    device memory)."""

    def __init__(self, host_q: torch.Tensor, host_s: torch.Tensor, E: int, d: int, f: int, n_slots: int,
                 G: int = 32, device=None):
        if host_q.is_cuda or host_s.is_cuda or not (host_q.is_pinned() and host_s.is_pinned()):
            raise ValueError("host_q and host_s must be page-locked CPU tensors")
        if host_q.dtype != torch.uint8 or host_s.dtype != torch.float32:
            raise ValueError("host_q must be uint8 and host_s float32")
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        qb, sc = expert_q_bytes(d, f), expert_s_count(d, f, G)
        self.host_q, self.host_s = host_q, host_s
        self.slot_q = torch.empty(n_slots * qb, dtype=torch.uint8, device=device)
        self.slot_s = torch.empty(n_slots * sc, dtype=torch.float32, device=device)
        self.E, self.d, self.f, self.G, self.n_slots = E, d, f, G, n_slots
        h = ctypes.c_void_p()
        _check(lib().moe_tier_create(E, d, f, G, ctypes.c_void_p(host_q.data_ptr()),
                                     ctypes.c_void_p(host_s.data_ptr()), _p(self.slot_q), _p(self.slot_s), n_slots,
                                     ctypes.byref(h)), "moe_tier_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            lib().moe_tier_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def pin(self, experts, copy_stream=None):
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(experts, dtype=np.int32))
        _check(lib().moe_tier_pin(self.h, ids.ctypes.data_as(ctypes.c_void_p), ids.size, _stream(copy_stream)),
               "moe_tier_pin")

    def prefetch(self, experts, copy_stream=None):
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(experts, dtype=np.int32))
        _check(lib().moe_tier_prefetch(self.h, ids.ctypes.data_as(ctypes.c_void_p), ids.size, _stream(copy_stream)),
               "moe_tier_prefetch")

    def unpin_all(self):
        _check(lib().moe_tier_unpin_all(self.h), "moe_tier_unpin_all")

    def stats(self) -> dict:
        import numpy as np
        st = np.zeros(4, np.uint64)
        _check(lib().moe_tier_stats(self.h, st.ctypes.data_as(ctypes.c_void_p)), "moe_tier_stats")
        return {"hits": int(st[0]), "misses": int(st[1]), "bytes_copied": int(st[2]), "calls": int(st[3])}

    def slots(self):
        import numpy as np
        ex = np.zeros(self.n_slots, np.int32)
        pn = np.zeros(self.n_slots, np.uint8)
        _check(lib().moe_tier_slots(self.h, ex.ctypes.data_as(ctypes.c_void_p), pn.ctypes.data_as(ctypes.c_void_p)),
               "moe_tier_slots")
        return ex, pn.astype(bool)


def tier_workspace_bytes(T: int, k: int, E: int, d: int, f: int, mode: int = MOE_MODE_AUTO) -> int:
    return int(lib().moe_tier_workspace_bytes(T, k, E, d, f, mode))


def moe_layer_forward_tier(x, w_gate, bias, tier: ExpertTier, shared_q, shared_s, k: int, normalize: int = 1,
                           route_scale: float = 1.0, top_p: float = 1.0, mode: int = MOE_MODE_AUTO, residual=None,
                           out=None, topk_idx=None, topk_w=None, hits=None, ws=None, err=None, stream=None,
                           copy_stream=None):
    """moe_layer_forward over an expert tier: waits on the host for the routing, copies the missing
    experts on copy_stream (a separate torch.cuda.Stream) while the resident ones are computed."""
    _need(x, torch.float32, "x")
    _need(shared_q, torch.uint8, "shared_q")
    _need(shared_s, torch.float32, "shared_s")
    if copy_stream is None:
        raise ValueError("copy_stream: a CUDA stream other than the compute stream")
    T, d = x.shape
    dev = x.device
    out = torch.empty((T, d), dtype=torch.float32, device=dev) if out is None else out
    if ws is None:
        ws = workspace(tier_workspace_bytes(T, k, tier.E, d, tier.f, mode), dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    wp, wn = _ws_ptr(ws)
    _check(lib().moe_layer_forward_tier(_p(x), _p(w_gate), _p(bias), tier.h, _p(shared_q), _p(shared_s),
                                        _p(residual), T, k, int(normalize), float(route_scale), float(top_p), mode,
                                        _p(out), _p(topk_idx), _p(topk_w), _p(hits), wp, wn, _p(err),
                                        _stream(stream), _stream(copy_stream)), "moe_layer_forward_tier")
    return out, err


def usage_save(path: str, hits, model_id: int) -> None:
    """Save hit counters [layers][E] (numpy uint64 or int64, host) for model_id."""
    import numpy as np
    h = np.ascontiguousarray(np.asarray(hits).astype(np.uint64))
    if h.ndim != 2:
        raise ValueError("hits must be [layers][E]")
    _check(lib().moe_usage_save(os.fsencode(path), h.ctypes.data_as(ctypes.c_void_p), h.shape[0], h.shape[1],
                                int(model_id) & (2 ** 64 - 1)), "moe_usage_save")


def usage_load(path: str, layers: int, E: int, model_id: int):
    """Hit counters [layers][E] from a usage file written for model_id; raises MoeError (status
    MOE_ERR_STALE for another model or shape, MOE_ERR_INVALID_ARG for a missing or damaged file)."""
    import numpy as np
    h = np.zeros((layers, E), np.uint64)
    _check(lib().moe_usage_load(os.fsencode(path), h.ctypes.data_as(ctypes.c_void_p), layers, E,
                                int(model_id) & (2 ** 64 - 1)), "moe_usage_load")
    return h


def usage_top(hits_layer, n: int):
    """The n most used experts of one layer (count descending, ties by ascending id)."""
    import numpy as np
    h = np.ascontiguousarray(np.asarray(hits_layer).astype(np.uint64)).reshape(-1)
    out = np.zeros(n, np.int32)
    _check(lib().moe_usage_top(h.ctypes.data_as(ctypes.c_void_p), h.size, n, out.ctypes.data_as(ctypes.c_void_p)),
           "moe_usage_top")
    return out
