"""CPU oracle for one Colibri GLM-5.2 MoE layer (fp64, plain C) -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never calls it, and it imports nothing
from the CUDA package.

The arithmetic lives in ``moe_oracle.c`` (see its header for the definitions
and the passages of "Public Colibri Observation and Revision Ledger" and the
colibri README that they follow).  This module compiles that file with gcc and
marshals numpy arrays to it; it performs no arithmetic of its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmoe_oracle.so`` (gcc, -O2).

    ``-ffp-contract=off`` keeps a*b+c as two rounded operations on every host
    (gcc contracts to FMA by default on aarch64), so x86 and Arm give the same
    fp64 bits.  OpenMP is used when the compiler supports it.
    """
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
        return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_D = ctypes.c_double


class _Layer(ctypes.Structure):
    _fields_ = [("x", _P), ("wg", _P), ("bias", _P), ("q_base", _P), ("s_base", _P),
                ("shared_q", _P), ("shared_s", _P), ("res", _P),
                ("T", _I), ("d", _I), ("f", _I), ("E", _I), ("k", _I), ("G", _I),
                ("normalize", _I), ("route_scale", _D), ("top_p", _D)]


def _declare(L: ctypes.CDLL) -> None:
    L.oracle_int4_unpack.argtypes = [_P, _I64, _P]
    L.oracle_int4_pack.argtypes = [_P, _I64, _P]
    L.oracle_int4_pack.restype = _I64
    L.oracle_dequant.argtypes = [_P, _P, _I64, _I64, _I, _P]
    L.oracle_expert_q_bytes.argtypes = [_I64, _I64]
    L.oracle_expert_q_bytes.restype = _I64
    L.oracle_expert_s_count.argtypes = [_I64, _I64, _I]
    L.oracle_expert_s_count.restype = _I64
    L.oracle_router_logits.argtypes = [_P, _P, _I, _I, _I, _P]
    L.oracle_route.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _D, _P, _P, _P, _P]
    L.oracle_route_topp.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _D, _D, _P, _P, _P, _P]
    L.oracle_route_from_logits.argtypes = [_P, _P, _I, _I, _I, _I, _D, _D, _P, _P, _P]
    L.oracle_union.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]
    L.oracle_union.restype = _I
    L.oracle_hits.argtypes = [_P, _I, _P]
    L.oracle_expert_ffn.argtypes = [_P, _P, _P, _I, _I, _I, _P]
    L.oracle_expert_ffn_tokens.argtypes = [_P, _P, _I, _P, _P, _I, _I, _I, _P]
    L.oracle_moe_layer_tokens.argtypes = [ctypes.POINTER(_Layer), _P, _I, _P, _P, _P]
    L.oracle_moe_layer_union.argtypes = [ctypes.POINTER(_Layer), _P, _P, _P, _P, _P,
                                         _P, _P, _P, _P]
    L.oracle_moe_layer_union.restype = _I
    L.oracle_threads.restype = _I
    L.oracle_set_threads.argtypes = [_I]
    L.oracle_rms_norm.argtypes = [_P, _I, _I, _D, _P]


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_P)


def threads() -> int:
    return int(lib().oracle_threads())


def set_threads(n: int) -> None:
    """OpenMP thread count of later oracle calls (results do not depend on it)."""
    lib().oracle_set_threads(int(n))


# ------------------------------------------------------------------ int4 ----

def int4_unpack(q: np.ndarray, n: int) -> np.ndarray:
    q = _c(q, np.uint8).reshape(-1)
    assert q.size * 2 >= n
    v = np.empty(n, dtype=np.int8)
    lib().oracle_int4_unpack(_ptr(q), n, _ptr(v))
    return v


def int4_pack(v: np.ndarray) -> tuple[np.ndarray, int]:
    v = _c(v, np.int8).reshape(-1)
    q = np.empty((v.size + 1) // 2, dtype=np.uint8)
    bad = lib().oracle_int4_pack(_ptr(v), v.size, _ptr(q))
    return q, int(bad)


def dequant(q: np.ndarray, s: np.ndarray, rows: int, cols: int, G: int) -> np.ndarray:
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    assert q.size >= rows * cols // 2 and s.size >= rows * cols // G
    w = np.empty((rows, cols), dtype=np.float64)
    lib().oracle_dequant(_ptr(q), _ptr(s), rows, cols, G, _ptr(w))
    return w


def expert_q_bytes(d: int, f: int) -> int:
    return int(lib().oracle_expert_q_bytes(d, f))


def expert_s_count(d: int, f: int, G: int) -> int:
    return int(lib().oracle_expert_s_count(d, f, G))


# ----------------------------------------------------------------- route ----

def router_logits(x: np.ndarray, wg: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    wg = _c(wg, np.float32)
    T, d = x.shape
    E = wg.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    lib().oracle_router_logits(_ptr(x), _ptr(wg), T, d, E, _ptr(out))
    return out


def route(x, wg, bias, k: int, normalize: int = 1, route_scale: float = 1.0, top_p: float = 1.0):
    """Returns (idx [T,k] int32, w [T,k] f64, logits [T,E] f64, keys [T,E] f64).
    top_p < 1 empties the pruned slots (id -1, weight 0)."""
    x = _c(x, np.float32)
    wg = _c(wg, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    T, d = x.shape
    E = wg.shape[0]
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    keys = np.empty((T, E), dtype=np.float64)
    lib().oracle_route_topp(_ptr(x), _ptr(wg), _ptr(bias), T, d, E, k, int(normalize),
                            float(route_scale), float(top_p), _ptr(idx), _ptr(w), _ptr(logits),
                            _ptr(keys))
    return idx, w, logits, keys


def route_from_logits(logits, bias, k: int, normalize: int = 1, route_scale: float = 1.0,
                      top_p: float = 1.0):
    """Routing of given fp64 logits [T,E]: (idx, w, keys) as in route()."""
    logits = _c(logits, np.float64)
    bias = None if bias is None else _c(bias, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    keys = np.empty((T, E), dtype=np.float64)
    lib().oracle_route_from_logits(_ptr(logits), _ptr(bias), T, E, k, int(normalize),
                                   float(route_scale), float(top_p), _ptr(idx), _ptr(w), _ptr(keys))
    return idx, w, keys


# ----------------------------------------------------------------- union ----

def union(idx: np.ndarray, E: int) -> dict:
    idx = _c(idx, np.int32)
    T, k = idx.shape
    P = T * k
    out = dict(counts=np.empty(E, np.int32), offsets=np.empty(E + 1, np.int32),
               perm=np.empty(P, np.int32), sorted_pair=np.empty(P, np.int32),
               uniq=np.empty(E, np.int32), n_uniq=np.zeros(1, np.int32))
    rc = lib().oracle_union(_ptr(idx), T, k, E, _ptr(out["counts"]), _ptr(out["offsets"]),
                            _ptr(out["perm"]), _ptr(out["sorted_pair"]), _ptr(out["uniq"]),
                            _ptr(out["n_uniq"]))
    if rc != 0:
        raise ValueError("expert id out of range")
    out["n_uniq"] = int(out["n_uniq"][0])
    return out


def hits(counts: np.ndarray, hits_arr: np.ndarray) -> None:
    counts = _c(counts, np.int32)
    assert hits_arr.dtype == np.uint64 and hits_arr.flags.c_contiguous
    lib().oracle_hits(_ptr(counts), counts.size, _ptr(hits_arr))


# ------------------------------------------------------------------- FFN ----

def expert_ffn(x_row, q_e, s_e, d: int, f: int, G: int) -> np.ndarray:
    x_row = _c(x_row, np.float32).reshape(-1)
    q_e = _c(q_e, np.uint8).reshape(-1)
    s_e = _c(s_e, np.float32).reshape(-1)
    assert x_row.size == d and q_e.size >= 3 * d * f // 2 and s_e.size >= 3 * d * f // G
    y = np.empty(d, dtype=np.float64)
    lib().oracle_expert_ffn(_ptr(x_row), _ptr(q_e), _ptr(s_e), d, f, G, _ptr(y))
    return y


def expert_ffn_tokens(x, tokens, q_e, s_e, d: int, f: int, G: int) -> np.ndarray:
    x = _c(x, np.float32)
    tokens = _c(tokens, np.int32).reshape(-1)
    q_e = _c(q_e, np.uint8).reshape(-1)
    s_e = _c(s_e, np.float32).reshape(-1)
    y = np.empty((tokens.size, d), dtype=np.float64)
    lib().oracle_expert_ffn_tokens(_ptr(x), _ptr(tokens), tokens.size, _ptr(q_e), _ptr(s_e),
                                   d, f, G, _ptr(y))
    return y


# ----------------------------------------------------------------- stack ----

def rms_norm(x: np.ndarray, eps: float = 1e-5) -> np.ndarray:
    """Rows of x divided by their RMS (unit weight), fp64: the input of a stacked layer."""
    x = _c(x, np.float32)
    T, d = x.shape
    out = np.empty((T, d), dtype=np.float64)
    lib().oracle_rms_norm(_ptr(x), T, d, float(eps), _ptr(out))
    return out


# ----------------------------------------------------------------- layer ----

class Layer:
    """One MoE layer's inputs (numpy, host).  Arrays are kept alive here."""

    def __init__(self, x, wg, bias, q_base, s_base, shared_q, shared_s, *, d, f, E, k,
                 G=32, normalize=1, route_scale=1.0, res=None, top_p=1.0):
        self.x = _c(x, np.float32)
        self.wg = _c(wg, np.float32)
        self.bias = None if bias is None else _c(bias, np.float32)
        self.q_base = _c(q_base, np.uint8)
        self.s_base = _c(s_base, np.float32)
        self.shared_q = _c(shared_q, np.uint8)
        self.shared_s = _c(shared_s, np.float32)
        self.res = None if res is None else _c(res, np.float32)
        self.T = self.x.shape[0]
        self.d, self.f, self.E, self.k, self.G = d, f, E, k, G
        self.normalize, self.route_scale, self.top_p = int(normalize), float(route_scale), float(top_p)
        assert self.x.shape == (self.T, d) and self.wg.shape == (E, d)
        assert self.q_base.size >= E * expert_q_bytes(d, f)
        assert self.s_base.size >= E * expert_s_count(d, f, G)

    def _struct(self) -> _Layer:
        return _Layer(_ptr(self.x), _ptr(self.wg), _ptr(self.bias), _ptr(self.q_base),
                      _ptr(self.s_base), _ptr(self.shared_q), _ptr(self.shared_s),
                      _ptr(self.res), self.T, self.d, self.f, self.E, self.k, self.G,
                      self.normalize, self.route_scale, self.top_p)

    def tokens(self, tokens) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """Dense masked evaluation of the listed tokens: (idx, w, out fp64)."""
        tokens = _c(tokens, np.int32).reshape(-1)
        n = tokens.size
        idx = np.empty((n, self.k), np.int32)
        w = np.empty((n, self.k), np.float64)
        out = np.empty((n, self.d), np.float64)
        s = self._struct()
        lib().oracle_moe_layer_tokens(ctypes.byref(s), _ptr(tokens), n, _ptr(idx), _ptr(w),
                                      _ptr(out))
        return idx, w, out

    def dense(self):
        return self.tokens(np.arange(self.T, dtype=np.int32))

    def union_path(self) -> dict:
        """Union-path evaluation of all tokens; returns routing, union arrays and out."""
        T, k, E, d = self.T, self.k, self.E, self.d
        r = dict(idx=np.empty((T, k), np.int32), w=np.empty((T, k), np.float64),
                 counts=np.empty(E, np.int32), offsets=np.empty(E + 1, np.int32),
                 perm=np.empty(T * k, np.int32), sorted_pair=np.empty(T * k, np.int32),
                 uniq=np.empty(E, np.int32), n_uniq=np.zeros(1, np.int32),
                 out=np.empty((T, d), np.float64))
        s = self._struct()
        rc = lib().oracle_moe_layer_union(ctypes.byref(s), _ptr(r["idx"]), _ptr(r["w"]),
                                          _ptr(r["counts"]), _ptr(r["offsets"]),
                                          _ptr(r["perm"]), _ptr(r["sorted_pair"]),
                                          _ptr(r["uniq"]), _ptr(r["n_uniq"]), _ptr(r["out"]))
        if rc != 0:
            raise ValueError("expert id out of range")
        r["n_uniq"] = int(r["n_uniq"][0])
        return r
