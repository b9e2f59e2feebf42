"""CPU oracle of the routed-expert layer -- TEST INFRASTRUCTURE.

A ctypes binding to ``k3moe_oracle.c``, the plain fp64 C restatement of the
layer from the kimi-k3-in-c README (Part II: section 4 for MXFP4, section 5 for
the floating-point contract, section 9 for the router, the Stable LatentMoE
expert loop and SiTU-GLU).  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package; the GPU library never
does, and the two share no code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3moe_oracle.c")
_LIB = os.path.join(_HERE, "libk3moe_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EMISSING, ENOMEM = 0, 1, 2, 3


class Cfg(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("group", ctypes.c_int32),
                ("situ_b1", ctypes.c_float), ("situ_b2", ctypes.c_float),
                ("renorm", ctypes.c_int32), ("routed_scale", ctypes.c_float)]


class Expert(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w1_packed", "w1_scale", "w3_packed", "w3_scale", "w2_packed", "w2_scale")]


def build(force: bool = False) -> str:
    """Compile the oracle into ``libk3moe_oracle.so`` beside its source."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                        "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
        return _LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        p, i, f, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
        cp = ctypes.POINTER(Cfg)
        sig = {
            "k3o_check_cfg": (i, [cp]),
            "k3o_e2m1": (d, [i]),
            "k3o_e8m0": (d, [i]),
            "k3o_bf16": (f, [ctypes.c_uint16]),
            "k3o_mxfp4_weight": (d, [p, p, i, i, i, i]),
            "k3o_mxfp4_matvec": (None, [p, p, p, p, i, i, i]),
            "k3o_bf16_matvec": (None, [p, p, p, i, i]),
            "k3o_situ": (d, [d, d, d, d]),
            "k3o_route": (i, [cp, i, p, p, p, p, p, p, p, p]),
            "k3o_select": (i, [cp, i, p, p, p, p, p]),
            "k3o_perm": (i, [i, i, i, p, p, p]),
            "k3o_forward": (i, [cp, i, p, p, p, p, p, p, p, p, p]),
            "k3o_moe": (i, [cp, i, p, p, p, p, p, p, p, p, p, p]),
            "k3o_forward_full": (i, [cp, i, i, d, i] + [p] * 11),
            "k3o_num_threads": (i, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return a.ctypes.data


def cfg(d, f, n_experts, top_k, n_shared, group=32, situ_b1=4.0, situ_b2=25.0,
        renorm=1, routed_scale=1.0) -> Cfg:
    return Cfg(d, f, n_experts, top_k, n_shared, group, situ_b1, situ_b2, renorm, routed_scale)


def _check(rc, what):
    if rc != OK:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return lib().k3o_num_threads()


def e2m1(code: int) -> float:
    return lib().k3o_e2m1(code)


def e8m0(byte: int) -> float:
    return lib().k3o_e8m0(byte)


def situ(g: float, u: float, b1: float = 4.0, b2: float = 25.0) -> float:
    return lib().k3o_situ(g, u, b1, b2)


def mxfp4_weight(packed, scales, cols, group, row, col) -> float:
    return lib().k3o_mxfp4_weight(_p(packed), _p(scales), cols, group, row, col)


def mxfp4_matvec(x: np.ndarray, packed: np.ndarray, scales: np.ndarray, group: int = 32) -> np.ndarray:
    rows, half = packed.shape
    xin = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    lib().k3o_mxfp4_matvec(_p(y), _p(xin), _p(packed), _p(scales), 2 * half, rows, group)
    return y


def bf16_matvec(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    rows, cols = W.shape
    xin = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    lib().k3o_bf16_matvec(_p(y), _p(xin), _p(W), cols, rows)
    return y


def route(c: Cfg, x: np.ndarray, Wr: np.ndarray, bias=None, want_scores: bool = False):
    """Returns idx [T,k] int32, w [T,k] float32, gap [T] float32 (+ sc, ch [T,E])."""
    T = x.shape[0]
    idx = np.empty((T, c.top_k), dtype=np.int32)
    w = np.empty((T, c.top_k), dtype=np.float32)
    gap = np.empty(T, dtype=np.float32)
    sc = np.empty((T, c.n_experts), dtype=np.float32) if want_scores else None
    ch = np.empty((T, c.n_experts), dtype=np.float32) if want_scores else None
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _check(lib().k3o_route(ctypes.byref(c), T, _p(x), _p(Wr), _p(b), _p(idx), _p(w),
                           _p(sc), _p(ch), _p(gap)), "route")
    if want_scores:
        return idx, w, gap, sc, ch
    return idx, w, gap


def select(c: Cfg, sc: np.ndarray, ch: np.ndarray):
    T = sc.shape[0]
    idx = np.empty((T, c.top_k), dtype=np.int32)
    w = np.empty((T, c.top_k), dtype=np.float32)
    gap = np.empty(T, dtype=np.float32)
    _check(lib().k3o_select(ctypes.byref(c), T, _p(np.ascontiguousarray(sc, np.float32)),
                            _p(np.ascontiguousarray(ch, np.float32)), _p(idx), _p(w), _p(gap)),
           "select")
    return idx, w, gap


def perm(idx: np.ndarray, E: int):
    """Stable counting sort of the slots by expert: (offsets [E+1], perm [T*k])."""
    T, k = idx.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    pm = np.empty(T * k, dtype=np.int32)
    _check(lib().k3o_perm(T, E, k, _p(np.ascontiguousarray(idx, np.int32)), _p(offsets), _p(pm)),
           "perm")
    return offsets, pm


class ExpertTable:
    """Per-expert pointer table for the oracle; experts not supplied are NULL."""

    def __init__(self, n_experts: int, experts: dict):
        self.keep = []
        self.arr = (Expert * n_experts)()
        for e, t in experts.items():
            fields = {}
            for name in ("w1_packed", "w1_scale", "w3_packed", "w3_scale", "w2_packed", "w2_scale"):
                a = np.ascontiguousarray(t[name], dtype=np.uint8)
                self.keep.append(a)
                fields[name] = a.ctypes.data
            self.arr[e] = Expert(**fields)


def forward(c: Cfg, x: np.ndarray, idx: np.ndarray, w: np.ndarray, experts: dict,
            shared: dict | None, want_shared: bool = False):
    """The expert part of the layer for given routing; returns out [T,d] float32
    (and the shared-expert part alone when asked)."""
    T = x.shape[0]
    table = ExpertTable(c.n_experts, experts)
    out = np.empty((T, c.d), dtype=np.float32)
    outs = np.empty((T, c.d), dtype=np.float32) if want_shared else None
    sh = shared or {}
    w1, w3, w2 = (np.ascontiguousarray(sh[n]) if n in sh else None for n in ("w1", "w3", "w2"))
    _check(lib().k3o_forward(ctypes.byref(c), T, _p(np.ascontiguousarray(x)),
                             _p(np.ascontiguousarray(idx, np.int32)),
                             _p(np.ascontiguousarray(w, np.float32)), ctypes.cast(table.arr, ctypes.c_void_p),
                             _p(w1), _p(w3), _p(w2), _p(out), _p(outs)), "forward")
    return (out, outs) if want_shared else out


def forward_full(c: Cfg, H: int, latent_norm: int, eps: float, h: np.ndarray, idx: np.ndarray,
                 w: np.ndarray, Wd: np.ndarray, experts: dict, gain, Wu: np.ndarray,
                 shared: dict | None) -> np.ndarray:
    """The full-width block for given routing (route first with ``route`` on a config
    whose d is H): h [T,H] bf16 bits, Wd [d,H], Wu [H,d] bf16 bits, gain [d] float32,
    shared {"w1","w3": [S*f,H], "w2": [H,S*f]} bf16 bits.  Returns out [T,H] float32."""
    T = h.shape[0]
    table = ExpertTable(c.n_experts, experts)
    out = np.empty((T, H), dtype=np.float32)
    sh = shared or {}
    w1, w3, w2 = (np.ascontiguousarray(sh[n]) if n in sh else None for n in ("w1", "w3", "w2"))
    g = None if gain is None else np.ascontiguousarray(gain, dtype=np.float32)
    _check(lib().k3o_forward_full(ctypes.byref(c), H, latent_norm, eps, T,
                                  _p(np.ascontiguousarray(h)), _p(np.ascontiguousarray(idx, np.int32)),
                                  _p(np.ascontiguousarray(w, np.float32)), _p(np.ascontiguousarray(Wd)),
                                  ctypes.cast(table.arr, ctypes.c_void_p), _p(g),
                                  _p(np.ascontiguousarray(Wu)), _p(w1), _p(w3), _p(w2), _p(out)),
           "forward_full")
    return out
