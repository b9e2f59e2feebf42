"""Seeded synthetic inputs for the routed-expert layer of a Kimi-K3-style latent MoE.

This package draws the layer's inputs and holds none of its arithmetic.  The
CPU oracle (``oracle/``) and the GPU library are both fed from it, so the two
see the same bytes.  The generator itself is C (``k3moe_gen.c``): a
counter-based splitmix64 stream, so any slice of any tensor is a pure function
of (seed, stream, index) and can be regenerated alone -- one routed expert at
a time, for instance, which is how the oracle gets the few experts it needs
without materialising the 15.7 GB table on the host.

Workloads (shapes and distributions of the routed-expert layer as the Kimi K3
write-ups state them: 896 routed experts, top-16, 2 shared experts, latent
3584, expert FFN 3072, MXFP4 experts with one E8M0 scale per 32 weights):

=============  =====  ====  ====  ===  ==  =  ===========================================
name           T      d     f     E    k   S  extra
=============  =====  ====  ====  ===  ==  =  ===========================================
tiny           4      256   128   32   4   1  scale exponents U[-8,-4]
decode_t1      1      3584  3072  896  16  2  scale exponents U[-10,-6]
decode_t64     64     3584  3072  896  16  2  as decode_t1
prefill_t4096  4096   3584  3072  896  16  2  1% of activation rows scaled by 8
prefill_t16k   16384  3584  3072  896  16  2  Zipf(s=1.1) routing bias, seeded ranks
full_tiny      4      128   128   8    2   1  full-width block, hidden 256
full_t1        1      3584  3072  896  16  2  full-width block, hidden 7168
full_t4096     4096   3584  3072  896  16  2  full-width block, hidden 7168, 1% rows x8
=============  =====  ====  ====  ===  ==  =  ===========================================

The full-width block (the Stable LatentMoE step around the layer) adds tokens of
width H ~ N(0,1), a full-width router ~ N(0, 0.02), down [d,H] ~ N(0, 1/H) and up
[H,d] ~ N(0, 1/d) projections, an RMSNorm gain 1 + N(0, 0.01), and the shared
experts fused to width S*f on the full width, ~ N(0, sigma_s).

Activations bf16 ~ N(0,1); router weights bf16 ~ N(0, 0.02); E2M1 codes
uniform over all 16 codes (so packed bytes are uniform over 0..255); shared
experts bf16 ~ N(0, sigma_s) with sigma_s the RMS of the routed weights.
Workload i uses seed i.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3moe_gen.c")
_LIB = os.path.join(_HERE, "libk3moe_gen.so")
_lock = threading.Lock()
_lib = None

# Stream ids: one per tensor, so tensors never share draws.
STREAM_X = 1
STREAM_ROUTER = 2
STREAM_BIAS_RANKS = 3
STREAM_OUTLIER_ROWS = 4
STREAM_SHARED_W1 = 10
STREAM_SHARED_W3 = 11
STREAM_SHARED_W2 = 12
STREAM_FULL_H = 20
STREAM_FULL_ROUTER = 21
STREAM_FULL_DOWN = 22
STREAM_FULL_UP = 23
STREAM_FULL_GAIN = 24
STREAM_FULL_SH1 = 25
STREAM_FULL_SH3 = 26
STREAM_FULL_SH2 = 27
EXPERT_TENSORS = ("w1_packed", "w1_scale", "w3_packed", "w3_scale", "w2_packed", "w2_scale")


def expert_stream(e: int, tensor: int) -> int:
    """Stream id of routed expert ``e``'s tensor number ``tensor`` (EXPERT_TENSORS order)."""
    return (1 << 40) + 8 * e + tensor


def build(force: bool = False) -> str:
    """Compile the generator into ``libk3moe_gen.so`` beside its source."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, sz, p = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
        lib.k3g_hash.restype = u64
        lib.k3g_hash.argtypes = [u64, u64, u64]
        lib.k3g_uniform.restype = ctypes.c_double
        lib.k3g_uniform.argtypes = [u64, u64, u64]
        lib.k3g_normal.restype = ctypes.c_double
        lib.k3g_normal.argtypes = [u64, u64, u64]
        lib.k3g_log.restype = ctypes.c_double
        lib.k3g_log.argtypes = [ctypes.c_double]
        lib.k3g_f32_to_bf16.restype = ctypes.c_uint16
        lib.k3g_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.k3g_bf16_normal.restype = None
        lib.k3g_bf16_normal.argtypes = [p, sz, u64, u64, u64, ctypes.c_double]
        lib.k3g_bytes.restype = None
        lib.k3g_bytes.argtypes = [p, sz, u64, u64, u64]
        lib.k3g_uniform_bytes.restype = None
        lib.k3g_uniform_bytes.argtypes = [p, sz, u64, u64, u64, ctypes.c_int, ctypes.c_int]
        lib.k3g_permutation.restype = None
        lib.k3g_permutation.argtypes = [p, ctypes.c_int32, u64, u64]
        lib.k3g_zipf_bias.restype = None
        lib.k3g_zipf_bias.argtypes = [p, ctypes.c_int32, u64, u64, ctypes.c_double, ctypes.c_double]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------------------- primitives

def bf16_normal(n: int, seed: int, stream: int, sigma: float, offset: int = 0) -> np.ndarray:
    """n bf16 draws (as uint16 bit patterns) of N(0, sigma^2)."""
    out = np.empty(n, dtype=np.uint16)
    _load().k3g_bf16_normal(_ptr(out), n, seed, stream, offset, float(sigma))
    return out


def random_bytes(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    assert offset % 8 == 0
    out = np.empty(n, dtype=np.uint8)
    _load().k3g_bytes(_ptr(out), n, seed, stream, offset)
    return out


def uniform_bytes(n: int, seed: int, stream: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _load().k3g_uniform_bytes(_ptr(out), n, seed, stream, offset, lo, hi)
    return out


def permutation(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().k3g_permutation(_ptr(out), n, seed, stream)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a 16-bit shift)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- workloads

def routed_weight_rms(exp_lo: int, exp_hi: int) -> float:
    """RMS of an MXFP4 weight with codes uniform over the 16 E2M1 codes and
    scale exponent uniform over [exp_lo, exp_hi]: sqrt(E[code^2] * E[4^e])."""
    e2m1_sq = (0.0 + 0.25 + 1.0 + 2.25 + 4.0 + 9.0 + 16.0 + 36.0) / 8.0  # 8.5625
    pow4 = sum(4.0 ** e for e in range(exp_lo, exp_hi + 1)) / (exp_hi - exp_lo + 1)
    return math.sqrt(e2m1_sq * pow4)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    S: int
    exp_lo: int
    exp_hi: int
    seed: int
    outlier_frac: float = 0.0
    outlier_scale: float = 8.0
    zipf_bias: bool = False
    zipf_s: float = 1.1
    zipf_scale: float = 0.1
    x_sigma: float = 1.0
    router_sigma: float = 0.02
    situ_b1: float = 4.0
    situ_b2: float = 25.0
    renorm: int = 1
    routed_scale: float = 1.0
    hidden: int = 0             # full-width block: width H of its tokens (0: latent layer only)
    latent_norm: int = 1        # full-width block: RMSNorm the aggregate
    rms_eps: float = 1e-5

    @property
    def shared_sigma(self) -> float:
        return routed_weight_rms(self.exp_lo, self.exp_hi)

    @property
    def scale_lo(self) -> int:
        return 127 + self.exp_lo

    @property
    def scale_hi(self) -> int:
        return 127 + self.exp_hi

    @property
    def expert_bytes(self) -> int:
        """Packed bytes of one routed expert: 3*f*d weights at 17/32 byte each."""
        return 3 * self.f * self.d * 17 // 32

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)

    def config_kwargs(self) -> dict:
        return dict(d=self.d, f=self.f, n_experts=self.E, top_k=self.k, n_shared=self.S,
                    group=32, situ_b1=self.situ_b1, situ_b2=self.situ_b2,
                    renorm=self.renorm, routed_scale=self.routed_scale)


_K3 = dict(d=3584, f=3072, E=896, k=16, S=2, exp_lo=-10, exp_hi=-6)
WORKLOADS = {
    "tiny": Workload("tiny", T=4, d=256, f=128, E=32, k=4, S=1, exp_lo=-8, exp_hi=-4, seed=0),
    "decode_t1": Workload("decode_t1", T=1, seed=1, **_K3),
    "decode_t64": Workload("decode_t64", T=64, seed=2, **_K3),
    "prefill_t4096": Workload("prefill_t4096", T=4096, seed=3, outlier_frac=0.01, **_K3),
    "prefill_t16k": Workload("prefill_t16k", T=16384, seed=4, zipf_bias=True, **_K3),
    # the full-width Stable LatentMoE block around the layer (hidden 7168)
    "full_tiny": Workload("full_tiny", T=4, d=128, f=128, E=8, k=2, S=1, exp_lo=-8, exp_hi=-4,
                          seed=5, hidden=256),
    "full_t1": Workload("full_t1", T=1, seed=6, hidden=7168, **_K3),
    "full_t4096": Workload("full_t4096", T=4096, seed=7, hidden=7168, outlier_frac=0.01, **_K3),
}


def make_x(w: Workload) -> np.ndarray:
    """Activations [T, d] as bf16 bits; a seeded 1% of rows scaled by 8 when asked."""
    x = bf16_normal(w.T * w.d, w.seed, STREAM_X, w.x_sigma).reshape(w.T, w.d)
    n_out = int(round(w.outlier_frac * w.T))
    if n_out:
        rows = outlier_rows(w)
        xf = bf16_to_f32(x[rows]) * np.float32(w.outlier_scale)   # exact: power of two
        x[rows] = f32_to_bf16(xf)
    return x


def outlier_rows(w: Workload) -> np.ndarray:
    n_out = int(round(w.outlier_frac * w.T))
    return np.sort(permutation(w.T, w.seed, STREAM_OUTLIER_ROWS)[:n_out])


def make_router(w: Workload) -> np.ndarray:
    """Router weights [E, d] as bf16 bits."""
    return bf16_normal(w.E * w.d, w.seed, STREAM_ROUTER, w.router_sigma).reshape(w.E, w.d)


def make_bias(w: Workload):
    """Per-expert routing bias [E] float32, or None for the unbiased workloads."""
    if not w.zipf_bias:
        return None
    out = np.empty(w.E, dtype=np.float32)
    _load().k3g_zipf_bias(_ptr(out), w.E, w.seed, STREAM_BIAS_RANKS, w.zipf_s, w.zipf_scale)
    return out


def make_expert(w: Workload, e: int) -> dict:
    """Routed expert e in checkpoint layout: packed [rows][cols/2] (low nibble =
    even column) and E8M0 scales [rows][cols/32].  w1, w3: [f, d]; w2: [d, f]."""
    f, d = w.f, w.d
    shapes = {"w1": (f, d), "w3": (f, d), "w2": (d, f)}
    out = {}
    for t, name in enumerate(EXPERT_TENSORS):
        mat, kind = name.split("_")
        rows, cols = shapes[mat]
        if kind == "packed":
            a = random_bytes(rows * cols // 2, w.seed, expert_stream(e, t)).reshape(rows, cols // 2)
        else:
            a = uniform_bytes(rows * cols // 32, w.seed, expert_stream(e, t),
                              w.scale_lo, w.scale_hi).reshape(rows, cols // 32)
        out[name] = a
    return out


def make_experts_block(w: Workload, e0: int, n: int) -> dict:
    """Experts e0..e0+n-1 stacked: each tensor gets a leading [n] axis."""
    blocks = [make_expert(w, e) for e in range(e0, e0 + n)]
    return {name: np.ascontiguousarray(np.stack([b[name] for b in blocks]))
            for name in EXPERT_TENSORS}


def make_shared(w: Workload) -> dict:
    """Dense shared experts as bf16 bits: w1, w3 [S, f, d]; w2 [S, d, f]."""
    S, f, d = w.S, w.f, w.d
    sig = w.shared_sigma
    return {
        "w1": bf16_normal(S * f * d, w.seed, STREAM_SHARED_W1, sig).reshape(S, f, d),
        "w3": bf16_normal(S * f * d, w.seed, STREAM_SHARED_W3, sig).reshape(S, f, d),
        "w2": bf16_normal(S * d * f, w.seed, STREAM_SHARED_W2, sig).reshape(S, d, f),
    }


# ----------------------------------------------------------------------------- full-width block

def make_h(w: Workload) -> np.ndarray:
    """Full-width tokens [T, H] as bf16 bits; a seeded 1% of rows scaled by 8 when asked."""
    h = bf16_normal(w.T * w.hidden, w.seed, STREAM_FULL_H, w.x_sigma).reshape(w.T, w.hidden)
    n_out = int(round(w.outlier_frac * w.T))
    if n_out:
        rows = outlier_rows(w)
        h[rows] = f32_to_bf16(bf16_to_f32(h[rows]) * np.float32(w.outlier_scale))
    return h


def make_full_router(w: Workload) -> np.ndarray:
    """Full-width router weights [E, H] as bf16 bits, N(0, router_sigma)."""
    return bf16_normal(w.E * w.hidden, w.seed, STREAM_FULL_ROUTER, w.router_sigma).reshape(w.E, w.hidden)


def make_full(w: Workload) -> dict:
    """The block's dense tensors: down [d, H] bf16 ~ N(0, 1/H) (a unit-variance token
    gives unit-variance latents), up [H, d] bf16 ~ N(0, 1/d) (likewise from the normed
    aggregate), gain [d] float32 = 1 + N(0, 0.1^2) in bf16 steps, and the fused shared
    experts sh1, sh3 [S*f, H], sh2 [H, S*f] bf16 ~ N(0, sigma_s^2)."""
    H, d, SI = w.hidden, w.d, w.S * w.f
    sig = w.shared_sigma
    return {
        "down": bf16_normal(d * H, w.seed, STREAM_FULL_DOWN, 1.0 / math.sqrt(H)).reshape(d, H),
        "up": bf16_normal(H * d, w.seed, STREAM_FULL_UP, 1.0 / math.sqrt(d)).reshape(H, d),
        "gain": (1.0 + bf16_to_f32(bf16_normal(d, w.seed, STREAM_FULL_GAIN, 0.1))).astype(np.float32),
        "sh1": bf16_normal(SI * H, w.seed, STREAM_FULL_SH1, sig).reshape(SI, H),
        "sh3": bf16_normal(SI * H, w.seed, STREAM_FULL_SH3, sig).reshape(SI, H),
        "sh2": bf16_normal(H * SI, w.seed, STREAM_FULL_SH2, sig).reshape(H, SI),
    }


__all__ = [
    "Workload", "WORKLOADS", "EXPERT_TENSORS", "build", "make_x", "make_router", "make_bias",
    "make_expert", "make_experts_block", "make_shared", "outlier_rows", "bf16_to_f32",
    "f32_to_bf16", "bf16_normal", "random_bytes", "uniform_bytes", "permutation",
    "routed_weight_rms", "expert_stream", "make_h", "make_full_router", "make_full",
]
