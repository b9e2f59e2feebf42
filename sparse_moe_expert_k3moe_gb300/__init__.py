"""Routed-expert layer of a Kimi-K3-style latent MoE on GB300 (sm_103a), and the
full-width Stable LatentMoE block around it (``k3moe_full_forward``, ``MoEBlock``).

A thin ctypes binding over ``libk3moe.so``; every function has the name of the C
entry point it calls (``include/k3moe.h``) and only marshals arguments: torch
tensors become device pointers, the current torch stream becomes the CUDA
stream.  All computation happens in the library's CUDA kernels; there is no
CPU fallback -- importing this package without the built library raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "K3MoEConfig", "K3MOE_OK", "K3MoEError", "lib", "k3moe_config", "k3moe_validate_config",
    "k3moe_packed_bytes", "k3moe_workspace_bytes", "k3moe_pack_mxfp4", "k3moe_unpack_mxfp4",
    "k3moe_route", "k3moe_router_scores", "k3moe_forward", "k3moe_forward_noalloc", "k3moe_device_status",
    "k3moe_check_wait_timeout", "k3moe_check_bounds", "k3moe_build_flags", "k3moe_strerror",
    "k3moe_launch_count", "k3moe_timing_enable", "k3moe_timing_read", "k3moe_timing_reset",
    "k3moe_set_prefill_gemm", "k3moe_get_prefill_gemm", "PREFILL_GEMM_F16", "PREFILL_GEMM_BLOCK_SCALED",
    "library_path", "MoELayer", "K3MoEFullDims", "k3moe_full_dims", "k3moe_full_workspace_bytes",
    "k3moe_full_forward", "MoEBlock",
]

_HERE = os.path.dirname(os.path.abspath(__file__))


def _lib_file() -> str:
    """The library of the variant K3MOE_BUILD_VARIANT names (libk3moe.so by default)."""
    from .build import lib_path
    return lib_path()

K3MOE_OK = 0
STATUS_NAMES = {0: "OK", 1: "EINVAL", 2: "ESHAPE", 3: "EALIGN", 4: "EWORKSPACE", 5: "ECUDA",
                6: "EDEVICE", 7: "ETIMEOUT"}
DEV_BAD_INDEX, DEV_BAD_OFFSETS, DEV_NAN_SCALE, DEV_TIMEOUT, DEV_BOUNDS = 0x1, 0x2, 0x4, 0x8, 0x10


class K3MoEConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("group", ctypes.c_int32),
                ("situ_b1", ctypes.c_float), ("situ_b2", ctypes.c_float),
                ("renorm", ctypes.c_int32), ("routed_scale", ctypes.c_float)]


class K3MoEFullDims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("latent_norm", ctypes.c_int32), ("rms_eps", ctypes.c_float)]


class K3MoEError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({k3moe_strerror(status)})")
        self.status = status


def library_path() -> str:
    return _lib_file()


_lib = None


def lib():
    """The loaded libk3moe.so.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        path = _lib_file()
        if not os.path.exists(path):
            raise ImportError(f"{os.path.basename(path)} is not built ({path}); run "
                              "`python -m sparse_moe_expert_k3moe_gb300.build`")
        L = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cp = ctypes.POINTER(K3MoEConfig)
        sig = {
            "k3moe_strerror": (ctypes.c_char_p, [ctypes.c_int]),
            "k3moe_validate_config": (ctypes.c_int, [cp]),
            "k3moe_packed_bytes": (sz, [cp]),
            "k3moe_workspace_bytes": (ctypes.c_int, [cp, i32, ctypes.POINTER(sz)]),
            "k3moe_pack_mxfp4": (ctypes.c_int, [cp, i32, i32] + [vp] * 6 + [vp, sz, vp, vp]),
            "k3moe_unpack_mxfp4": (ctypes.c_int, [cp, i32, i32, vp, sz] + [vp] * 6 + [vp]),
            "k3moe_route": (ctypes.c_int, [cp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "k3moe_router_scores": (ctypes.c_int, [cp, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
            "k3moe_forward": (ctypes.c_int, [cp, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp, vp,
                                             vp, sz, vp]),
            "k3moe_device_status": (ctypes.c_int, [vp, vp, ctypes.POINTER(i32)]),
            "k3moe_check_wait_timeout": (ctypes.c_int, [vp, i64, vp]),
            "k3moe_check_bounds": (ctypes.c_int, [vp, i32, i32, vp]),
            "k3moe_build_flags": (i32, []),
            "k3moe_forward_noalloc": (ctypes.c_int, [cp, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp,
                                                     vp, vp, vp, vp]),
            "k3moe_full_workspace_bytes": (ctypes.c_int, [cp, ctypes.POINTER(K3MoEFullDims), i32,
                                                          ctypes.POINTER(sz)]),
            "k3moe_full_forward": (ctypes.c_int, [cp, ctypes.POINTER(K3MoEFullDims), i32, vp, vp, vp, vp,
                                                  vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                  sz, vp]),
            "k3moe_launch_count": (i64, []),
            "k3moe_set_prefill_gemm": (ctypes.c_int, [i32]),
            "k3moe_get_prefill_gemm": (i32, []),
            "k3moe_timing_enable": (None, [i32]),
            "k3moe_timing_read": (i32, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i64),
                                        ctypes.POINTER(ctypes.c_double), i32]),
            "k3moe_timing_reset": (None, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


# ----------------------------------------------------------------------------- marshalling helpers

def _ptr(t):
    """Device pointer of a tensor (or None / int passthrough)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(what, rc):
    if rc != K3MOE_OK:
        raise K3MoEError(what, rc)


def k3moe_config(d, f, n_experts, top_k, n_shared, group=32, situ_b1=4.0, situ_b2=25.0,
                 renorm=1, routed_scale=1.0) -> K3MoEConfig:
    return K3MoEConfig(d, f, n_experts, top_k, n_shared, group, situ_b1, situ_b2, renorm,
                       routed_scale)


def k3moe_strerror(status: int) -> str:
    return lib().k3moe_strerror(status).decode()


def k3moe_validate_config(cfg: K3MoEConfig) -> int:
    return lib().k3moe_validate_config(ctypes.byref(cfg))


def k3moe_packed_bytes(cfg: K3MoEConfig) -> int:
    return lib().k3moe_packed_bytes(ctypes.byref(cfg))


def k3moe_workspace_bytes(cfg: K3MoEConfig, T_max: int) -> int:
    out = ctypes.c_size_t(0)
    _check("k3moe_workspace_bytes", lib().k3moe_workspace_bytes(ctypes.byref(cfg), T_max,
                                                                ctypes.byref(out)))
    return out.value


def k3moe_pack_mxfp4(cfg, expert_lo, n_in, w1_packed, w1_scale, w3_packed, w3_scale, w2_packed,
                     w2_scale, table, table_bytes=None, ws=None, stream=None):
    tb = table_bytes if table_bytes is not None else table.numel() * table.element_size()
    _check("k3moe_pack_mxfp4", lib().k3moe_pack_mxfp4(
        ctypes.byref(cfg), expert_lo, n_in, _ptr(w1_packed), _ptr(w1_scale), _ptr(w3_packed),
        _ptr(w3_scale), _ptr(w2_packed), _ptr(w2_scale), _ptr(table), tb, _ptr(ws),
        _stream(stream)))


def k3moe_unpack_mxfp4(cfg, expert_lo, n_out, table, w1_packed, w1_scale, w3_packed, w3_scale,
                       w2_packed, w2_scale, table_bytes=None, stream=None):
    tb = table_bytes if table_bytes is not None else table.numel() * table.element_size()
    _check("k3moe_unpack_mxfp4", lib().k3moe_unpack_mxfp4(
        ctypes.byref(cfg), expert_lo, n_out, _ptr(table), tb, _ptr(w1_packed), _ptr(w1_scale),
        _ptr(w3_packed), _ptr(w3_scale), _ptr(w2_packed), _ptr(w2_scale), _stream(stream)))


def k3moe_router_scores(cfg, T, x, w_router, bias, scores, choice, ws, ws_bytes=None, stream=None):
    wb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check("k3moe_router_scores", lib().k3moe_router_scores(
        ctypes.byref(cfg), T, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(scores), _ptr(choice),
        _ptr(ws), wb, _stream(stream)))


def k3moe_route(cfg, T, x, w_router, bias, idx, weight, offsets, perm, ws, ws_bytes=None,
                stream=None):
    wb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check("k3moe_route", lib().k3moe_route(
        ctypes.byref(cfg), T, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(idx), _ptr(weight),
        _ptr(offsets), _ptr(perm), _ptr(ws), wb, _stream(stream)))


def k3moe_forward(cfg, T, x, idx, weight, offsets, perm, expert_table, sh_w1, sh_w3, sh_w2, out,
                  ws, ws_bytes=None, table_bytes=None, stream=None):
    wb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    tb = table_bytes if table_bytes is not None else expert_table.numel() * expert_table.element_size()
    _check("k3moe_forward", lib().k3moe_forward(
        ctypes.byref(cfg), T, _ptr(x), _ptr(idx), _ptr(weight), _ptr(offsets), _ptr(perm),
        _ptr(expert_table), tb, _ptr(sh_w1), _ptr(sh_w3), _ptr(sh_w2), _ptr(out), _ptr(ws), wb,
        _stream(stream)))


def k3moe_check_wait_timeout(ws, limit_cycles, stream=None):
    """Runs the library's bounded waits on an mbarrier nothing arrives on, each giving up
    after limit_cycles cycles: sets the timeout bit of ws's status word."""
    _check("k3moe_check_wait_timeout", lib().k3moe_check_wait_timeout(_ptr(ws), int(limit_cycles),
                                                                      _stream(stream)))


def k3moe_check_bounds(ws, index, limit, stream=None):
    """Runs one index check of the kernels' kind on index against [0, limit): a debug
    build records K3MOE_DEV_BOUNDS in ws's status word when it fails."""
    _check("k3moe_check_bounds", lib().k3moe_check_bounds(_ptr(ws), int(index), int(limit), _stream(stream)))


def k3moe_build_flags():
    """BUILD_DEBUG (0x1) when the loaded library was compiled with -DK3MOE_DEBUG."""
    return int(lib().k3moe_build_flags())


BUILD_DEBUG = 0x1


def k3moe_forward_noalloc(cfg, T, x, idx, weight, offsets, perm, expert_table, sh_w1, sh_w3,
                          sh_w2, out, status_out=None, table_bytes=None, stream=None):
    """k3moe_forward with the library's built-in scratch instead of a workspace, for
    callers that cannot allocate device memory; see include/k3moe.h."""
    tb = table_bytes if table_bytes is not None else expert_table.numel() * expert_table.element_size()
    _check("k3moe_forward_noalloc", lib().k3moe_forward_noalloc(
        ctypes.byref(cfg), T, _ptr(x), _ptr(idx), _ptr(weight), _ptr(offsets), _ptr(perm),
        _ptr(expert_table), tb, _ptr(sh_w1), _ptr(sh_w3), _ptr(sh_w2), _ptr(out),
        _ptr(status_out), _stream(stream)))


def k3moe_full_dims(hidden, latent_norm=1, rms_eps=1e-5) -> K3MoEFullDims:
    return K3MoEFullDims(hidden, latent_norm, rms_eps)


def k3moe_full_workspace_bytes(cfg: K3MoEConfig, fd: K3MoEFullDims, T_max: int) -> int:
    out = ctypes.c_size_t(0)
    _check("k3moe_full_workspace_bytes", lib().k3moe_full_workspace_bytes(
        ctypes.byref(cfg), ctypes.byref(fd), T_max, ctypes.byref(out)))
    return out.value


def k3moe_full_forward(cfg, fd, T, h, w_router, bias, w_down, expert_table, norm_gain, w_up, sh_w1,
                       sh_w3, sh_w2, idx, weight, offsets, perm, out, ws, ws_bytes=None,
                       table_bytes=None, stream=None):
    wb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    tb = table_bytes if table_bytes is not None else expert_table.numel() * expert_table.element_size()
    _check("k3moe_full_forward", lib().k3moe_full_forward(
        ctypes.byref(cfg), ctypes.byref(fd), T, _ptr(h), _ptr(w_router), _ptr(bias), _ptr(w_down),
        _ptr(expert_table), tb, _ptr(norm_gain), _ptr(w_up), _ptr(sh_w1), _ptr(sh_w3), _ptr(sh_w2),
        _ptr(idx), _ptr(weight), _ptr(offsets), _ptr(perm), _ptr(out), _ptr(ws), wb,
        _stream(stream)))


def k3moe_device_status(ws, stream=None):
    """(status, code): synchronises the stream, reads and clears the device status word."""
    code = ctypes.c_int32(0)
    rc = lib().k3moe_device_status(_ptr(ws), _stream(stream), ctypes.byref(code))
    return rc, code.value


def k3moe_launch_count() -> int:
    return lib().k3moe_launch_count()


PREFILL_GEMM_DEFAULT, PREFILL_GEMM_F16, PREFILL_GEMM_BLOCK_SCALED = 0, 1, 2


def k3moe_set_prefill_gemm(variant: int):
    """The kernel of the routed gate/up projection on the prefill path: PREFILL_GEMM_F16
    (dequantised weights), PREFILL_GEMM_BLOCK_SCALED (kind::mxf8f6f4 on the packed codes
    and scales) or PREFILL_GEMM_DEFAULT; process-wide."""
    _check("k3moe_set_prefill_gemm", lib().k3moe_set_prefill_gemm(int(variant)))


def k3moe_get_prefill_gemm() -> int:
    return int(lib().k3moe_get_prefill_gemm())


def k3moe_timing_enable(on: bool):
    lib().k3moe_timing_enable(1 if on else 0)


def k3moe_timing_read() -> dict:
    L = lib()
    n = L.k3moe_timing_read(None, None, None, 0)
    names = (ctypes.c_char_p * max(n, 1))()
    launches = (ctypes.c_int64 * max(n, 1))()
    ms = (ctypes.c_double * max(n, 1))()
    n = L.k3moe_timing_read(names, launches, ms, n)
    return {names[i].decode(): (launches[i], ms[i]) for i in range(n)}


def k3moe_timing_reset():
    lib().k3moe_timing_reset()


# ----------------------------------------------------------------------------- convenience holders

def _capture(call, x, out):
    """call(x, out) recorded as a CUDA graph on x's device.  One eager call on a side
    stream first settles the library's cached launch attributes and GEMM plans, so that
    capture itself only enqueues work.  The graph reads x and writes out, the routing
    buffers and the workspace where they are now: copy the next tokens into x, then
    replay().  The library's launches keep their programmatic dependencies as graph edges."""
    import torch
    cur = torch.cuda.current_stream(x.device)
    side = torch.cuda.Stream(device=x.device)
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        call(x, out)
    cur.wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(x, out)
    return g


class MoELayer:
    """Holds one layer's device tensors (packed expert table, router, bias,
    shared experts) and a workspace, and calls k3moe_route + k3moe_forward.
    Allocation is torch's; every computation is the library's."""

    def __init__(self, cfg: K3MoEConfig, T_max: int, device="cuda"):
        import torch
        self.cfg = cfg
        self.device = torch.device(device)
        self.T_max = T_max
        self.table = torch.empty(k3moe_packed_bytes(cfg), dtype=torch.uint8, device=self.device)
        self.ws_bytes = k3moe_workspace_bytes(cfg, T_max)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.w_router = None
        self.bias = None
        self.sh_w1 = self.sh_w3 = self.sh_w2 = None
        E, k = cfg.n_experts, cfg.top_k
        self.idx = torch.empty((T_max, k), dtype=torch.int32, device=self.device)
        self.weight = torch.empty((T_max, k), dtype=torch.float32, device=self.device)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=self.device)
        self.perm = torch.empty(T_max * k, dtype=torch.int32, device=self.device)

    def pack_experts(self, expert_lo, n, w1_packed, w1_scale, w3_packed, w3_scale, w2_packed,
                     w2_scale, stream=None):
        k3moe_pack_mxfp4(self.cfg, expert_lo, n, w1_packed, w1_scale, w3_packed, w3_scale,
                         w2_packed, w2_scale, self.table, ws=self.ws, stream=stream)

    def route(self, x, stream=None):
        T = x.shape[0]
        k3moe_route(self.cfg, T, x, self.w_router, self.bias, self.idx, self.weight, self.offsets,
                    self.perm, self.ws, self.ws_bytes, stream)

    def scores(self, x, stream=None):
        """(sc, ch) [T][E] f32 device tensors: the router scores k3moe_route selects from."""
        import torch
        T = x.shape[0]
        sc = torch.empty((T, self.cfg.n_experts), dtype=torch.float32, device=self.device)
        ch = torch.empty_like(sc)
        k3moe_router_scores(self.cfg, T, x, self.w_router, self.bias, sc, ch, self.ws, self.ws_bytes,
                            stream)
        return sc, ch

    def forward(self, x, out, stream=None, routing=None):
        T = x.shape[0]
        idx, weight, offsets, perm = routing or (self.idx, self.weight, self.offsets, self.perm)
        k3moe_forward(self.cfg, T, x, idx, weight, offsets, perm, self.table, self.sh_w1,
                      self.sh_w3, self.sh_w2, out, self.ws, self.ws_bytes, stream=stream)

    def __call__(self, x, out, stream=None):
        self.route(x, stream)
        self.forward(x, out, stream)
        return out

    def capture(self, x, out):
        """Record route + forward on the fixed buffers x [T][d] bf16 and out [T][d] f32 as
        a CUDA graph and return the torch.cuda.CUDAGraph (see _capture)."""
        return _capture(self, x, out)


class MoEBlock:
    """Holds one full-width block's device tensors (the routed experts' packed table,
    the full-width router, the down and up projections, the norm gain and the fused
    shared experts) and a workspace, and calls k3moe_full_forward.  Allocation is
    torch's; every computation is the library's."""

    def __init__(self, cfg: K3MoEConfig, fd: K3MoEFullDims, T_max: int, device="cuda"):
        import torch
        self.cfg, self.fd = cfg, fd
        self.device = torch.device(device)
        self.T_max = T_max
        self.table = torch.empty(k3moe_packed_bytes(cfg), dtype=torch.uint8, device=self.device)
        self.ws_bytes = k3moe_full_workspace_bytes(cfg, fd, T_max)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.w_router = self.bias = self.w_down = self.w_up = self.gain = None
        self.sh_w1 = self.sh_w3 = self.sh_w2 = None
        E, k = cfg.n_experts, cfg.top_k
        self.idx = torch.empty((T_max, k), dtype=torch.int32, device=self.device)
        self.weight = torch.empty((T_max, k), dtype=torch.float32, device=self.device)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=self.device)
        self.perm = torch.empty(T_max * k, dtype=torch.int32, device=self.device)

    def pack_experts(self, expert_lo, n, w1_packed, w1_scale, w3_packed, w3_scale, w2_packed,
                     w2_scale, stream=None):
        k3moe_pack_mxfp4(self.cfg, expert_lo, n, w1_packed, w1_scale, w3_packed, w3_scale,
                         w2_packed, w2_scale, self.table, ws=self.ws, stream=stream)

    def forward(self, h, out, stream=None):
        T = h.shape[0]
        k3moe_full_forward(self.cfg, self.fd, T, h, self.w_router, self.bias, self.w_down,
                           self.table, self.gain, self.w_up, self.sh_w1, self.sh_w3, self.sh_w2,
                           self.idx, self.weight, self.offsets, self.perm, out, self.ws,
                           self.ws_bytes, stream=stream)
        return out

    __call__ = forward

    def capture(self, h, out):
        """k3moe_full_forward on the fixed buffers h [T][H] and out [T][H] as a CUDA graph
        (see _capture)."""
        return _capture(self, h, out)
