"""The C ABI library: it loads, exports every entry point include/k3moe.h declares,
and its host-side validation rejects bad input before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from sparse_moe_expert_k3moe_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "k3moe.h")


@pytest.fixture(scope="module")
def k3():
    kbuild.build()
    import sparse_moe_expert_k3moe_gb300 as k3
    k3.lib()
    return k3


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(k3moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("k3moe_route", "k3moe_forward", "k3moe_pack_mxfp4", "k3moe_workspace_bytes",
                 "k3moe_device_status", "k3moe_packed_bytes"):
        assert must in names


def test_library_exports_every_declared_symbol(k3):
    raw = ctypes.CDLL(k3.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def k3_cfg(k3, **over):
    kw = dict(d=3584, f=3072, n_experts=896, top_k=16, n_shared=2)
    kw.update(over)
    return k3.k3moe_config(**kw)


def test_config_validation(k3):
    assert k3.k3moe_validate_config(k3_cfg(k3)) == 0
    assert k3.k3moe_validate_config(k3_cfg(k3, d=256, f=128, n_experts=32, top_k=4, n_shared=1)) == 0
    bad = [dict(d=0), dict(f=0), dict(n_experts=0), dict(top_k=0), dict(group=16),
           dict(situ_b1=0.0), dict(situ_b2=-1.0), dict(situ_b1=float("inf")), dict(renorm=2),
           dict(routed_scale=float("nan")), dict(top_k=900), dict(n_shared=-1)]
    for b in bad:
        assert k3.k3moe_validate_config(k3_cfg(k3, **b)) == 1, b
    for b in (dict(d=3600), dict(f=100), dict(n_experts=2048), dict(top_k=17, n_experts=64),
              dict(n_shared=9)):
        assert k3.k3moe_validate_config(k3_cfg(k3, **b)) == 2, b


def test_sizes(k3):
    cfg = k3_cfg(k3)
    assert k3.k3moe_packed_bytes(cfg) == 896 * (2 * 17547264 + 1024)
    tiny = k3_cfg(k3, d=256, f=128, n_experts=32, top_k=4, n_shared=1)
    assert k3.k3moe_packed_bytes(tiny) == 32 * (2 * 52224 + 1024)
    w1 = k3.k3moe_workspace_bytes(cfg, 1)
    w64 = k3.k3moe_workspace_bytes(cfg, 64)
    assert 256 < w1 < w64
    assert k3.k3moe_workspace_bytes(cfg, 0) >= 256
    with pytest.raises(k3.K3MoEError):
        k3.k3moe_workspace_bytes(cfg, -1)
    assert k3.k3moe_packed_bytes(k3_cfg(k3, d=0)) == 0
    # the K3 shape's workspace, pinned so that it cannot grow unnoticed: under 1 MiB for one
    # token; the last mat-vec T (447) is the peak below the tensor-core path; T = 4096
    MiB = 1 << 20
    assert w1 < 1 * MiB
    assert k3.k3moe_workspace_bytes(cfg, 447) <= 211 * MiB
    assert k3.k3moe_workspace_bytes(cfg, 448) == k3.k3moe_workspace_bytes(cfg, 447)
    assert k3.k3moe_workspace_bytes(cfg, 4096) <= 985 * MiB


def test_prefill_gemm_switch(k3):
    """The process-wide choice of the prefill gate/up kernel: 0 (default), 1 (f16 on
    dequantised weights), 2 (block-scaled); anything else is refused and changes nothing."""
    assert k3.k3moe_get_prefill_gemm() == 0
    try:
        for v in (2, 1, 0):
            k3.k3moe_set_prefill_gemm(v)
            assert k3.k3moe_get_prefill_gemm() == v
        k3.k3moe_set_prefill_gemm(2)
        for bad in (-1, 3):
            with pytest.raises(k3.K3MoEError):
                k3.k3moe_set_prefill_gemm(bad)
            assert k3.k3moe_get_prefill_gemm() == 2
    finally:
        k3.k3moe_set_prefill_gemm(0)


def test_host_validation_rejects_before_launch(k3):
    L = k3.lib()
    cfg = k3_cfg(k3)
    vp = ctypes.c_void_p
    A = 0x10000000  # fake, 256-aligned addresses: never dereferenced on the host
    big = 1 << 40
    # no workspace
    rc = L.k3moe_route(ctypes.byref(cfg), 4, vp(A), vp(A), None, vp(A), vp(A), vp(A), vp(A),
                       None, 0, None)
    assert rc == 4
    # misaligned activations
    rc = L.k3moe_route(ctypes.byref(cfg), 4, vp(A + 2), vp(A), None, vp(A), vp(A), vp(A), vp(A),
                       vp(A), big, None)
    assert rc == 3
    # workspace too small
    rc = L.k3moe_route(ctypes.byref(cfg), 4, vp(A), vp(A), None, vp(A), vp(A), vp(A), vp(A),
                       vp(A), 1024, None)
    assert rc == 4
    # T out of range, missing outputs, bad config
    assert L.k3moe_route(ctypes.byref(cfg), -1, vp(A), vp(A), None, vp(A), vp(A), vp(A), vp(A),
                         vp(A), big, None) == 2
    assert L.k3moe_route(ctypes.byref(cfg), 4, vp(A), vp(A), None, None, vp(A), vp(A), vp(A),
                         vp(A), big, None) == 1
    bad = k3_cfg(k3, top_k=0)
    assert L.k3moe_route(ctypes.byref(bad), 4, vp(A), vp(A), None, vp(A), vp(A), vp(A), vp(A),
                         vp(A), big, None) == 1
    # forward: table too small, missing shared experts, misaligned table
    tb = k3.k3moe_packed_bytes(cfg)
    args = lambda table, tbytes, sh: (ctypes.byref(cfg), 4, vp(A), vp(A), vp(A), vp(A), vp(A),
                                      vp(table), tbytes, sh, sh, sh, vp(A), vp(A), big, None)
    assert L.k3moe_forward(*args(A, tb - 1, vp(A))) == 2
    assert L.k3moe_forward(*args(A, tb, None)) == 1
    assert L.k3moe_forward(*args(A + 16, tb, vp(A))) == 3
    # T = 0 is a no-op for forward
    assert L.k3moe_forward(ctypes.byref(cfg), 0, None, None, None, None, None, None, 0, None,
                           None, None, None, None, 0, None) == 0
    # pack: range outside the table, misaligned source
    assert L.k3moe_pack_mxfp4(ctypes.byref(cfg), 890, 10, *([vp(A)] * 6), vp(A), big, None,
                              None) == 2
    assert L.k3moe_pack_mxfp4(ctypes.byref(cfg), 0, 1, vp(A + 8), *([vp(A)] * 5), vp(A), big,
                              None, None) == 3
    assert k3.k3moe_strerror(4).startswith("workspace")
    # the bounded-wait check: no workspace, a limit outside 1 .. 4e9 cycles
    assert L.k3moe_check_wait_timeout(None, 1000, None) == 4
    assert L.k3moe_check_wait_timeout(vp(A + 8), 1000, None) == 4
    assert L.k3moe_check_wait_timeout(vp(A), 0, None) == 2
    assert L.k3moe_check_wait_timeout(vp(A), 4000000001, None) == 2
    # the index-check hook: no workspace, an empty range; the build flags
    assert L.k3moe_check_bounds(None, 0, 4, None) == 4
    assert L.k3moe_check_bounds(vp(A + 8), 0, 4, None) == 4
    assert L.k3moe_check_bounds(vp(A), 0, 0, None) == 2
    want = k3.BUILD_DEBUG if k3.library_path().endswith("libk3moe_debug.so") else 0
    assert k3.k3moe_build_flags() == want
    # no-allocation forward: T beyond the largest any call accepts, a misaligned status word
    nargs = lambda T, st: (ctypes.byref(cfg), T, vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), tb,
                           vp(A), vp(A), vp(A), vp(A), st, None)
    assert L.k3moe_forward_noalloc(*nargs((1 << 20) + 1, None)) == 2
    assert L.k3moe_forward_noalloc(*nargs(0, vp(A + 2))) == 3


def test_full_block_validation_and_sizes(k3):
    cfg = k3_cfg(k3)
    fd = k3.k3moe_full_dims(7168)
    w1 = k3.k3moe_full_workspace_bytes(cfg, fd, 1)
    w4096 = k3.k3moe_full_workspace_bytes(cfg, fd, 4096)
    assert k3.k3moe_workspace_bytes(cfg, 1) + (32 << 20) < w1 < w4096
    # the block's own buffers at T = 4096: z, a, y at width d; gate, up, act at S*f
    assert w4096 >= 4096 * (3584 * (2 + 4 + 2) + 2 * 3072 * (4 + 4 + 2)) + (32 << 20)
    for bad, code in ((dict(hidden=0), 1), (dict(latent_norm=2), 1), (dict(rms_eps=0.0), 1),
                      (dict(rms_eps=float("nan")), 1), (dict(hidden=7000), 2), (dict(hidden=16384), 2)):
        kw = dict(hidden=7168, latent_norm=1, rms_eps=1e-5)
        kw.update(bad)
        with pytest.raises(k3.K3MoEError) as ei:
            k3.k3moe_full_workspace_bytes(cfg, k3.k3moe_full_dims(**kw), 4)
        assert ei.value.status == code, bad
    L = k3.lib()
    vp = ctypes.c_void_p
    A = 0x10000000  # fake, 256-aligned addresses: never dereferenced on the host
    big = 1 << 40

    def call(h=A, gain=A, ws=A, ws_bytes=big, fdim=fd):
        return L.k3moe_full_forward(ctypes.byref(cfg), ctypes.byref(fdim), 4, vp(h), vp(A), None, vp(A),
                                    vp(A), big, vp(gain) if gain else None, vp(A), vp(A), vp(A), vp(A),
                                    vp(A), vp(A), vp(A), vp(A), vp(A), vp(ws) if ws else None,
                                    ws_bytes, None)
    assert call(h=A + 2) == 3                         # misaligned tokens
    assert call(gain=0) == 1                          # the norm needs its gain
    assert call(ws=0) == 4                            # no workspace
    assert call(ws_bytes=1024) == 4                   # workspace too small
    assert call(fdim=k3.k3moe_full_dims(7168, rms_eps=-1.0)) == 1


@pytest.mark.parametrize("kw", [
    dict(),                                                          # K3: mat-vec path below T = 448
    dict(d=256, f=128, n_experts=32, top_k=4, n_shared=1),
    dict(d=256, f=8192, n_experts=8, top_k=1, n_shared=8),          # big split partials at T = 1
])
def test_workspace_covers_every_smaller_t(k3, kw):
    """k3moe_workspace_bytes(T_max) serves every call with T <= T_max, so it never
    shrinks as T_max grows, across the switch from the mat-vec to the tensor-core path
    (where one call's own layout does shrink)."""
    cfg = k3_cfg(k3, **kw)
    fd = k3.k3moe_full_dims(512)
    for size in (lambda T: k3.k3moe_workspace_bytes(cfg, T),
                 lambda T: k3.k3moe_full_workspace_bytes(cfg, fd, T)):
        sizes = [size(T) for T in range(0, 600)]
        assert all(b >= a for a, b in zip(sizes, sizes[1:]))
