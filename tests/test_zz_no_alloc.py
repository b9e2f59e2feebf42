"""k3moe_forward_noalloc: the forward pass for callers that cannot allocate device
memory (plugins and serving hooks handed only inputs and outputs, fixed-budget
real-time callers); it takes no workspace, its scratch is an array inside the library.

Its output must match k3moe_forward's (same routing, same weights) within the
layer's output tolerance on two calls in a row, and a T whose scratch would not fit
must be refused before anything runs.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import k3moe_inputs as ki
from gpu_util import assert_out_close

torch = pytest.importorskip("torch")

NOALLOC_LIMIT = 32 << 20


@pytest.fixture(scope="module")
def k3():
    from sparse_moe_expert_k3moe_gb300 import build as kbuild
    kbuild.build()
    import sparse_moe_expert_k3moe_gb300 as k3
    return k3


def test_noalloc_limit_covers_decode_at_k3_shape(k3):
    cfg = k3.k3moe_config(**ki.WORKLOADS["decode_t64"].config_kwargs())
    assert k3.k3moe_workspace_bytes(cfg, 64) <= NOALLOC_LIMIT


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["micro", "decode_t1"])
def test_noalloc_matches_forward_twice(k3, name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from k3moe_inputs.device import build_layer
    w = (ki.Workload("micro", T=37, d=384, f=256, E=16, k=4, S=2, exp_lo=-7, exp_hi=-3, seed=60)
         if name == "micro" else ki.WORKLOADS[name])
    layer = build_layer(w)
    L = k3.lib()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        x = ki.make_x(w.with_(seed=w.seed + 100 * call))
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        layer.route(xd)
        ref = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
        layer.forward(xd, ref)                          # existing entry point, caller workspace
        got = torch.full((w.T, w.d), float("nan"), dtype=torch.float32, device="cuda")
        rc = L.k3moe_forward_noalloc(
            ctypes.byref(layer.cfg), w.T, xd.data_ptr(), layer.idx.data_ptr(),
            layer.weight.data_ptr(), layer.offsets.data_ptr(), layer.perm.data_ptr(),
            layer.table.data_ptr(), layer.table.numel(),
            *(t.data_ptr() for t in (layer.sh_w1, layer.sh_w3, layer.sh_w2)),
            got.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, k3.k3moe_strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_out_close(got.cpu().numpy(), ref.cpu().numpy(), f"{name} call {call}")


@pytest.mark.gpu
def test_noalloc_zero_tokens_reports_clean_status(k3):
    """No tokens: nothing is computed, and the optional status word still reports this
    call (clean), not what an earlier call left there."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg = k3.k3moe_config(**ki.WORKLOADS["tiny"].config_kwargs())
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    L = k3.lib()
    rc = L.k3moe_forward_noalloc(ctypes.byref(cfg), 0, None, None, None, None, None, None, 0,
                                 None, None, None, None, status.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.gpu
def test_noalloc_refuses_oversized_t(k3):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = ki.WORKLOADS["prefill_t4096"]
    cfg = k3.k3moe_config(**w.config_kwargs())
    assert k3.k3moe_workspace_bytes(cfg, w.T) > NOALLOC_LIMIT
    A = 1 << 30                      # aligned placeholder addresses: refused before any use
    L = k3.lib()
    rc = L.k3moe_forward_noalloc(ctypes.byref(cfg), w.T, A, A, A, A, A, A,
                                 k3.k3moe_packed_bytes(cfg), A, A, A, A, None, None)
    assert rc == 4                   # K3MOE_EWORKSPACE
