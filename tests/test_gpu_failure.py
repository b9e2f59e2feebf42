"""Failure reporting on the GPU, without a fault: every device-side wait of the library is
bounded, and one that runs out sets the status word's timeout bit and lets its kernel
return (kimi-k3-in-c README, Part II, section 9: a fault is counted, never silent).

k3moe_check_wait_timeout runs both of the library's wait routines on an mbarrier that
nothing arrives on, with a short limit (1e6 cycles, about half a millisecond): the waits
give up, k3moe_device_status reports K3MOE_ETIMEOUT with the timeout bit, and a normal
layer call on the same context afterwards is clean and correct."""
import numpy as np
import pytest

import k3moe_inputs as ki
import oracle
from gpu_util import assert_out_close, ocfg, oracle_experts

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def k3():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_expert_k3moe_gb300 import build as kbuild
    kbuild.build()
    import sparse_moe_expert_k3moe_gb300 as k3
    return k3


def test_bounded_wait_gives_up_and_reports(k3):
    from k3moe_inputs.device import build_layer
    w = ki.WORKLOADS["tiny"]
    layer = build_layer(w)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0
    k3.k3moe_check_wait_timeout(layer.ws, 1_000_000)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 7 and code & k3.DEV_TIMEOUT              # K3MOE_ETIMEOUT
    # the status word was cleared by the read, and the context is still usable
    x = ki.make_x(w)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    out = torch.empty((w.T, w.d), dtype=torch.float32, device="cuda")
    layer(xd, out)
    rc, code = k3.k3moe_device_status(layer.ws)
    assert rc == 0 and code == 0
    ref = oracle.forward(ocfg(w), x, layer.idx.cpu().numpy(), layer.weight.cpu().numpy(),
                         oracle_experts(w, range(w.E)), ki.make_shared(w))
    assert_out_close(out.cpu().numpy(), ref, "after a timed-out wait")
