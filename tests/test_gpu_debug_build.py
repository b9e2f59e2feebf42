"""The debug build (-DK3MOE_DEBUG): device-side index checks at the point of use.

Kernels check the indices they derive from other kernels' output (unit lists, offsets,
positions, slots) before they use them; every build keeps the guards that protect an
access, and a debug build also records a failed check as K3MOE_DEV_BOUNDS in the status
word (kimi-k3-in-c README, Part II, section 9: a fault is counted, never silent).

- the record path: k3moe_check_bounds runs one check on an index out of range; the
  debug build reports K3MOE_DEV_BOUNDS and stays usable, the release build records
  nothing;
- the debug build on the parity cases: the small layers (both forward paths, every
  shape class of the suite), shape alternation, graph replay, one workspace reused
  across both forward paths and both mat-vec schedules, and the full K3 shape at T = 1
  (the single-token schedule), each of which asserts a clean status word after every
  call -- so no check fires on valid input.
The debug library is built on the GPU machine and loaded by a child process
(K3MOE_BUILD_VARIANT=debug); the release library in this process is untouched.
"""
import os
import subprocess
import sys

import pytest

from sparse_moe_expert_k3moe_gb300 import build as kbuild

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import torch, sparse_moe_expert_k3moe_gb300 as k3
assert k3.library_path().endswith("libk3moe_debug.so"), k3.library_path()
assert k3.k3moe_build_flags() == k3.BUILD_DEBUG
cfg = k3.k3moe_config(d=256, f=128, n_experts=32, top_k=4, n_shared=1)
ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
k3.k3moe_check_bounds(ws, 2, 3)
assert k3.k3moe_device_status(ws) == (0, 0)
k3.k3moe_check_bounds(ws, 3, 3)
rc, code = k3.k3moe_device_status(ws)
assert rc == 6 and code == k3.DEV_BOUNDS, (rc, code)
k3.k3moe_check_bounds(ws, -1, 3)
rc, code = k3.k3moe_device_status(ws)
assert rc == 6 and code == k3.DEV_BOUNDS, (rc, code)
assert k3.k3moe_device_status(ws) == (0, 0)      # read and cleared
print("debug record path ok")
"""


def _debug_env():
    return dict(os.environ, K3MOE_BUILD_VARIANT="debug")


@pytest.fixture(scope="module")
def k3():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kbuild.build()
    import sparse_moe_expert_k3moe_gb300 as k3
    return k3


@pytest.fixture(scope="module")
def debug_lib(k3):
    path = kbuild.build(v="debug")
    assert os.path.exists(path)
    return path


def test_release_build_records_no_bounds(k3):
    assert k3.k3moe_build_flags() == 0
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    k3.k3moe_check_bounds(ws, 7, 3)
    assert k3.k3moe_device_status(ws) == (0, 0)


def test_debug_build_records_a_bad_index(debug_lib):
    r = subprocess.run([sys.executable, "-c", _CHILD], capture_output=True, text=True, env=_debug_env(),
                       cwd=ROOT, timeout=600)
    print(r.stdout.strip())
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


def test_debug_build_is_clean_on_the_parity_cases(debug_lib):
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-q", "-m", "gpu",
           "-p", "no:cacheprovider", "-k",
           "small_layer_parity or alternating_shapes or graph_replay or zero_tokens or injected_oracle_routing"
           " or reuse or (full_forward_parity and decode_t1)"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=_debug_env(), cwd=ROOT, timeout=1800)
    tail = r.stdout.strip().splitlines()
    print(tail[-1] if tail else "")
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-3000:]
