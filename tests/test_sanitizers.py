"""Sanitizer runs of the host code (CPU only).

The kimi-k3-in-c README (Part I, "Getting started", and Part V, "Reference") builds its
C code under AddressSanitizer and UndefinedBehaviorSanitizer in CI.  Here:

- the CPU oracle and the seeded input generator, linked with a C driver
  (``tests/sanitize/oracle_driver.c``) that calls every entry point, the edge cases
  (k = E, E = k = 1, no shared expert, T = 0) and the error paths, built with
  ``-fsanitize=address,undefined -fno-sanitize-recover=all`` and leak checking on;
- the GPU library's host code (argument validation, sizes, workspace layout, the
  C-ABI error paths), built as the ``sanitize`` variant and driven by the CPU ABI tests
  in a child process with the ASan runtime preloaded.  No GPU is touched.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _asan_runtime():
    gcc = shutil.which("gcc")
    if not gcc:
        return None
    path = subprocess.run([gcc, "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


needs_asan = pytest.mark.skipif(_asan_runtime() is None, reason="gcc with the ASan runtime is not available")


@needs_asan
def test_oracle_and_generator_under_asan_ubsan(tmp_path):
    exe = str(tmp_path / "oracle_driver")
    srcs = [os.path.join(ROOT, "tests", "sanitize", "oracle_driver.c"),
            os.path.join(ROOT, "oracle", "k3moe_oracle.c"),
            os.path.join(ROOT, "k3moe_inputs", "k3moe_gen.c")]
    cmd = ["gcc", "-O1", "-g", "-std=c99", "-fopenmp", "-ffp-contract=off", "-Wall", "-Wextra", "-Werror",
           "-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer",
           "-o", exe] + srcs + ["-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:halt_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1", OMP_NUM_THREADS="2")
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=600)
    print(r.stdout.strip())
    assert r.returncode == 0, r.stdout + r.stderr
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, r.stderr


@needs_asan
@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc is not available")
def test_library_host_code_under_asan_ubsan():
    from sparse_moe_expert_k3moe_gb300 import build as kbuild
    lib = kbuild.build(v="sanitize")
    assert os.path.exists(lib)
    env = dict(os.environ, K3MOE_BUILD_VARIANT="sanitize", LD_PRELOAD=_asan_runtime(),
               ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0:halt_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_abi.py"), "-q", "-m", "not gpu",
           "-p", "no:cacheprovider"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT, timeout=900)
    print(r.stdout.strip().splitlines()[-1] if r.stdout.strip() else "")
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, r.stderr[-4000:]
    # the child really loaded the sanitized library
    probe = [sys.executable, "-c",
             "import sparse_moe_expert_k3moe_gb300 as k3; k3.lib(); print(k3.library_path())"]
    r = subprocess.run(probe, capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("libk3moe_asan.so"), r.stdout + r.stderr
