"""Builds libk3moe.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

Variants (the environment variable K3MOE_BUILD_VARIANT picks the one the package loads):
  release   libk3moe.so: the product;
  debug     libk3moe_debug.so: -DK3MOE_DEBUG, device-side index checks that set the
            K3MOE_DEV_BOUNDS status bit and skip the access;
  sanitize  libk3moe_asan.so: host code under AddressSanitizer and UndefinedBehaviorSanitizer
            (load it with the ASan runtime preloaded).

Usage: python -m sparse_moe_expert_k3moe_gb300.build [--force] [--variant debug|sanitize]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-Wall",
                     "--diag-suppress", "177", "-I", os.path.join(HERE, "..", "include")]
_SAN = "-fsanitize=address,-fsanitize=undefined,-fno-sanitize-recover=all,-fno-omit-frame-pointer"
# variant: (library, build folder, extra compile flags, extra link flags)
VARIANTS = {
    "release": ("libk3moe.so", "_build", [], []),
    "debug": ("libk3moe_debug.so", "_build_debug", ["-DK3MOE_DEBUG"], []),
    "sanitize": ("libk3moe_asan.so", "_build_asan", ["-Xcompiler", _SAN], ["-Xcompiler", _SAN]),
}


def variant() -> str:
    v = os.environ.get("K3MOE_BUILD_VARIANT", "release") or "release"
    if v not in VARIANTS:
        raise ValueError(f"K3MOE_BUILD_VARIANT={v!r}: one of {sorted(VARIANTS)}")
    return v


def lib_path(v: str | None = None) -> str:
    return os.path.join(HERE, VARIANTS[v or variant()][0])


LIB = lib_path("release")


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        [os.path.join(HERE, "..", "include", "k3moe.h"), os.path.abspath(__file__)]


def up_to_date(v: str | None = None) -> bool:
    lib = lib_path(v)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, v: str | None = None) -> str:
    """Builds one variant (default: the one K3MOE_BUILD_VARIANT names) and returns its path."""
    v = v or variant()
    lib_name, build_dir, cflags, lflags = VARIANTS[v]
    lib = lib_path(v)
    if not force and up_to_date(v):
        return lib
    build_dir = os.path.join(HERE, build_dir)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc] + NVCC_FLAGS + cflags + ["-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + lflags + ["-shared", "-cudart", "static", "-o", tmp] + objs + \
        ["-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    var = sys.argv[sys.argv.index("--variant") + 1] if "--variant" in sys.argv else None
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, v=var))
