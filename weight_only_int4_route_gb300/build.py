"""Build libmoe.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ is compiled to an object in parallel, then the objects are
linked into weight_only_int4_route_gb300/libmoe.so against the shared CUDA runtime
(the same libcudart soname PyTorch loads, so both share one runtime instance).

build(checked=True) compiles the same sources with MOE_CHECKED=1 into libmoe_checked.so:
the kernels then bounds-check the indices they read from device memory and report
violations through moe_check_status instead of reading or writing out of range.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe.so")
BUILD_CHECKED = os.path.join(ROOT, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libmoe_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def cuda_lib_dir() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        p = os.path.join(home, sub)
        if os.path.isdir(p):
            return p
    return os.path.join(home, "lib64")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in sources() + headers() + [__file__])


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), "-c", src, "-o", obj, "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "--expt-relaxed-constexpr", "-Xptxas=-warn-spills", *extra]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          checked: bool = False) -> str:
    """Compile every CUDA source and link libmoe.so (libmoe_checked.so with checked=True);
    returns the library path."""
    lib, build_dir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    extra = list(extra or []) + (["-DMOE_CHECKED=1"] if checked else [])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(sources()), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp, *objs, *ARCH, "-cudart", "shared",
           "-Xlinker", "-rpath," + cuda_lib_dir()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib


def build_all(force: bool = False, verbose: bool = False) -> None:
    """Both libraries, the plain and the checked one, compiled side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        list(ex.map(lambda c: build(force=force, verbose=verbose, checked=c), (False, True)))


if __name__ == "__main__":
    build_all(force="--force" in sys.argv, verbose=True)
