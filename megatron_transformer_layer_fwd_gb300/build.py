"""Builds libmgb.so in-tree for sm_103a (GB300) with nvcc.

Each .cu under csrc/ compiles to an object in parallel, then one shared
library is linked next to this file. The CUDA runtime is linked statically;
the CUDA driver's tensor-map encoder is looked up at run time, so the library
needs no libcuda at link time and loads on machines without a GPU.

    python -m megatron_transformer_layer_fwd_gb300.build
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmgb.so")
# the checking build: kernels compiled with -DMGB_CHECK=1 (device-side
# consistency checks that record MGB_ERR_DEVICE_CHECK); loaded by MGB_LIB=check
BUILD_CHECK = os.path.join(HERE, "_build_check")
LIB_CHECK = os.path.join(HERE, "libmgb_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xcompiler", "-Wall", "-Xcompiler", "-Wno-unused-function"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp(paths) -> float:
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, extra: list[str], bdir: str = BUILD) -> str:
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          check: bool = False) -> str:
    """Compile csrc/*.cu and link libmgb.so (check: libmgb_check.so with the
    device-side checks); skipped when it is up to date."""
    extra = list(extra or [])
    lib, bdir = (LIB_CHECK, BUILD_CHECK) if check else (LIB, BUILD)
    if check:
        extra.append("-DMGB_CHECK=1")
    srcs = sources()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "mgb.h"))
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _stamp(srcs + headers):
        return lib
    os.makedirs(bdir, exist_ok=True)
    if verbose:
        extra.append("-Xptxas=-v")
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, bdir), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, check="--check" in sys.argv))
