"""Build libep.so (the CUDA dispatch / combine library) in-tree with nvcc for sm_103a.

Each .cu file compiles in its own nvcc process (in parallel), then one shared link.  The
library links the shared CUDA runtime so it shares the process's runtime with PyTorch.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libep.so")
SOURCES = ("ep_api.cu", "ep_route.cu", "ep_scatter.cu", "ep_combine.cu", "ep_noalloc.cu",
           "ep_fp8wire.cu", "ep_grouped.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libep.so")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
           [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          defines=(), lib_path: str = LIB, build_dir: str = BUILD_DIR) -> str:
    """Compile libep.so; `defines` (e.g. ["EP_COMBINE_STAGES=4"]) and a separate lib_path /
    build_dir let a caller build tuning variants side by side."""
    if not force and lib_path == LIB and not defines and not _stale():
        return LIB
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
             "-I", CSRC] + [f"-D{d}" for d in defines]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", *ARCH, "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))
