"""Build libmoe_swiglu_nvfp4.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "moe_nvfp4.cu"), os.path.join(PKG, "csrc", "moe_l1_gemm.cu")]
HEADERS = [os.path.join(PKG, "csrc", "nvfp4_device.cuh")]
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "libmoe_swiglu_nvfp4.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = SOURCES + HEADERS + [os.path.join(INCLUDE, "moe_nvfp4.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles every source to an object in parallel, then links the shared
    library (one -gencode: sm_103a)."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
             "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]
    if verbose:
        flags.append("-Xptxas=-v")
    with tempfile.TemporaryDirectory(dir=OUT_DIR) as tmpdir:
        objs, procs = [], []
        for src in SOURCES:
            obj = os.path.join(tmpdir, os.path.basename(src) + ".o")
            objs.append(obj)
            procs.append(subprocess.Popen([nvcc(), *flags, "-c", "-o", obj, src]))
        codes = [p.wait() for p in procs]
        if any(codes):
            raise subprocess.CalledProcessError(max(codes), "nvcc")
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
