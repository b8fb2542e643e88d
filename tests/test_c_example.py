"""The C ABI from a plain C program (tests/c_example/quantize_from_c.c),
compiled with gcc against include/moe_nvfp4.h and linked with the library
and the CUDA runtime: host-side argument errors without a GPU, and one
quantize-only call on the GPU compared with the oracle."""
import glob
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SOURCE = os.path.join(ROOT, "tests", "c_example", "quantize_from_c.c")


def _cudart_dir():
    for d in [os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib")] + \
            sorted(glob.glob(os.path.join(CUDA, "targets", "*", "lib"))):
        if glob.glob(os.path.join(d, "libcudart.so*")):
            return d
    return None


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    gcc = shutil.which("gcc")
    cudart = _cudart_dir()
    if gcc is None or cudart is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA runtime is missing")
    from moe_swiglu_epilogue_gb300 import build, library_path
    build.build()
    lib = library_path()
    out = str(tmp_path_factory.mktemp("c_example") / "quantize_from_c")
    subprocess.run([gcc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                    SOURCE, "-o", out,
                    "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib), "-L", cudart, "-lcudart",
                    "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + cudart], check=True)
    return out


def test_c_program_gets_the_documented_error_codes(exe):
    out = subprocess.run([exe], capture_output=True, text=True, check=True, timeout=60).stdout.splitlines()
    # width not a multiple of 16, negative rows, null input, bad clamp, rows == 0, ABI version
    assert [int(v) for v in out[0].split()] == [-2, -4, -1, -5, 0, 6]
    assert "16" in out[1]                                 # the message names the width rule


@pytest.mark.gpu
def test_c_program_quantizes_like_the_oracle(exe, tmp_path):
    import oracle
    from moe_swiglu_epilogue_gb300 import workloads as W
    oracle.build()
    w = W.quantize_normal(rows=64, K=512, seed=9)
    src, dst = tmp_path / "x.bin", tmp_path / "out.bin"
    np.ascontiguousarray(w.data, dtype=np.uint16).tofile(src)
    subprocess.run([exe, "run", str(src), str(dst), str(w.rows), str(w.width)], check=True, timeout=120)
    got = np.fromfile(dst, dtype=np.uint8)
    rp, rs = oracle.quantize_nvfp4(w.data)
    assert np.array_equal(got[:rp.size], rp.ravel()) and np.array_equal(got[rp.size:], rs.ravel())
