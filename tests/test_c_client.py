"""The C ABI used from plain C: tests/c_abi_client.c includes
include/gemm_gather.h as C11, owns its device memory (cudaMalloc), and runs a
group all-gather and a fused matmul + all-gather through libgemm_gather.so,
checking the results on the host (bit patterns for the gather, exact integer
products for the fused call).  It links against either build, the release
libgemm_gather.so or the checked libgemm_gather_checked.so (same calls, with
device-side bounds checks; a check firing on these valid calls would leave a
status word non-zero and fail the client).  Compiling and linking it needs no
GPU; running it does."""
import os
import subprocess

import pytest

from gemm_gather_gb300 import _lib

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


BUILDS = {"release": "gemm_gather", "checked": "gemm_gather_checked"}


def _build(out_dir, build: str = "release") -> str:
    exe = os.path.join(str(out_dir), f"c_abi_client_{build}")
    libdir = os.path.dirname(_lib.LIB_PATH)
    cudalib = os.path.join(CUDA, "lib64")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Werror", os.path.join(HERE, "c_abi_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, f"-l{BUILDS[build]}", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}:{cudalib}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


@pytest.mark.parametrize("build", sorted(BUILDS))
def test_c_client_compiles_against_the_header(tmp_path, build):
    assert os.path.exists(_build(tmp_path, build))


@pytest.mark.gpu
@pytest.mark.parametrize("build", sorted(BUILDS))
def test_c_client_runs(tmp_path, build):
    exe = _build(tmp_path, build)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi client ok" in r.stdout
