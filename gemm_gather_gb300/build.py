"""Build the C-ABI library from csrc/ with nvcc for sm_103a, in two builds:

* libgemm_gather.so, the release build;
* libgemm_gather_checked.so, the checked build: the same calls, with the
  gather kernels' device-side bounds checks compiled in (GG_CHECKED=1; only
  the translation units that read the macro are compiled twice).

Every translation unit is compiled in parallel, then each library is linked
against the shared CUDA runtime.  Output: gemm_gather_gb300/_build/.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgemm_gather.so")
LIB_CHECKED = os.path.join(BUILD, "libgemm_gather_checked.so")
SOURCES = ["gg_api.cu", "ag_kernels.cu", "mag_kernel.cu", "tensor_maps.cu", "fill_kernel.cu"]
CHECKED_SOURCES = ["gg_api.cu", "ag_kernels.cu"]  # the units that read GG_CHECKED
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "gemm_gather.h"))
    files.append(__file__)
    return max(os.path.getmtime(f) for f in files if os.path.exists(f))


def _fresh(path: str) -> bool:
    return os.path.exists(path) and os.path.getmtime(path) >= _deps_mtime()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile both builds (if anything changed); return the release library's path."""
    if not force and _fresh(LIB) and _fresh(LIB_CHECKED):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(job: tuple[str, bool]) -> str:
        src, checked = job
        obj = os.path.join(BUILD, src.replace(".cu", "_checked.o" if checked else ".o"))
        defs = ["-DGG_CHECKED=1"] if checked else []
        cmd = [nvcc, *ARCH, *FLAGS, *defs, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    jobs = [(src, False) for src in SOURCES] + [(src, True) for src in CHECKED_SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = dict(zip(jobs, ex.map(compile_one, jobs)))

    def link(path: str, checked: bool) -> None:
        units = [objs[(src, checked and src in CHECKED_SOURCES)] for src in SOURCES]
        tmp = path + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *units]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"linking {os.path.basename(path)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)

    link(LIB_CHECKED, True)
    link(LIB, False)  # last: its time stamp marks the whole build as fresh
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
