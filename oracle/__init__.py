"""Oracle for the all-gather over a symmetric heap and the fused matmul + all-gather.

TEST INFRASTRUCTURE ONLY.  ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module; the product path (``gemm_gather_gb300``) never does, and this module
imports nothing from it.  The arithmetic lives in ``gg_oracle.c`` (plain C,
float64 for the matmul); this file only builds it with gcc and marshals numpy
arrays through ctypes.

The heap is modelled as a flat ``uint8`` numpy array of ``H`` partitions of
``part_bytes`` each (partition ``h`` is logical rank ``h``'s symmetric heap,
iris #594 "Local validation": independent allocations stand for ranks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gg_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgg_oracle.so")
_CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-Wall"]

_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1  # 16-bit float formats understood by decode16/encode16


def build(out_path: str = _LIB_PATH, defines: tuple[str, ...] = ()) -> str:
    """Compile gg_oracle.c with gcc into ``out_path`` (skipped when up to date)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    if (not defines and os.path.exists(out_path)
            and os.path.getmtime(out_path) >= os.path.getmtime(_SRC)):
        return out_path
    cmd = ["gcc", *_CFLAGS, *[f"-D{d}" for d in defines], "-o", out_path, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_group_index.argtypes = [i32, i32, i32, i32]
    lib.oracle_group_index.restype = i32
    lib.oracle_gather_contribution.argtypes = [vp, i64, i32, vp, i64, i64, i64,
                                               i64, i64, i32, i32, i32, i32, i32]
    lib.oracle_gather_contribution.restype = i32
    lib.oracle_all_gather.argtypes = [vp, vp, i64, i32, i64, i64, i64, i64, i64,
                                      i64, i32, i32, i32, i32]
    lib.oracle_all_gather.restype = i32
    lib.oracle_all_to_all.argtypes = [vp, vp, i64, i32, i64, i64, i64, i64, i64,
                                      i64, i32, i32, i32, i32]
    lib.oracle_all_to_all.restype = i32
    lib.oracle_decode16.argtypes = [ctypes.c_uint16, i32]
    lib.oracle_decode16.restype = ctypes.c_double
    lib.oracle_encode16.argtypes = [ctypes.c_double, i32]
    lib.oracle_encode16.restype = ctypes.c_uint16
    lib.oracle_matmul_f64.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64,
                                      i32, vp, i64]
    lib.oracle_matmul_f64.restype = i32
    lib.oracle_round16.argtypes = [vp, i64, vp, i64, i64, i64, i32]
    lib.oracle_round16.restype = None
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_set_threads.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first when needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


class Oracle:
    """numpy front end of one oracle build (the default one, or a test variant)."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    # -- group resolution (iris #591, Description §1) ------------------------
    def group_index(self, h: int, rank_start: int, rank_stride: int, world_size: int) -> int:
        return int(self.lib.oracle_group_index(h, rank_start, rank_stride, world_size))

    # -- all-gather (iris PR #626 "Summary"; iris #594 "Multi-GPU CI") ------
    def gather_contribution(self, heap: np.ndarray, part_bytes: int, src: np.ndarray,
                            out_off: int, ld_out: int, M: int, N: int,
                            group: tuple[int, int, int], src_rank: int) -> None:
        """Rank ``src_rank`` writes its block ``src`` (M x N, any dtype, row pitch
        from its strides) into its row block of every member's output, in place."""
        assert heap.dtype == np.uint8 and heap.flags.c_contiguous
        H = heap.size // part_bytes
        esize = src.dtype.itemsize
        ld_in = src.strides[0] // esize if src.ndim == 2 else N
        rc = self.lib.oracle_gather_contribution(
            heap.ctypes.data, part_bytes, H, src.ctypes.data, ld_in, out_off, ld_out,
            M, N, esize, *group, src_rank)
        if rc:
            raise ValueError("oracle_gather_contribution rejected its arguments")

    def all_gather(self, heap: np.ndarray, part_bytes: int, in_off: int, ld_in: int,
                   out_off: int, ld_out: int, M: int, N: int, esize: int,
                   group: tuple[int, int, int]) -> None:
        """Every member's block at ``in_off`` is gathered into every member's
        output at ``out_off``; updates ``heap`` in place."""
        assert heap.dtype == np.uint8 and heap.flags.c_contiguous
        H = heap.size // part_bytes
        snapshot = heap.copy()
        rc = self.lib.oracle_all_gather(heap.ctypes.data, snapshot.ctypes.data,
                                        part_bytes, H, in_off, ld_in, out_off, ld_out,
                                        M, N, esize, *group)
        if rc:
            raise ValueError("oracle_all_gather rejected its arguments")

    # -- all-to-all (iris #594 "Compiler inspection and grouping") ----------
    def all_to_all(self, heap: np.ndarray, part_bytes: int, in_off: int, ld_in: int,
                   out_off: int, ld_out: int, M: int, N: int, esize: int,
                   group: tuple[int, int, int]) -> None:
        """Member d's output row block i = member i's input row block d (each
        input is W*M x N); updates ``heap`` in place."""
        assert heap.dtype == np.uint8 and heap.flags.c_contiguous
        H = heap.size // part_bytes
        snapshot = heap.copy()
        rc = self.lib.oracle_all_to_all(heap.ctypes.data, snapshot.ctypes.data, part_bytes, H,
                                        in_off, ld_in, out_off, ld_out, M, N, esize, *group)
        if rc:
            raise ValueError("oracle_all_to_all rejected its arguments")

    # -- 16-bit formats -------------------------------------------------------
    def decode16(self, bits: int, fmt: int) -> float:
        return float(self.lib.oracle_decode16(bits, fmt))

    def encode16(self, x: float, fmt: int) -> int:
        return int(self.lib.oracle_encode16(x, fmt))

    # -- fused matmul (iris PR #626 "Summary", "Benchmark") ------------------
    def matmul_f64(self, A: np.ndarray, B: np.ndarray, fmt: int,
                   rows: np.ndarray | None = None) -> np.ndarray:
        """float64 A @ B of 16-bit operands given as uint16 bit patterns
        (A: M x K, B: K x N, any row pitch).  ``rows`` restricts the result to
        those rows of A (returned in that order)."""
        assert A.dtype == np.uint16 and B.dtype == np.uint16
        M, K = A.shape
        K2, N = B.shape
        assert K == K2
        # an empty operand (K == 0) is never read; numpy gives it no usable strides
        assert A.size == 0 or A.strides[1] == 2
        assert B.size == 0 or B.strides[1] == 2
        lda = A.strides[0] // 2 if A.size else K
        ldb = B.strides[0] // 2 if B.size else N
        R = M if rows is None else len(rows)
        C = np.empty((R, N), dtype=np.float64)
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        rc = self.lib.oracle_matmul_f64(A.ctypes.data, lda, B.ctypes.data, ldb, C.ctypes.data, N,
                                        M, N, K, fmt,
                                        None if rows_arr is None else rows_arr.ctypes.data, R)
        if rc:
            raise MemoryError("oracle_matmul_f64: out of memory")
        return C

    def round16(self, C: np.ndarray, fmt: int) -> np.ndarray:
        """Round a float64 block to 16-bit bit patterns (nearest even)."""
        C = np.ascontiguousarray(C, dtype=np.float64)
        M, N = C.shape
        out = np.empty((M, N), dtype=np.uint16)
        self.lib.oracle_round16(C.ctypes.data, N, out.ctypes.data, N, M, N, fmt)
        return out

    def matmul_all_gather(self, heap: np.ndarray, part_bytes: int, a_off: int, lda: int,
                          B: np.ndarray, out_off: int, ld_out: int, M: int, N: int, K: int,
                          fmt: int, group: tuple[int, int, int]) -> dict[int, np.ndarray]:
        """Fused form: each member r computes C_r = A_r @ B (A_r: M x K at
        ``a_off`` in its partition, row pitch lda), rounds it to 16 bits and
        gathers it into every member's output.  Updates ``heap`` in place and
        returns the float64 products {group index: C_r} for tolerance checks."""
        start, stride, W = group
        snapshot = heap.copy()
        products = {}
        for i in range(W):
            r = start + i * stride
            base = r * part_bytes + a_off
            a_rows = snapshot[base: base + ((M - 1) * lda + K) * 2].view(np.uint16)
            A = np.lib.stride_tricks.as_strided(a_rows, shape=(M, K), strides=(lda * 2, 2))
            C = self.matmul_f64(A, B, fmt)
            products[i] = C
            self.gather_contribution(heap, part_bytes, self.round16(C, fmt), out_off,
                                     ld_out, M, N, group, r)
        return products

    # -- threads ---------------------------------------------------------------
    def set_threads(self, n: int) -> None:
        self.lib.oracle_set_threads(n)

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


def default() -> Oracle:
    return Oracle()
