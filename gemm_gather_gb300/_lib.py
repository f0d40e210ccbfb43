"""ctypes loader of the C-ABI library (built in-tree by gemm_gather_gb300.build).

The release build, libgemm_gather.so, is loaded unless the environment sets
GEMM_GATHER_CHECKED=1, which loads the checked build,
libgemm_gather_checked.so (the same calls with device-side bounds checks in
the gather kernels; see gg_checked_build in include/gemm_gather.h).  Importing
this module fails loudly when the chosen library has not been built: there is
no fallback path of any kind.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
CHECKED = os.environ.get("GEMM_GATHER_CHECKED", "0") == "1"
LIB_PATH = os.path.join(HERE, "_build",
                        "libgemm_gather_checked.so" if CHECKED else "libgemm_gather.so")

GG_OK = 0
GG_ERR_INVALID_ARG = -1
GG_ERR_ALIGNMENT = -2
GG_ERR_NOT_IN_HEAP = -3
GG_ERR_UNSUPPORTED = -4
GG_ERR_CUDA = -5
GG_ERR_TIMEOUT = -6

GG_F16, GG_BF16, GG_F32 = 0, 1, 2
GG_AG_AUTO, GG_AG_BULK, GG_AG_VECTOR, GG_AG_TMA = 0, 1, 2, 3
GG_MAG_AUTO, GG_MAG_1SM, GG_MAG_2SM = 0, 1, 2
GG_COLL_ALL_GATHER, GG_COLL_ALL_GATHER_PARTITIONED, GG_COLL_ALL_TO_ALL = 0, 1, 2
GG_MAX_WORLD = 64
GG_MAX_HEAPS = 1024
GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N, GG_FUSED_BLOCK_N_WIDE = 128, 256, 512
GG_WORKSPACE_SLOT_BYTES = 128
GG_CLAIM_AUTO, GG_CLAIM_ALWAYS, GG_CLAIM_NEVER = 0, 1, 2
GG_STORE_PLAIN, GG_STORE_EVICT_FIRST = 0, 1

# Every entry point declared in include/gemm_gather.h.
EXPORTS = (
    "gg_heap_create", "gg_heap_wrap", "gg_heap_bases", "gg_heap_info", "gg_heap_destroy",
    "gg_heap_set_workspace",
    "gg_all_gather", "gg_all_gather_noalloc", "gg_all_gather_path", "gg_all_gather_check",
    "gg_all_gather_grouped",
    "gg_all_gather_partitioned", "gg_all_to_all", "gg_collective_check",
    "gg_matmul_all_gather", "gg_matmul_all_gather_path", "gg_matmul_all_gather_check",
    "gg_matmul_all_gather_plan",
    "gg_set_claim_policy", "gg_get_claim_policy", "gg_set_store_policy", "gg_get_store_policy",
    "gg_set_wait_limit_ns", "gg_get_wait_limit_ns", "gg_debug_inject_stall",
    "gg_device_status", "gg_clear_device_status",
    "gg_set_trace", "gg_trace_read",
    "gg_last_error", "gg_status_string", "gg_version", "gg_checked_build",
)


class Tile(ctypes.Structure):
    _fields_ = [("block_m", ctypes.c_int), ("block_n", ctypes.c_int)]


class TraceRecord(ctypes.Structure):
    _fields_ = [("start_ns", ctypes.c_uint64), ("start_cycles", ctypes.c_uint64),
                ("end_ns", ctypes.c_uint64), ("end_cycles", ctypes.c_uint64)]


class Group(ctypes.Structure):
    _fields_ = [("rank_start", ctypes.c_int), ("rank_stride", ctypes.c_int),
                ("world_size", ctypes.c_int)]


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    sz = ctypes.c_size_t
    pp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "gg_heap_create": ([vp, sz, i32, vp, vp, pp], i32),
        "gg_heap_wrap": ([vp, sz, i32, vp, pp], i32),
        "gg_heap_bases": ([vp, ctypes.POINTER(u64), i32], i32),
        "gg_heap_info": ([vp, ctypes.POINTER(i32), ctypes.POINTER(sz)], i32),
        "gg_heap_destroy": ([vp], i32),
        "gg_heap_set_workspace": ([vp, vp, sz], i32),
        "gg_all_gather": ([vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group, vp, vp],
                          i32),
        "gg_all_gather_noalloc": ([vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group, vp,
                                   vp], i32),
        "gg_all_gather_path": ([vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group, vp,
                                vp, i32], i32),
        "gg_all_gather_check": ([vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group, i32,
                                 ctypes.POINTER(i32)], i32),
        "gg_all_gather_grouped": ([vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group,
                                   i32, vp, vp, i32], i32),
        "gg_all_gather_partitioned": ([vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group,
                                       vp, vp, i32], i32),
        "gg_all_to_all": ([vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group, vp, vp, i32],
                          i32),
        "gg_collective_check": ([i32, vp, i32, vp, i64, vp, i64, i64, i64, i32, Tile, i32, Group,
                                 i32, i32, ctypes.POINTER(i32)], i32),
        "gg_matmul_all_gather": ([vp, i32, vp, i64, vp, i64, vp, i64, i64, i64, i64, i32, Tile,
                                  i32, Group, vp, vp], i32),
        "gg_matmul_all_gather_path": ([vp, i32, vp, i64, vp, i64, vp, i64, i64, i64, i64, i32,
                                       Tile, i32, Group, vp, vp, i32], i32),
        "gg_matmul_all_gather_check": ([vp, i32, vp, i64, vp, i64, vp, i64, i64, i64, i64, i32,
                                        Tile, i32, Group], i32),
        "gg_matmul_all_gather_plan": ([vp, i32, vp, i64, vp, i64, vp, i64, i64, i64, i64, i32,
                                       Tile, i32, Group, i32, ctypes.POINTER(i32)], i32),
        "gg_set_claim_policy": ([i32], i32),
        "gg_get_claim_policy": ([], i32),
        "gg_set_store_policy": ([i32], i32),
        "gg_get_store_policy": ([], i32),
        "gg_set_wait_limit_ns": ([u64], i32),
        "gg_get_wait_limit_ns": ([], u64),
        "gg_debug_inject_stall": ([i32], i32),
        "gg_device_status": ([vp, ctypes.POINTER(i32)], i32),
        "gg_clear_device_status": ([vp], i32),
        "gg_last_error": ([], ctypes.c_char_p),
        "gg_status_string": ([i32], ctypes.c_char_p),
        "gg_version": ([], i32),
        "gg_checked_build": ([], i32),
        "gg_set_trace": ([i32], i32),
        "gg_trace_read": ([vp, ctypes.POINTER(TraceRecord), ctypes.POINTER(TraceRecord)], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()' or "
            "python gemm_gather_gb300/build.py)")
    return _declare(ctypes.CDLL(LIB_PATH))


lib = load()


class GGError(RuntimeError):
    """A gemm_gather call returned a status other than GG_OK."""

    def __init__(self, status: int, message: str):
        self.status = status
        name = lib.gg_status_string(status).decode()
        super().__init__(f"{name}: {message}")


def check(status: int) -> None:
    if status != GG_OK:
        raise GGError(status, lib.gg_last_error().decode())
