"""gemm_gather for GB300: tiled all-gather over a symmetric heap, alone and
fused into the epilogue of a matmul (iris PR #626, iris #594, iris #591).

Thin Python binding of the C ABI in include/gemm_gather.h (same names, minus
the ``gg_`` prefix).  It only marshals arguments: torch tensors become device
pointers, the current torch stream becomes the launch stream.  Every step of
the data path runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from ._lib import (GG_AG_AUTO, GG_AG_BULK, GG_AG_TMA, GG_AG_VECTOR, GG_BF16, GG_MAG_1SM, GG_MAG_2SM,
                   GG_MAG_AUTO, GG_COLL_ALL_GATHER, GG_COLL_ALL_GATHER_PARTITIONED,
                   GG_COLL_ALL_TO_ALL, GG_ERR_ALIGNMENT,
                   GG_ERR_CUDA, GG_ERR_INVALID_ARG, GG_ERR_NOT_IN_HEAP, GG_ERR_TIMEOUT,
                   GG_ERR_UNSUPPORTED, GG_F16, GG_F32, GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N,
                   GG_FUSED_BLOCK_N_WIDE,
                   GG_CLAIM_ALWAYS, GG_CLAIM_AUTO, GG_CLAIM_NEVER, GG_MAX_WORLD, GG_OK,
                   GG_WORKSPACE_SLOT_BYTES,
                   GGError, Group, Tile, check, lib, LIB_PATH)

__all__ = [
    "heap_create", "heap_wrap", "heap_bases", "heap_info", "heap_destroy", "heap_set_workspace",
    "all_gather", "all_gather_noalloc",
    "all_gather_check", "all_gather_grouped", "all_gather_partitioned", "all_to_all",
    "collective_check", "matmul_all_gather", "matmul_all_gather_check", "matmul_all_gather_plan",
    "set_claim_policy",
    "get_claim_policy", "CLAIM_POLICIES", "set_store_policy", "get_store_policy",
    "STORE_POLICIES", "set_wait_limit_ns",
    "get_wait_limit_ns", "debug_inject_stall", "device_status", "clear_device_status",
    "checked_build", "set_trace", "trace_read", "SymmetricHeap", "Heap", "GGError", "DTYPE_CODES", "PATHS",
    "FUSED_TILE", "FUSED_TILE_WIDE", "FUSED_PATHS",
]

DTYPE_CODES = {torch.float16: GG_F16, torch.bfloat16: GG_BF16, torch.float32: GG_F32}
PATHS = {"auto": GG_AG_AUTO, "bulk": GG_AG_BULK, "vector": GG_AG_VECTOR, "tma": GG_AG_TMA}
FUSED_PATHS = {"auto": GG_MAG_AUTO, "1sm": GG_MAG_1SM, "2sm": GG_MAG_2SM}
FUSED_TILE = (GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N)             # 128 x 256 per CTA
FUSED_TILE_WIDE = (GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N_WIDE)   # 128 x 512 per CTA (CTA pairs)
CLAIM_POLICIES = {"auto": GG_CLAIM_AUTO, "always": GG_CLAIM_ALWAYS, "never": GG_CLAIM_NEVER}
STORE_POLICIES = {"plain": 0, "evict_first": 1}  # GG_STORE_PLAIN, GG_STORE_EVICT_FIRST


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


# torch's own accessors of the current device and its current raw stream
# (what torch.cuda.current_stream() wraps, without building a Stream object:
# a few microseconds per call that small launches would otherwise pay)
_current_device = getattr(torch._C, "_cuda_getDevice", None)
_current_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int | None:
    if stream is None:
        if not torch.cuda.is_initialized():
            return None  # the legacy default stream
        if _current_device is not None and _current_raw_stream is not None:
            return _current_raw_stream(_current_device()) or None
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _dtype(d) -> int:
    if isinstance(d, torch.dtype):
        return DTYPE_CODES[d]
    return {"f16": GG_F16, "bf16": GG_BF16, "f32": GG_F32}.get(d, d)


@dataclass
class Heap:
    """Host handle of a symmetric heap (wraps ``gg_heap*``)."""
    handle: int

    def __del__(self):
        if getattr(self, "handle", None):
            lib.gg_heap_destroy(self.handle)
            self.handle = None


# --------------------------------------------------------------------------- #
# C ABI, one function per entry point                                         #
# --------------------------------------------------------------------------- #

def heap_create(dev_base, bytes_per_rank: int, num_heaps: int, dev_bases_table,
                stream=None) -> Heap:
    out = ctypes.c_void_p()
    check(lib.gg_heap_create(_ptr(dev_base), bytes_per_rank, num_heaps, _ptr(dev_bases_table),
                             _stream(stream), ctypes.byref(out)))
    return Heap(out.value)


def heap_wrap(dev_base, bytes_per_rank: int, num_heaps: int, dev_bases_table) -> Heap:
    out = ctypes.c_void_p()
    check(lib.gg_heap_wrap(_ptr(dev_base), bytes_per_rank, num_heaps, _ptr(dev_bases_table),
                           ctypes.byref(out)))
    return Heap(out.value)


def heap_bases(heap: Heap, n: int | None = None) -> list[int]:
    if n is None:
        n = heap_info(heap)[0]
    buf = (ctypes.c_uint64 * n)()
    check(lib.gg_heap_bases(heap.handle, buf, n))
    return list(buf)


def heap_info(heap: Heap) -> tuple[int, int]:
    h, part = ctypes.c_int(), ctypes.c_size_t()
    check(lib.gg_heap_info(heap.handle, ctypes.byref(h), ctypes.byref(part)))
    return h.value, part.value


def heap_destroy(heap: Heap) -> None:
    if heap.handle:
        check(lib.gg_heap_destroy(heap.handle))
        heap.handle = None


def heap_set_workspace(heap: Heap, dev_work, nbytes: int) -> None:
    """Workspace for load-balanced launches (``dev_work`` None and 0 bytes: none)."""
    check(lib.gg_heap_set_workspace(heap.handle, _ptr(dev_work), nbytes))


def all_gather(heap: Heap, rank: int, input, ld_in: int, output, ld_out: int, M: int, N: int,
               dtype, tile: tuple[int, int], comm_programs: int,
               group: tuple[int, int, int], status=None, stream=None, path: str = "auto") -> None:
    check(lib.gg_all_gather_path(heap.handle, rank, _ptr(input), ld_in, _ptr(output), ld_out, M,
                                 N, _dtype(dtype), Tile(*tile), comm_programs, Group(*group),
                                 _ptr(status), _stream(stream), PATHS[path]))


def all_gather_noalloc(heap: Heap, rank: int, input, ld_in: int, output, ld_out: int, M: int,
                       N: int, dtype, tile: tuple[int, int], comm_programs: int,
                       group: tuple[int, int, int], status=None, stream=None) -> None:
    """gg_all_gather for callers that cannot allocate device memory: a
    claiming launch keeps its counter in the library's static device array
    (shared by every call on the device; calls that overlap on the GPU race)."""
    check(lib.gg_all_gather_noalloc(heap.handle, rank, _ptr(input), ld_in, _ptr(output), ld_out,
                                    M, N, _dtype(dtype), Tile(*tile), comm_programs, Group(*group),
                                    _ptr(status), _stream(stream)))


def all_gather_check(heap: Heap, rank: int, input, ld_in: int, output, ld_out: int, M: int,
                     N: int, dtype, tile: tuple[int, int], comm_programs: int,
                     group: tuple[int, int, int], path: str = "auto") -> str:
    """Validate without launching; returns the path a launch would take."""
    chosen = ctypes.c_int()
    check(lib.gg_all_gather_check(heap.handle, rank, _ptr(input), ld_in, _ptr(output), ld_out, M,
                                  N, _dtype(dtype), Tile(*tile), comm_programs, Group(*group),
                                  PATHS[path], ctypes.byref(chosen)))
    return {GG_AG_AUTO: "none", GG_AG_BULK: "bulk", GG_AG_VECTOR: "vector",
            GG_AG_TMA: "tma"}[chosen.value]


def all_gather_grouped(heap: Heap, rank: int, input, ld_in: int, output, ld_out: int, M: int,
                       N: int, dtype, tile: tuple[int, int], comm_programs: int,
                       group: tuple[int, int, int], dests_per_wait: int, status=None, stream=None,
                       path: str = "auto") -> None:
    check(lib.gg_all_gather_grouped(heap.handle, rank, _ptr(input), ld_in, _ptr(output), ld_out,
                                    M, N, _dtype(dtype), Tile(*tile), comm_programs, Group(*group),
                                    dests_per_wait, _ptr(status), _stream(stream), PATHS[path]))


def all_gather_partitioned(heap: Heap, rank: int, input, ld_in: int, output, ld_out: int, M: int,
                           N: int, dtype, tile: tuple[int, int], comm_programs: int,
                           group: tuple[int, int, int], status=None, stream=None,
                           path: str = "auto") -> None:
    check(lib.gg_all_gather_partitioned(heap.handle, rank, _ptr(input), ld_in, _ptr(output),
                                        ld_out, M, N, _dtype(dtype), Tile(*tile), comm_programs,
                                        Group(*group), _ptr(status), _stream(stream),
                                        PATHS[path]))


def all_to_all(heap: Heap, rank: int, input, ld_in: int, output, ld_out: int, M: int, N: int,
               dtype, tile: tuple[int, int], comm_programs: int, group: tuple[int, int, int],
               status=None, stream=None, path: str = "auto") -> None:
    check(lib.gg_all_to_all(heap.handle, rank, _ptr(input), ld_in, _ptr(output), ld_out, M, N,
                            _dtype(dtype), Tile(*tile), comm_programs, Group(*group),
                            _ptr(status), _stream(stream), PATHS[path]))


COLLECTIVES = {"all_gather": GG_COLL_ALL_GATHER,
               "all_gather_partitioned": GG_COLL_ALL_GATHER_PARTITIONED,
               "all_to_all": GG_COLL_ALL_TO_ALL}


def collective_check(kind: str, heap: Heap, rank: int, input, ld_in: int, output, ld_out: int,
                     M: int, N: int, dtype, tile: tuple[int, int], comm_programs: int,
                     group: tuple[int, int, int], dests_per_wait: int = 0,
                     path: str = "auto") -> str:
    """Validate without launching; returns the path a launch would take."""
    chosen = ctypes.c_int()
    check(lib.gg_collective_check(COLLECTIVES[kind], heap.handle, rank, _ptr(input), ld_in,
                                  _ptr(output), ld_out, M, N, _dtype(dtype), Tile(*tile),
                                  comm_programs, Group(*group), dests_per_wait, PATHS[path],
                                  ctypes.byref(chosen)))
    return {GG_AG_AUTO: "none", GG_AG_BULK: "bulk", GG_AG_VECTOR: "vector",
            GG_AG_TMA: "tma"}[chosen.value]


def matmul_all_gather(heap: Heap, rank: int, A, lda: int, B, ldb: int, output, ld_out: int,
                      M: int, N: int, K: int, dtype, tile: tuple[int, int], comm_programs: int,
                      group: tuple[int, int, int], status=None, stream=None,
                      path: str = "auto") -> None:
    check(lib.gg_matmul_all_gather_path(heap.handle, rank, _ptr(A), lda, _ptr(B), ldb,
                                        _ptr(output), ld_out, M, N, K, _dtype(dtype), Tile(*tile),
                                        comm_programs, Group(*group), _ptr(status),
                                        _stream(stream), FUSED_PATHS[path]))


def matmul_all_gather_check(heap: Heap, rank: int, A, lda: int, B, ldb: int, output,
                            ld_out: int, M: int, N: int, K: int, dtype, tile: tuple[int, int],
                            comm_programs: int, group: tuple[int, int, int]) -> None:
    check(lib.gg_matmul_all_gather_check(heap.handle, rank, _ptr(A), lda, _ptr(B), ldb,
                                         _ptr(output), ld_out, M, N, K, _dtype(dtype),
                                         Tile(*tile), comm_programs, Group(*group)))


def matmul_all_gather_plan(heap: Heap, rank: int, A, lda: int, B, ldb: int, output, ld_out: int,
                           M: int, N: int, K: int, dtype, tile: tuple[int, int],
                           comm_programs: int, group: tuple[int, int, int],
                           path: str = "auto") -> str:
    """Validate without launching; returns the kernel variant a launch would
    run ("1sm" or "2sm"; "none" when there is nothing to launch)."""
    chosen = ctypes.c_int()
    check(lib.gg_matmul_all_gather_plan(heap.handle, rank, _ptr(A), lda, _ptr(B), ldb,
                                        _ptr(output), ld_out, M, N, K, _dtype(dtype), Tile(*tile),
                                        comm_programs, Group(*group), FUSED_PATHS[path],
                                        ctypes.byref(chosen)))
    return {GG_MAG_AUTO: "none", GG_MAG_1SM: "1sm", GG_MAG_2SM: "2sm"}[chosen.value]


def set_claim_policy(policy: str) -> None:
    """Which launches claim runs of tiles from the heap's workspace:
    "auto", "always" or "never"."""
    check(lib.gg_set_claim_policy(CLAIM_POLICIES[policy]))


def get_claim_policy() -> str:
    code = int(lib.gg_get_claim_policy())
    return next(k for k, v in CLAIM_POLICIES.items() if v == code)


def set_store_policy(policy: str) -> None:
    """L2 hint on the all-gather family's tensor-map and bulk stores:
    "evict_first" (the library's default) or "plain" (none).  Results are
    identical."""
    check(lib.gg_set_store_policy(STORE_POLICIES[policy]))


def get_store_policy() -> str:
    code = int(lib.gg_get_store_policy())
    return next(k for k, v in STORE_POLICIES.items() if v == code)


def set_wait_limit_ns(ns: int) -> None:
    check(lib.gg_set_wait_limit_ns(ns))


def get_wait_limit_ns() -> int:
    return int(lib.gg_get_wait_limit_ns())


def debug_inject_stall(enable: bool) -> None:
    check(lib.gg_debug_inject_stall(1 if enable else 0))


def device_status(stream=None) -> int:
    """The library's status word of the current device (where launches given
    no status word report a wait that gave up), after ``stream``'s queued work."""
    out = ctypes.c_int()
    check(lib.gg_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def clear_device_status(stream=None) -> None:
    """Reset the library's status word of the current device to 0 (on ``stream``)."""
    check(lib.gg_clear_device_status(_stream(stream)))


def set_trace(enable: bool) -> None:
    """Launches after this call record their first CTA's start and end wall time
    and SM cycle counter (gg_set_trace); False stops it."""
    check(lib.gg_set_trace(1 if enable else 0))


def trace_read(stream=None) -> dict:
    """The last traced launch of each kernel family, after ``stream``'s queued
    work: {"all_gather": {...}, "matmul_all_gather": {...}}, each with the raw
    record, its wall time (ns), SM cycles and clock (MHz; None if unwritten)."""
    from ._lib import TraceRecord
    rec = {k: TraceRecord() for k in ("all_gather", "matmul_all_gather")}
    check(lib.gg_trace_read(_stream(stream), ctypes.byref(rec["all_gather"]),
                            ctypes.byref(rec["matmul_all_gather"])))
    out = {}
    for k, r in rec.items():
        ns, cyc = r.end_ns - r.start_ns, r.end_cycles - r.start_cycles
        out[k] = {"start_ns": r.start_ns, "end_ns": r.end_ns, "start_cycles": r.start_cycles,
                  "end_cycles": r.end_cycles, "ns": ns, "cycles": cyc,
                  "sm_mhz": cyc * 1e3 / ns if r.end_ns > r.start_ns else None}
    return out


def checked_build() -> bool:
    """True when the loaded library is the checked build (GEMM_GATHER_CHECKED=1 at
    import): the gather kernels bound every access and report GG_ERR_NOT_IN_HEAP."""
    return bool(lib.gg_checked_build())


# --------------------------------------------------------------------------- #
# Device memory for a heap (torch allocates; the library never does)          #
# --------------------------------------------------------------------------- #

class SymmetricHeap:
    """H partitions of ``part_bytes`` each in one torch device allocation,
    plus the device heap-bases table, registered with ``gg_heap_create``."""

    ALIGN = 256

    def __init__(self, num_heaps: int, part_bytes: int, device="cuda", fill: int | None = None,
                 stream=None, workspace_slots: int = 64):
        if part_bytes % self.ALIGN:
            part_bytes += self.ALIGN - part_bytes % self.ALIGN
        self.H = num_heaps
        self.part_bytes = part_bytes
        raw = torch.empty(num_heaps * part_bytes + self.ALIGN, dtype=torch.uint8, device=device)
        shift = (-raw.data_ptr()) % self.ALIGN
        self._raw = raw
        self.storage = raw[shift: shift + num_heaps * part_bytes]
        if fill is not None:
            self.storage.fill_(fill)
        self.table = torch.empty(num_heaps, dtype=torch.int64, device=device)
        self.heap = heap_create(self.storage, part_bytes, num_heaps, self.table, stream=stream)
        # load-balancing counters (each launch that uses a slot zeroes it first)
        self.workspace = None
        if workspace_slots:
            nbytes = workspace_slots * GG_WORKSPACE_SLOT_BYTES
            ws = torch.zeros(nbytes + self.ALIGN, dtype=torch.uint8, device=device)
            shift = (-ws.data_ptr()) % self.ALIGN
            self._ws_raw = ws
            self.workspace = ws[shift: shift + nbytes]
            heap_set_workspace(self.heap, self.workspace, nbytes)

    @property
    def base(self) -> int:
        return self.storage.data_ptr()

    def partition(self, h: int) -> torch.Tensor:
        return self.storage[h * self.part_bytes: (h + 1) * self.part_bytes]

    def view(self, h: int, offset: int, rows: int, cols: int, ld: int,
             dtype: torch.dtype) -> torch.Tensor:
        """rows x cols view (row pitch ld elements) at ``offset`` in partition h."""
        es = torch.empty((), dtype=dtype).element_size()
        assert offset % es == 0
        n = ((rows - 1) * ld + cols) if rows else 0
        flat = self.partition(h)[offset: offset + n * es].view(dtype)
        return flat.as_strided((rows, cols), (ld, 1))

    def ptr(self, h: int, offset: int) -> int:
        return self.base + h * self.part_bytes + offset
