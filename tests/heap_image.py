"""Host-side heap images for the tests: H partitions, each holding a guard
band, an input block, a guard band, a gathered output and a guard band, the
rest filled with the sentinel byte.  Shared by the oracle pins and the GPU
parity tests (placement only; no arithmetic of the method)."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from gg_inputs import SENTINEL_BYTE

GUARD = 256  # bytes of sentinel before and after every buffer


def _align(x: int, a: int) -> int:
    return (x + a - 1) // a * a


@dataclass
class Layout:
    H: int
    part_bytes: int
    in_off: int
    ld_in: int
    out_off: int
    ld_out: int
    M: int
    N: int
    W: int
    esize: int

    @property
    def in_bytes(self) -> int:
        return ((self.M - 1) * self.ld_in + self.N) * self.esize if self.M else 0

    @property
    def out_bytes(self) -> int:
        rows = self.W * self.M
        return ((rows - 1) * self.ld_out + self.N) * self.esize if rows else 0


def make_layout(H: int, W: int, M: int, N: int, esize: int, ld_in: int | None = None,
                ld_out: int | None = None, align: int = 256, extra_in: int = 0,
                extra_out: int = 0) -> Layout:
    """Place the input at a guard-separated offset and the output after it.
    ``extra_in`` / ``extra_out`` shift the buffers by that many bytes past an
    ``align`` boundary (for misalignment cases)."""
    ld_in = N if ld_in is None else ld_in
    ld_out = N if ld_out is None else ld_out
    in_off = _align(GUARD, align) + extra_in
    in_bytes = max(M * ld_in * esize, 1)
    out_off = _align(in_off + in_bytes + GUARD, align) + extra_out
    out_bytes = max(W * M * ld_out * esize, 1)
    part = _align(out_off + out_bytes + GUARD, 2 * 1024 * 1024 if out_bytes > (1 << 24) else 4096)
    return Layout(H, part, in_off, ld_in, out_off, ld_out, M, N, W, esize)


def sentinel_heap(lay: Layout) -> np.ndarray:
    return np.full(lay.H * lay.part_bytes, SENTINEL_BYTE, dtype=np.uint8)


def put_block(heap: np.ndarray, lay: Layout, h: int, block: np.ndarray, off: int, ld: int) -> None:
    """Write an M x N block (any dtype of lay.esize bytes) at ``off`` in
    partition h with row pitch ``ld`` elements."""
    raw = np.ascontiguousarray(block).view(np.uint8).reshape(block.shape[0], -1)
    base = h * lay.part_bytes + off
    for m in range(block.shape[0]):
        s = base + m * ld * lay.esize
        heap[s: s + raw.shape[1]] = raw[m]


def get_block(heap: np.ndarray, lay: Layout, h: int, off: int, rows: int, ld: int,
              cols: int, dtype) -> np.ndarray:
    """Read a rows x cols block at ``off`` in partition h (row pitch ld)."""
    es = np.dtype(dtype).itemsize
    base = h * lay.part_bytes + off
    out = np.empty((rows, cols), dtype=dtype)
    for m in range(rows):
        s = base + m * ld * es
        out[m] = heap[s: s + cols * es].view(dtype)
    return out


def output_mask(lay: Layout, members: list[int]) -> np.ndarray:
    """True on the bytes a gather may change: the N valid columns of the W*M
    output rows of every member partition."""
    mask = np.zeros(lay.H * lay.part_bytes, dtype=bool)
    for h in members:
        base = h * lay.part_bytes + lay.out_off
        for r in range(lay.W * lay.M):
            s = base + r * lay.ld_out * lay.esize
            mask[s: s + lay.N * lay.esize] = True
    return mask
