"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method: it only draws numbers.  Both
the oracle side and the CUDA side receive the same host tensors from here.

Recipe (one ``torch.Generator`` on the CPU, seeded; values drawn in float32
and rounded to the target 16-bit type with round-to-nearest-even):
  * uniform[-1, 1]:      2 * U[0, 1) - 1
  * normal(0, 1) * scale (scale = 1/sqrt(K) for GEMM operands)
  * integer-valued:      uniform integers in [lo, hi]  (exact-product tests)
  * index-coded:         element bits = a hash of (rank, row, column), so a
                         misplaced, duplicated or missing element is visible.
Ranks draw in heap order 0..H-1, then the shared operand B.
"""
from __future__ import annotations

import torch

SENTINEL_BYTE = 0xA5  # fill of padding, guard bands and inactive heaps

DTYPES = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "f32": torch.float32,
}


def generator(seed: int = 0, device="cpu") -> torch.Generator:
    """Seeded generator; on the CPU unless a device is named (benchmarks of
    large shapes draw on the GPU; parity tests always draw on the CPU)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def uniform_pm1(shape, dtype: torch.dtype, gen: torch.Generator) -> torch.Tensor:
    u = torch.rand(shape, generator=gen, dtype=torch.float32, device=gen.device)
    return (2.0 * u - 1.0).to(dtype)


def normal(shape, dtype: torch.dtype, gen: torch.Generator, scale: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=gen.device)
    return (x * scale).to(dtype)


def integers(shape, lo: int, hi: int, dtype: torch.dtype, gen: torch.Generator) -> torch.Tensor:
    return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int64,
                         device=gen.device).to(dtype)


def _mix32(x: torch.Tensor) -> torch.Tensor:
    # 32-bit integer finaliser (xorshift-multiply), on int64 holding uint32 values
    mask = 0xFFFFFFFF
    x = x & mask
    x = ((x ^ (x >> 16)) * 0x7FEB352D) & mask
    x = ((x ^ (x >> 15)) * 0x846CA68B) & mask
    return x ^ (x >> 16)


def index_packed(rank: int, M: int, N: int, esize: int) -> torch.Tensor:
    """An M x N block whose element bits are (rank, m, n) packed into bit
    fields, so every element of every rank is distinct and decodable.  For
    16-bit elements: rank < 4, m < 32, n < 512 (bits 14-15, 9-13, 0-8); for
    32-bit elements: rank < 256, m < 4096, n < 4096 (bits 24-31, 12-23, 0-11).
    Returned as int16/int32 raw bit patterns."""
    if esize == 2:
        if not (rank < 4 and M <= 32 and N <= 512):
            raise ValueError("index_packed (16-bit) needs rank < 4, M <= 32, N <= 512")
        shift_r, shift_m = 14, 9
    elif esize == 4:
        if not (rank < 256 and M <= 4096 and N <= 4096):
            raise ValueError("index_packed (32-bit) needs rank < 256, M, N <= 4096")
        shift_r, shift_m = 24, 12
    else:
        raise ValueError("index_packed supports 2- and 4-byte elements")
    m = torch.arange(M, dtype=torch.int64).view(M, 1)
    n = torch.arange(N, dtype=torch.int64).view(1, N)
    bits = (rank << shift_r) | (m << shift_m) | n
    top = 1 << (8 * esize - 1)
    bits = bits - ((bits >= top).to(torch.int64) << (8 * esize))
    return bits.to(torch.int16 if esize == 2 else torch.int32)


def index_packed_decode(bits: torch.Tensor, esize: int):
    """Inverse of index_packed: (rank, m, n) tensors from raw bit patterns."""
    u = bits.to(torch.int64) & ((1 << (8 * esize)) - 1)
    if esize == 2:
        return u >> 14, (u >> 9) & 31, u & 511
    return u >> 24, (u >> 12) & 4095, u & 4095


def index_coded(rank: int, M: int, N: int, esize: int) -> torch.Tensor:
    """An M x N block whose element bits hash (rank, m, n); dtype int16/int32
    (raw bit patterns for 16- or 32-bit elements)."""
    m = torch.arange(M, dtype=torch.int64).view(M, 1)
    n = torch.arange(N, dtype=torch.int64).view(1, N)
    key = (rank * 1_000_003 + m * 65_537 + n * 257) & 0xFFFFFFFF
    h = _mix32(key + 0x9E3779B9)
    if esize == 2:
        h = h & 0xFFFF
        return (h - ((h >= 0x8000).to(torch.int64) << 16)).to(torch.int16)
    if esize == 4:
        return (h - ((h >= 0x80000000).to(torch.int64) << 32)).to(torch.int32)
    raise ValueError("index_coded supports 2- and 4-byte elements")
