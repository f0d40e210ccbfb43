"""Seeded random calls of the C ABI's validation (no GPU needed).

The kernels trust the host checks: every byte a launch reads or writes must
lie inside the heap, and a gather's input must not overlap any member's
output.  So for 15000 seeded random argument sets each *_check entry point
must either reject with one of the documented status codes, or accept a
request whose buffers, computed here from the arguments alone, stay inside
their partitions (input, gathered output, A; B outside every member's output)
and do not overlap.  gg_heap_wrap and the *_check calls touch no device
state: the addresses below are never dereferenced."""
import random

import pytest

import gemm_gather_gb300 as gg
from gemm_gather_gb300 import _lib

BASE = 1 << 36
TABLE = 1 << 40
PART = 1 << 22
H = 8
ES = {_lib.GG_F16: 2, _lib.GG_BF16: 2, _lib.GG_F32: 4}
DOCUMENTED = {_lib.GG_ERR_INVALID_ARG, _lib.GG_ERR_ALIGNMENT, _lib.GG_ERR_NOT_IN_HEAP,
              _lib.GG_ERR_UNSUPPORTED}
KINDS = ["all_gather", "all_gather_partitioned", "all_to_all"]


def _extent(rows, ld, n, es):
    return ((rows - 1) * ld + n) * es if rows > 0 and n > 0 else 0


def _group(rng):
    W = rng.choice([1, 2, 3, 4, 8, 9])
    stride = rng.choice([1, 1, 2, 3])
    start = rng.choice([0, 0, 1, 2])
    return start, stride, W


def _symmetric_offset(ptr):
    """A heap pointer's byte offset within whichever partition holds it."""
    assert BASE <= ptr < BASE + H * PART, hex(ptr)
    return (ptr - BASE) % PART


def _pick(rng, good, bad, p_good=0.8):
    """Mostly a valid value, sometimes an invalid or edge one."""
    return rng.choice(good) if rng.random() < p_good else rng.choice(bad)


def _offset(rng):
    # mostly aligned buffers inside the partition, sometimes odd or out of range
    o = _pick(rng, [0, 256, 4096, 1 << 20, PART // 2], [PART - 4096, PART + 512, -256])
    return o + _pick(rng, [0], [2, 4, 8, 16], 0.7)


@pytest.mark.parametrize("seed", range(6))
def test_collective_checks_accept_only_in_bounds_requests(seed):
    rng = random.Random(seed)
    heap = gg.heap_wrap(BASE, PART, H, TABLE)
    accepted = 0
    for _ in range(1500):
        kind = rng.choice(KINDS)
        start, stride, W = _group(rng)
        members = [start + i * stride for i in range(W)]
        rank = _pick(rng, [-1, -1, members[0], members[-1]], [rng.randrange(-2, H + 1)])
        dtype = rng.choice([_lib.GG_F16, _lib.GG_BF16, _lib.GG_F32])
        es = ES[dtype]
        M = _pick(rng, [1, 7, 64, 300], [0])
        N = _pick(rng, [1, 24, 256, 520], [0])
        ld_in = N + _pick(rng, [0, 8, 3], [-1])
        ld_out = N + _pick(rng, [0, 16, 5], [-1])
        tile = (_pick(rng, [1, 8, 16, 32], [0, 256, 300]), _pick(rng, [8, 64, 256], [1, 512]))
        programs = _pick(rng, [1, 4, 148], [0, 70000])
        in_off, out_off = _offset(rng), _offset(rng)
        in_home = start if rank == -1 else (rank if 0 <= rank < H else 0)
        inp = BASE + in_home * PART + in_off
        out = BASE + start * PART + out_off
        path = rng.choice(["auto", "auto", "tma", "bulk", "vector"])
        try:
            gg.collective_check(kind, heap, rank, inp, ld_in, out, ld_out, M, N, dtype, tile,
                                programs, (start, stride, W), 0, path)
        except gg.GGError as e:
            assert e.status in DOCUMENTED, (kind, e)
            continue
        accepted += 1
        if M == 0 or N == 0:
            continue
        in_rows = W * M if kind == "all_to_all" else M
        in_ext, out_ext = _extent(in_rows, ld_in, N, es), _extent(W * M, ld_out, N, es)
        assert all(0 <= m < H for m in members)
        out_off = _symmetric_offset(out)
        assert out_off + out_ext <= PART, (kind, out_off, out_ext)
        if rank == -1:
            in_off = _symmetric_offset(inp)
            assert in_off + in_ext <= PART
            assert in_off + in_ext <= out_off or out_off + out_ext <= in_off
        else:
            assert rank in members
            for m in members:  # an external input overlaps no member's output
                o0 = BASE + m * PART + out_off
                assert inp + in_ext <= o0 or o0 + out_ext <= inp
        assert 1 <= tile[0] <= 256 and tile[0] * tile[1] * es <= 32768
        assert 1 <= programs <= 65535
    assert accepted > 100  # the generator reaches the accepting side often enough


@pytest.mark.parametrize("seed", range(4))
def test_fused_check_accepts_only_in_bounds_requests(seed):
    rng = random.Random(100 + seed)
    heap = gg.heap_wrap(BASE, PART, H, TABLE)
    accepted = 0
    for _ in range(1500):
        start, stride, W = _group(rng)
        members = [start + i * stride for i in range(W)]
        rank = _pick(rng, [-1, -1, members[0]], [rng.randrange(-1, H)])
        dtype = _pick(rng, [_lib.GG_F16, _lib.GG_BF16], [_lib.GG_F32])
        M = _pick(rng, [1, 100, 256], [0])
        N = _pick(rng, [8, 256, 264], [0, 7])
        K = _pick(rng, [16, 64, 136], [0])
        lda = K + _pick(rng, [0, 8], [3, -8])
        ldb = N + _pick(rng, [0, 8], [2])
        ld_out = N + _pick(rng, [0, 8], [1, -8])
        tile = _pick(rng, [(128, 256), (128, 512)], [(128, 128), (256, 256), (256, 512)])
        programs = _pick(rng, [1, 2, 152], [0, 70000])
        a_off, out_off = _offset(rng), _offset(rng)
        a_home = start if rank == -1 else (rank if 0 <= rank < H else 0)
        A = BASE + a_home * PART + a_off
        out = BASE + start * PART + out_off
        B = _pick(rng, [BASE + 9 * PART], [BASE + start * PART + out_off, BASE + 9 * PART + 4])
        try:
            gg.matmul_all_gather_check(heap, rank, A, lda, B, ldb, out, ld_out, M, N, K, dtype,
                                       tile, programs, (start, stride, W))
        except gg.GGError as e:
            assert e.status in DOCUMENTED, e
            continue
        accepted += 1
        if M == 0 or N == 0:
            continue
        assert dtype in (_lib.GG_F16, _lib.GG_BF16) and tile in ((128, 256), (128, 512))
        assert tile == (128, 256) or programs >= 2  # the wide tile runs on CTA pairs
        if K == 0:  # the zero fill: only the output is written, A and B never read
            out_ext = _extent(W * M, ld_out, N, 2)
            assert _symmetric_offset(out) + out_ext <= PART
            assert out % 16 == 0 and ld_out % 8 == 0 and N % 8 == 0
            continue
        a_ext, out_ext = _extent(M, lda, K, 2), _extent(W * M, ld_out, N, 2)
        b_ext = _extent(K, ldb, N, 2)
        out_off = _symmetric_offset(out)
        assert out_off + out_ext <= PART
        assert (A | B | out) % 16 == 0 and lda % 8 == 0 and ldb % 8 == 0 and ld_out % 8 == 0
        if rank == -1:
            a_off = _symmetric_offset(A)
            assert a_off + a_ext <= PART
            assert a_off + a_ext <= out_off or out_off + out_ext <= a_off
        for m in members:
            o0 = BASE + m * PART + out_off
            assert B + b_ext <= o0 or o0 + out_ext <= B
            if rank != -1:
                assert A + a_ext <= o0 or o0 + out_ext <= A
    assert accepted > 100
