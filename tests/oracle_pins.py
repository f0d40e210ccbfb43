"""Pins of the oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` (the real build or a build
with a planted mistake, see test_oracle_mutants.py) and raises AssertionError
when the oracle disagrees with what the pages and the mathematics fix:

* placement of the gather by brute force on tiny sizes with index-packed
  inputs (every element encodes its own (rank, row, column), decoded by the
  test), plus the invariants of iris #594 "Local validation" (padding, guards,
  inactive heaps untouched) and the special case W = 1 (a plain 2-D copy);
* group membership by divisibility (iris #591, Description §1);
* 16-bit decoding/encoding against numpy float16 and torch bfloat16;
* the float64 matmul against numpy's float64 matmul within the classical
  summation error bound, and exactly on integer-valued operands, one-hot rows,
  an identity B and all-ones operands (closed forms).
"""
from __future__ import annotations

import numpy as np
import torch

import gg_inputs
from tests import heap_image as hi

# --------------------------------------------------------------------------- #
# group resolution                                                            #
# --------------------------------------------------------------------------- #


def pin_group_index(o) -> None:
    for (H, start, stride, W) in [(8, 0, 1, 8), (8, 1, 2, 4), (8, 0, 2, 4), (5, 4, 1, 1),
                                  (9, 2, 3, 3), (4, 0, 1, 2)]:
        for h in range(H + 2):
            d = h - start
            expect = d // stride if (d >= 0 and d % stride == 0 and d // stride < W) else -1
            got = o.group_index(h, start, stride, W)
            assert got == expect, (H, start, stride, W, h, got, expect)


# --------------------------------------------------------------------------- #
# all-gather placement                                                        #
# --------------------------------------------------------------------------- #

# (H, group, M, N, ld_in pad, ld_out pad, esize)
GATHER_CASES = [
    (1, (0, 1, 1), 3, 5, 0, 0, 2),
    (2, (0, 1, 2), 4, 7, 1, 3, 2),
    (3, (0, 1, 3), 5, 16, 0, 2, 2),
    (4, (0, 1, 4), 17, 40, 2, 1, 2),
    (4, (0, 1, 4), 1, 1, 0, 0, 2),
    (4, (1, 2, 2), 6, 9, 0, 5, 2),
    (8, (1, 2, 4), 7, 33, 1, 7, 4),
    (8, (0, 2, 4), 9, 12, 0, 0, 4),
    (6, (2, 1, 3), 2, 3, 0, 1, 4),
]


def _members(group):
    s, st, W = group
    return [s + i * st for i in range(W)]


def _packed_setup(H, group, M, N, pad_in, pad_out, esize):
    W = group[2]
    lay = hi.make_layout(H, W, M, N, esize, ld_in=N + pad_in, ld_out=N + pad_out)
    heap = hi.sentinel_heap(lay)
    npdt = np.int16 if esize == 2 else np.int32
    for h in _members(group):
        blk = gg_inputs.index_packed(h, M, N, esize).numpy().astype(npdt)
        hi.put_block(heap, lay, h, blk, lay.in_off, lay.ld_in)
    return lay, heap, npdt


def _check_packed_outputs(heap, before, lay, group, npdt, blocks=None):
    """Every member's output row block i holds member(i)'s element (m, n);
    every byte outside the outputs is unchanged."""
    members = _members(group)
    W, M, N = group[2], lay.M, lay.N
    all_blocks = blocks is None
    blocks = range(W) if all_blocks else blocks
    for d in members:
        out = hi.get_block(heap, lay, d, lay.out_off, W * M, lay.ld_out, N, npdt)
        for i in blocks:
            r, m, n = gg_inputs.index_packed_decode(torch.from_numpy(out[i * M:(i + 1) * M]),
                                                    lay.esize)
            assert bool((r == members[i]).all()), ("rank field", d, i)
            assert bool((m == torch.arange(M).view(M, 1)).all()), ("row field", d, i)
            assert bool((n == torch.arange(N).view(1, N)).all()), ("column field", d, i)
    mask = hi.output_mask(lay, members)
    if not all_blocks:
        # only the written blocks may differ
        mask = np.zeros_like(mask)
        for d in members:
            for i in blocks:
                base = d * lay.part_bytes + lay.out_off
                for rr in range(i * M, (i + 1) * M):
                    s = base + rr * lay.ld_out * lay.esize
                    mask[s: s + N * lay.esize] = True
    assert np.array_equal(heap[~mask], before[~mask]), "bytes outside the output changed"


def pin_gather_packed(o) -> None:
    for (H, group, M, N, pi, po, es) in GATHER_CASES:
        lay, heap, npdt = _packed_setup(H, group, M, N, pi, po, es)
        before = heap.copy()
        o.all_gather(heap, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out,
                     M, N, es, group)
        _check_packed_outputs(heap, before, lay, group, npdt)


def pin_gather_single_contribution(o) -> None:
    """One rank's call writes its own row block, and only that, everywhere."""
    for (H, group, M, N, pi, po, es) in GATHER_CASES:
        lay, heap, npdt = _packed_setup(H, group, M, N, pi, po, es)
        members = _members(group)
        i = len(members) - 1
        h = members[i]
        src = hi.get_block(heap, lay, h, lay.in_off, M, lay.ld_in, N, npdt)
        before = heap.copy()
        o.gather_contribution(heap, lay.part_bytes, src, lay.out_off, lay.ld_out, M, N,
                              group, h)
        _check_packed_outputs(heap, before, lay, group, npdt, blocks=[i])


def pin_gather_w1_copy(o) -> None:
    """W = 1 reduces to a plain 2-D copy of the block (numpy slicing)."""
    rng = np.random.default_rng(1)
    for (M, N, ld_in, ld_out, dt) in [(5, 7, 9, 8, np.float32), (3, 4, 4, 6, np.float16),
                                       (1, 33, 40, 33, np.int16)]:
        es = np.dtype(dt).itemsize
        lay = hi.make_layout(3, 1, M, N, es, ld_in=ld_in, ld_out=ld_out)
        heap = hi.sentinel_heap(lay)
        blk = rng.standard_normal((M, N)).astype(dt)
        hi.put_block(heap, lay, 2, blk, lay.in_off, ld_in)
        o.all_gather(heap, lay.part_bytes, lay.in_off, ld_in, lay.out_off, ld_out, M, N, es,
                     (2, 1, 1))
        out = hi.get_block(heap, lay, 2, lay.out_off, M, ld_out, N, dt)
        assert out.tobytes() == blk.tobytes()


# --------------------------------------------------------------------------- #
# all-to-all                                                                  #
# --------------------------------------------------------------------------- #

A2A_CASES = [
    # (H, group, M, N, ld_in pad, ld_out pad)
    (1, (0, 1, 1), 3, 5, 0, 0),
    (2, (0, 1, 2), 4, 7, 1, 3),
    (3, (0, 1, 3), 5, 16, 0, 2),
    (8, (1, 2, 4), 6, 9, 2, 0),
    (6, (2, 1, 3), 1, 1, 0, 1),
]


def _a2a_setup(H, group, M, N, pi, po):
    W = group[2]
    # input W*M x N per member; the output has the same shape
    lay = hi.make_layout(H, W, W * M, N, 4, ld_in=N + pi, ld_out=N + po)
    heap = hi.sentinel_heap(lay)
    for h in _members(group):
        blk = gg_inputs.index_packed(h, W * M, N, 4).numpy()
        hi.put_block(heap, lay, h, blk, lay.in_off, lay.ld_in)
    return lay, heap


def pin_all_to_all_packed(o) -> None:
    """out_d row block i = member i's input row block d, decoded element by element."""
    for (H, group, M, N, pi, po) in A2A_CASES:
        lay, heap = _a2a_setup(H, group, M, N, pi, po)
        W = group[2]
        members = _members(group)
        before = heap.copy()
        o.all_to_all(heap, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                     4, group)
        for di, d in enumerate(members):
            out = hi.get_block(heap, lay, d, lay.out_off, W * M, lay.ld_out, N, np.int32)
            for i in range(W):
                r, m, n = gg_inputs.index_packed_decode(torch.from_numpy(out[i * M:(i + 1) * M]), 4)
                assert bool((r == members[i]).all()), ("rank", d, i)
                assert bool((m == di * M + torch.arange(M).view(M, 1)).all()), ("row", d, i)
                assert bool((n == torch.arange(N).view(1, N)).all()), ("col", d, i)
        # only the W*M x N outputs of the members change
        mask = np.zeros(lay.H * lay.part_bytes, dtype=bool)
        for d in members:
            base = d * lay.part_bytes + lay.out_off
            for rr in range(W * M):
                s0 = base + rr * lay.ld_out * 4
                mask[s0: s0 + N * 4] = True
        assert np.array_equal(heap[~mask], before[~mask])


def pin_all_to_all_twice_is_identity(o) -> None:
    """Exchanging twice returns every member's original blocks (an involution)."""
    rng = np.random.default_rng(3)
    for (H, group, M, N) in [(4, (0, 1, 4), 3, 6), (7, (1, 3, 2), 2, 5), (3, (0, 1, 3), 1, 2)]:
        W = group[2]
        lay = hi.make_layout(H, W, W * M, N, 2)
        heap = hi.sentinel_heap(lay)
        orig = {}
        for h in _members(group):
            orig[h] = rng.integers(-30000, 30000, size=(W * M, N)).astype(np.int16)
            hi.put_block(heap, lay, h, orig[h], lay.in_off, N)
        o.all_to_all(heap, lay.part_bytes, lay.in_off, N, lay.out_off, N, M, N, 2, group)
        # second exchange: the outputs become the inputs
        o.all_to_all(heap, lay.part_bytes, lay.out_off, N, lay.in_off, N, M, N, 2, group)
        for h in _members(group):
            back = hi.get_block(heap, lay, h, lay.in_off, W * M, N, N, np.int16)
            assert np.array_equal(back, orig[h]), h


def pin_all_to_all_w1_copy(o) -> None:
    lay = hi.make_layout(2, 1, 5, 7, 4, ld_in=9, ld_out=8)
    heap = hi.sentinel_heap(lay)
    blk = np.arange(35, dtype=np.int32).reshape(5, 7) * 7919
    hi.put_block(heap, lay, 1, blk, lay.in_off, 9)
    o.all_to_all(heap, lay.part_bytes, lay.in_off, 9, lay.out_off, 8, 5, 7, 4, (1, 1, 1))
    assert np.array_equal(hi.get_block(heap, lay, 1, lay.out_off, 5, 8, 7, np.int32), blk)


# --------------------------------------------------------------------------- #
# 16-bit formats                                                              #
# --------------------------------------------------------------------------- #

def _ref_decode_all(fmt):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if fmt == 0:
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def pin_decode16(o) -> None:
    for fmt in (0, 1):
        ref = _ref_decode_all(fmt)
        got = np.array([o.decode16(b, fmt) for b in range(65536)])
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan), fmt
        assert np.array_equal(got[~nan], ref[~nan]), fmt
        # signed zeros
        assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), fmt


def _encode_cases():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(6000).astype(np.float32)
    with np.errstate(over="ignore"):
        big = (x * np.float32(1e38)).astype(np.float32)
    x = np.concatenate([
        x, x * 1e-5, x * 1e-8, x * 3e4, big,
        # exact ties and neighbours at several scales (binary16 and bfloat16)
        np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 2 ** -25,
                  3 * 2 ** -25, 2 ** -24 * 1.5, 65504.0, 65519.0, 65520.0, 7e4, 0.0,
                  -0.0, 2 ** -133, 3 * 2 ** -134, 3.3895314e38], dtype=np.float32),
    ]).astype(np.float32)
    return np.concatenate([x, -x])


def pin_encode16(o) -> None:
    x = _encode_cases()
    with np.errstate(over="ignore"):
        ref16 = x.astype(np.float16).view(np.uint16)
    refbf = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got16 = np.array([o.encode16(float(v), 0) for v in x], dtype=np.uint16)
    gotbf = np.array([o.encode16(float(v), 1) for v in x], dtype=np.uint16)
    assert np.array_equal(got16, ref16), np.nonzero(got16 != ref16)[0][:5]
    assert np.array_equal(gotbf, refbf), np.nonzero(gotbf != refbf)[0][:5]


# --------------------------------------------------------------------------- #
# float64 matmul                                                              #
# --------------------------------------------------------------------------- #

def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _as_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def pin_matmul_numpy(o) -> None:
    """float64 result within the summation error bound of numpy's float64 matmul."""
    g = gg_inputs.generator(3)
    for fmt, dt in ((0, torch.float16), (1, torch.bfloat16)):
        for (M, N, K) in [(7, 9, 13), (33, 17, 64), (5, 40, 300), (1, 1, 1)]:
            A = gg_inputs.normal((M, K), dt, g)
            B = gg_inputs.normal((K, N), dt, g, scale=K ** -0.5)
            C = o.matmul_f64(_bits(A), _bits(B), fmt)
            Af, Bf = _as_f64(A), _as_f64(B)
            ref = Af @ Bf
            bound = 2.0 * K * np.finfo(np.float64).eps * (np.abs(Af) @ np.abs(Bf)) + 1e-300
            assert np.all(np.abs(C - ref) <= bound), (fmt, M, N, K)


def pin_matmul_integers_exact(o) -> None:
    g = gg_inputs.generator(5)
    for fmt, dt in ((0, torch.float16), (1, torch.bfloat16)):
        for (M, N, K) in [(8, 16, 64), (13, 7, 5), (1, 3, 2)]:
            A = gg_inputs.integers((M, K), -2, 2, dt, g)
            B = gg_inputs.integers((K, N), -2, 2, dt, g)
            C = o.matmul_f64(_bits(A), _bits(B), fmt)
            ref = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy()
            assert np.array_equal(C, ref.astype(np.float64)), (fmt, M, N, K)


def pin_matmul_closed_forms(o) -> None:
    g = gg_inputs.generator(9)
    for fmt, dt in ((0, torch.float16), (1, torch.bfloat16)):
        M, N, K = 6, 10, 12
        B = gg_inputs.normal((K, N), dt, g)
        # one-hot rows of A pick rows of B exactly
        pick = [3, 0, 11, 7, 7, 5]
        A = torch.zeros((M, K), dtype=dt)
        for m, k in enumerate(pick):
            A[m, k] = 1
        C = o.matmul_f64(_bits(A), _bits(B), fmt)
        assert np.array_equal(C, _as_f64(B)[pick]), fmt
        # identity B reproduces A
        A2 = gg_inputs.normal((M, K), dt, g)
        I = torch.eye(K, dtype=dt)
        C2 = o.matmul_f64(_bits(A2), _bits(I), fmt)
        assert np.array_equal(C2, _as_f64(A2)), fmt
        # all ones: every entry is K
        ones_a, ones_b = torch.ones((M, K), dtype=dt), torch.ones((K, N), dtype=dt)
        C3 = o.matmul_f64(_bits(ones_a), _bits(ones_b), fmt)
        assert np.all(C3 == K), fmt
        # negation of A negates C (sign)
        C4 = o.matmul_f64(_bits(-A2), _bits(B), fmt)
        C5 = o.matmul_f64(_bits(A2), _bits(B), fmt)
        assert np.array_equal(C4, -C5), fmt


def pin_matmul_row_sample(o) -> None:
    g = gg_inputs.generator(11)
    A = gg_inputs.normal((20, 24), torch.float16, g)
    B = gg_inputs.normal((24, 9), torch.float16, g)
    full = o.matmul_f64(_bits(A), _bits(B), 0)
    rows = np.array([19, 0, 5, 5, 12])
    part = o.matmul_f64(_bits(A), _bits(B), 0, rows=rows)
    assert np.array_equal(part, full[rows])


def pin_fused_integers(o) -> None:
    """Fused form on integer-valued operands: every member's output holds the
    exact integer products of every member, in group order; nothing else
    changes."""
    g = gg_inputs.generator(13)
    for fmt, dt, npdt in ((0, torch.float16, np.float16), (1, torch.bfloat16, None)):
        H, group, M, N, K = 6, (1, 2, 3), 5, 12, 16
        W = group[2]
        members = _members(group)
        lay = hi.make_layout(H, W, M, N, 2, ld_in=K + 4, ld_out=N + 2)
        heap = hi.sentinel_heap(lay)
        A = {h: gg_inputs.integers((M, K), -2, 2, dt, g) for h in members}
        B = gg_inputs.integers((K, N), -2, 2, dt, g)
        for h in members:
            hi.put_block(heap, lay, h, _bits(A[h]), lay.in_off, lay.ld_in)
        before = heap.copy()
        prods = o.matmul_all_gather(heap, lay.part_bytes, lay.in_off, lay.ld_in, _bits(B),
                                    lay.out_off, lay.ld_out, M, N, K, fmt, group)
        Bi = B.to(torch.int64).numpy()
        for i, h in enumerate(members):
            ref = A[h].to(torch.int64).numpy() @ Bi
            assert np.array_equal(prods[i], ref.astype(np.float64))
            for d in members:
                out = hi.get_block(heap, lay, d, lay.out_off, W * M, lay.ld_out, N, np.uint16)
                blk = torch.from_numpy(out[i * M:(i + 1) * M].view(np.int16))
                val = blk.view(dt).to(torch.int64).numpy()
                assert np.array_equal(val, ref), (fmt, i, d)
        mask = hi.output_mask(lay, members)
        assert np.array_equal(heap[~mask], before[~mask])


def pin_fused_empty_contraction(o) -> None:
    """K = 0: every product is the empty sum, +0 (numpy's matmul of an M x 0 by
    a 0 x N matrix agrees), so every member's gathered output holds all-zero
    bit patterns in its data columns and nothing else changes."""
    for fmt in (0, 1):
        H, group, M, N = 5, (0, 2, 3), 7, 24
        W = group[2]
        members = _members(group)
        lay = hi.make_layout(H, W, M, N, 2, ld_in=8, ld_out=N + 8)
        heap = hi.sentinel_heap(lay)
        before = heap.copy()
        A0 = np.zeros((M, 0), dtype=np.float64)
        B = np.zeros((0, N), dtype=np.uint16)  # 0 x N, row pitch N
        prods = o.matmul_all_gather(heap, lay.part_bytes, lay.in_off, lay.ld_in, B, lay.out_off,
                                    lay.ld_out, M, N, 0, fmt, group)
        for i in range(W):
            assert np.array_equal(prods[i], A0 @ np.zeros((0, N))), (fmt, i)
            assert not np.signbit(prods[i]).any()
        for d in members:
            out = hi.get_block(heap, lay, d, lay.out_off, W * M, lay.ld_out, N, np.uint16)
            assert not out.any(), (fmt, d)
        mask = hi.output_mask(lay, members)
        assert np.array_equal(heap[~mask], before[~mask])
        # the padding columns inside the output region keep their bytes too
        assert hi.output_mask(lay, members).sum() == W * W * M * N * 2


ALL_PINS = [
    pin_group_index,
    pin_gather_packed,
    pin_gather_single_contribution,
    pin_gather_w1_copy,
    pin_all_to_all_packed,
    pin_all_to_all_twice_is_identity,
    pin_all_to_all_w1_copy,
    pin_decode16,
    pin_encode16,
    pin_matmul_numpy,
    pin_matmul_integers_exact,
    pin_matmul_closed_forms,
    pin_matmul_row_sample,
    pin_fused_integers,
    pin_fused_empty_contraction,
]
