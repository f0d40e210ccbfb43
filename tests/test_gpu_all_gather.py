"""Parity of the CUDA all-gather with the oracle, through the C ABI.

Every case builds the same heap image on the host and on the device (sentinel
everywhere, inputs in each member's partition), runs the kernel on the device
and the oracle on the host, and compares the WHOLE heap byte for byte:
gathered blocks, padding columns, guard bands, inputs and inactive heaps
(iris #594, "Local validation").  Bit-exact is the bar (a gather is a copy).
"""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

pytestmark = pytest.mark.gpu

DT = {2: torch.float16, 4: torch.float32}


def _fill_inputs(heap, lay, members, seed, packed):
    for h in members:
        if packed:
            blk = gg_inputs.index_packed(h, lay.M, lay.N, lay.esize).numpy()
        else:
            blk = gg_inputs.index_coded(h * 7919 + seed, lay.M, lay.N, lay.esize).numpy()
        hi.put_block(heap, lay, h, blk, lay.in_off, lay.ld_in)


def _run_case(oracle, H, group, M, N, es, tile, programs, pad_in=0, pad_out=0, path="auto",
              extra_in=0, extra_out=0, mode="group", seed=0):
    import gemm_gather_gb300 as gg
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    lay = hi.make_layout(H, W, M, N, es, ld_in=N + pad_in, ld_out=N + pad_out,
                         extra_in=extra_in, extra_out=extra_out)
    host = hi.sentinel_heap(lay)
    packed = (es == 2 and H <= 4 and M <= 32 and N <= 512) or (es == 4 and M <= 4096 and N <= 4096)
    _fill_inputs(host, lay, members, seed, packed)
    sh = device_heap(lay, host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dt = DT[es]
    if mode == "group":
        gg.all_gather(sh.heap, -1, sh.ptr(members[0], lay.in_off), lay.ld_in,
                      sh.ptr(members[-1], lay.out_off), lay.ld_out, M, N, dt, tile, programs,
                      group, status=status, path=path)
    elif mode == "ranks":
        # the pages' single-GPU validation: one launch per logical rank, in turn
        for h in members:
            gg.all_gather(sh.heap, h, sh.ptr(h, lay.in_off), lay.ld_in, sh.ptr(h, lay.out_off),
                          lay.ld_out, M, N, dt, tile, programs, group, status=status, path=path)
    elif mode == "external":
        # single-rank calls whose input lives outside the heap
        for h in members:
            npdt = {2: np.int16, 4: np.int32}[es]
            ext = torch.from_numpy(hi.get_block(host, lay, h, lay.in_off, M, lay.ld_in, N, npdt))
            ext = ext.to("cuda")
            gg.all_gather(sh.heap, h, ext, N, sh.ptr(h, lay.out_off), lay.ld_out, M, N, dt, tile,
                          programs, group, status=status, path=path)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


# (H, group, M, N, elem bytes, tile, programs, pad_in, pad_out)
CASES = [
    (2, (0, 1, 2), 64, 256, 2, (8, 256), 4, 0, 0),           # 2-rank 64x256 f16, 8x256 tile
    (1, (0, 1, 1), 5, 7, 2, (8, 256), 1, 0, 0),              # W = 1, partial tile
    (3, (0, 1, 3), 17, 40, 2, (4, 16), 5, 3, 5),             # ragged rows and columns
    (4, (0, 1, 4), 32, 512, 2, (16, 128), 148, 0, 8),        # more programs than items
    (4, (0, 1, 4), 130, 300, 4, (32, 128), 7, 4, 12),        # f32, ragged tails, padding
    (8, (1, 2, 4), 33, 264, 4, (8, 256), 16, 0, 0),          # strided subgroup, inactive heaps
    (8, (0, 2, 4), 64, 1000, 2, (8, 256), 9, 8, 0),          # strided subgroup from heap 0
    (8, (0, 1, 8), 257, 513, 2, (32, 64), 64, 7, 9),         # explicit 32x64 runs as 32x64
    (5, (2, 1, 3), 1, 1, 4, (1, 1), 2, 0, 0),                # 1 x 1 blocks
    (8, (0, 1, 8), 100, 4096, 2, (8, 256), 148, 0, 0),       # several waves of work items
    (4, (0, 1, 4), 64, 2048, 4, (256, 32), 3, 0, 0),         # tall tile, few programs
    (64, (0, 1, 64), 9, 40, 2, (8, 16), 37, 0, 0),           # 64 ranks: stores wrap the lanes
    (40, (3, 1, 33), 5, 264, 4, (4, 64), 20, 0, 8),          # 33 ranks from heap 3
    (8, (0, 1, 8), 64, 1024, 2, (8, 256), 400, 0, 0),        # more programs than SMs
]


@pytest.mark.parametrize("path", ["auto", "tma", "bulk", "vector"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}e{c[4]}t{c[5]}p{c[6]}")
def test_group_launch_matches_oracle(oracle, case, path):
    H, group, M, N, es, tile, programs, pi, po = case
    pitches_ok = ((N + pi) * es) % 16 == 0 and ((N + po) * es) % 16 == 0 \
        and (tile[1] * es) % 16 == 0
    if path == "bulk" and not (pitches_ok and (N * es) % 16 == 0):
        pytest.skip("bulk path needs 16-byte rows and tiles")
    if path == "tma" and not (pitches_ok and tile[1] <= 256):
        pytest.skip("tensor-map path needs 16-byte pitches and tile rows")
    _run_case(oracle, H, group, M, N, es, tile, programs, pi, po, path=path)


@pytest.mark.parametrize("path", ["auto", "bulk"])
@pytest.mark.parametrize("case", CASES[:8], ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}")
def test_single_rank_launches_match_oracle(oracle, case, path):
    H, group, M, N, es, tile, programs, pi, po = case
    if path == "bulk" and not (((N + pi) * es) % 16 == 0 and ((N + po) * es) % 16 == 0
                               and (tile[1] * es) % 16 == 0 and (N * es) % 16 == 0):
        pytest.skip("bulk path needs 16-byte rows and tiles")
    _run_case(oracle, H, group, M, N, es, tile, programs, pi, po, mode="ranks", path=path)


@pytest.mark.parametrize("case", CASES[:4], ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}")
def test_external_input_matches_oracle(oracle, case):
    H, group, M, N, es, tile, programs, pi, po = case
    _run_case(oracle, H, group, M, N, es, tile, programs, pi, po, mode="external")


@pytest.mark.parametrize("extra_in,extra_out,es", [(2, 0, 2), (0, 2, 2), (4, 8, 2), (8, 4, 4),
                                                   (4, 0, 4), (2, 6, 2)])
def test_misaligned_buffers_take_vector_path(oracle, extra_in, extra_out, es):
    import gemm_gather_gb300 as gg
    lay = hi.make_layout(4, 4, 9, 40, es, extra_in=extra_in, extra_out=extra_out)
    h = gg.heap_wrap(1 << 32, lay.part_bytes, 4, 1 << 33)
    chosen = gg.all_gather_check(h, -1, (1 << 32) + lay.in_off, 40, (1 << 32) + lay.out_off, 40,
                                 9, 40, DT[es], (8, 32), 4, (0, 1, 4))
    assert chosen == "vector"
    _run_case(oracle, 4, (0, 1, 4), 9, 40, es, (8, 32), 4, extra_in=extra_in,
              extra_out=extra_out)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_dtype_bits_copied_exactly(oracle, dtype):
    """Values including NaN payloads, infinities, -0 and subnormals survive."""
    import gemm_gather_gb300 as gg
    es = torch.empty((), dtype=dtype).element_size()
    M, N, W = 16, 64, 3
    lay = hi.make_layout(W, W, M, N, es)
    host = hi.sentinel_heap(lay)
    rng = np.random.default_rng(5)
    npdt = {2: np.uint16, 4: np.uint32}[es]
    for h in range(W):
        bits = rng.integers(0, 1 << (8 * es), size=(M, N), dtype=np.uint64).astype(npdt)
        hi.put_block(host, lay, h, bits, lay.in_off, lay.ld_in)
    sh = device_heap(lay, host)
    gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), N, sh.ptr(0, lay.out_off), N, M, N, dtype,
                  (8, 64), 4, (0, 1, W))
    got = download(sh)
    oracle.all_gather(host, lay.part_bytes, lay.in_off, N, lay.out_off, N, M, N, es, (0, 1, W))
    assert np.array_equal(got, host), first_diff(got, host, lay)


def test_empty_inputs_launch_nothing():
    import gemm_gather_gb300 as gg
    lay = hi.make_layout(2, 2, 4, 16, 2)
    host = hi.sentinel_heap(lay)
    sh = device_heap(lay, host)
    for M, N in [(0, 16), (4, 0), (0, 0)]:
        gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), 16, sh.ptr(0, lay.out_off), 16, M, N,
                      torch.float16, (8, 256), 4, (0, 1, 2))
    assert np.array_equal(download(sh), host)


def test_repeated_launches_are_idempotent(oracle):
    """Launching the same gather twice leaves the same heap (no state carried)."""
    _run_case(oracle, 4, (0, 1, 4), 48, 512, 2, (8, 256), 8)
    _run_case(oracle, 4, (0, 1, 4), 48, 512, 2, (8, 256), 8, seed=3)


def test_binding_uses_torch_current_stream():
    """With no stream given, the binding launches on torch's current stream of
    the current device (the raw handle torch.cuda.current_stream() wraps)."""
    from gemm_gather_gb300 import _stream
    torch.cuda.init()
    s = torch.cuda.Stream()
    assert _stream(None) == (torch.cuda.current_stream().cuda_stream or None)
    with torch.cuda.stream(s):
        assert _stream(None) == s.cuda_stream
    assert _stream(s) == s.cuda_stream


@pytest.fixture
def plain_stores():
    """Every other test runs with the library's default hint (evict_first);
    these run the plain stores."""
    import gemm_gather_gb300 as gg
    gg.set_store_policy("plain")
    yield
    gg.set_store_policy("evict_first")


@pytest.mark.parametrize("path", ["tma", "bulk", "vector"])
@pytest.mark.parametrize("mode", ["group", "ranks"])
def test_store_policy_plain_changes_no_byte(oracle, plain_stores, path, mode):
    """Plain stores (no L2 hint, gg_set_store_policy) leave the whole heap
    exactly as the oracle's: ragged tiles, padded pitches, a strided subgroup
    with inactive heaps."""
    _run_case(oracle, 8, (1, 2, 3), 72, 520, 2, (16, 128), 7, pad_in=8, pad_out=24, path=path,
              mode=mode)
    _run_case(oracle, 4, (0, 1, 4), 256, 1024, 4, (8, 256), 148, path=path, mode=mode, seed=2)


def test_store_policy_collectives(oracle, plain_stores):
    """The partitioned all-gather, the grouped all-gather and the all-to-all
    with plain stores: the result is unchanged."""
    from tests.test_gpu_collectives import (PART_CASES, test_all_to_all_matches_oracle,
                                            test_grouped_all_gather_matches_oracle,
                                            test_partitioned_all_gather_matches_oracle)
    test_partitioned_all_gather_matches_oracle(oracle, PART_CASES[3], "tma")
    test_grouped_all_gather_matches_oracle(oracle, 3, "tma")
    test_grouped_all_gather_matches_oracle(oracle, 2, "bulk")
    from tests.test_gpu_collectives import A2A_CASES
    test_all_to_all_matches_oracle(oracle, A2A_CASES[3], "tma", "group")
