"""Parity of the neighbouring collectives with the oracle, through the C ABI:
the partitioned all-gather (one destination per program), the grouped
all-gather (a bounded number of destination stores per wait) and the
all-to-all.  As for the all-gather, the device heap and a host image start
identical and the WHOLE heap must match byte for byte afterwards."""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

pytestmark = pytest.mark.gpu

DT = {2: torch.float16, 4: torch.float32}
NPDT = {2: np.int16, 4: np.int32}


def _tma_ok(N, pi, po, es, tile):
    return ((N + pi) * es) % 16 == 0 and ((N + po) * es) % 16 == 0 and (tile[1] * es) % 16 == 0 \
        and tile[1] <= 256


def _gather_setup(H, group, M, N, es, pi, po, seed):
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    lay = hi.make_layout(H, W, M, N, es, ld_in=N + pi, ld_out=N + po)
    host = hi.sentinel_heap(lay)
    for h in members:
        hi.put_block(host, lay, h, gg_inputs.index_coded(h * 131 + seed, M, N, es).numpy(),
                     lay.in_off, lay.ld_in)
    return lay, host, members


# (H, group, M, N, elem bytes, tile, programs, pad_in, pad_out)
PART_CASES = [
    (2, (0, 1, 2), 64, 256, 2, (8, 256), 4, 0, 0),
    (3, (0, 1, 3), 17, 40, 2, (4, 16), 5, 3, 5),
    (4, (0, 1, 4), 130, 300, 4, (32, 128), 7, 4, 12),
    (8, (1, 2, 4), 33, 264, 4, (8, 256), 16, 0, 0),
    (8, (0, 1, 8), 100, 4096, 2, (8, 256), 148, 0, 0),
    (8, (0, 1, 8), 64, 512, 2, (16, 128), 8, 0, 0),        # exactly one program per destination
    (64, (0, 1, 64), 9, 40, 2, (8, 16), 70, 0, 0),         # 64 destinations
    (40, (3, 1, 33), 5, 264, 4, (4, 64), 300, 0, 8),       # 33 destinations, more programs than SMs
]


@pytest.mark.parametrize("path", ["auto", "tma", "vector"])
@pytest.mark.parametrize("case", PART_CASES, ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}e{c[4]}p{c[6]}")
def test_partitioned_all_gather_matches_oracle(oracle, case, path):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs, pi, po = case
    if path == "tma" and not _tma_ok(N, pi, po, es, tile):
        pytest.skip("tensor-map path needs 16-byte pitches and tile rows")
    lay, host, members = _gather_setup(H, group, M, N, es, pi, po, 1)
    sh = device_heap(lay, host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.all_gather_partitioned(sh.heap, -1, sh.ptr(members[0], lay.in_off), lay.ld_in,
                              sh.ptr(members[0], lay.out_off), lay.ld_out, M, N, DT[es], tile,
                              programs, group, status=status, path=path)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


def test_partitioned_single_rank_launches(oracle):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs = 6, (1, 2, 3), 40, 512, 2, (8, 256), 9
    lay, host, members = _gather_setup(H, group, M, N, es, 0, 0, 2)
    sh = device_heap(lay, host)
    for h in members:
        gg.all_gather_partitioned(sh.heap, h, sh.ptr(h, lay.in_off), N, sh.ptr(h, lay.out_off), N,
                                  M, N, DT[es], tile, programs, group)
    got = download(sh)
    oracle.all_gather(host, lay.part_bytes, lay.in_off, N, lay.out_off, N, M, N, es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


@pytest.mark.parametrize("path", ["tma", "bulk"])
@pytest.mark.parametrize("dests_per_wait", [1, 2, 3, 5, 8])
def test_grouped_all_gather_matches_oracle(oracle, dests_per_wait, path):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs = 8, (0, 1, 8), 72, 1024, 2, (8, 256), 20
    lay, host, members = _gather_setup(H, group, M, N, es, 0, 8, 3)
    sh = device_heap(lay, host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.all_gather_grouped(sh.heap, -1, sh.ptr(0, lay.in_off), lay.ld_in, sh.ptr(0, lay.out_off),
                          lay.ld_out, M, N, DT[es], tile, programs, group, dests_per_wait,
                          status=status, path=path)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


def test_grouped_strided_subgroup(oracle):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs = 8, (1, 2, 4), 33, 264, 4, (8, 256), 16
    lay, host, members = _gather_setup(H, group, M, N, es, 0, 0, 4)
    sh = device_heap(lay, host)
    gg.all_gather_grouped(sh.heap, -1, sh.ptr(1, lay.in_off), N, sh.ptr(1, lay.out_off), N, M, N,
                          DT[es], tile, programs, group, 3)
    got = download(sh)
    oracle.all_gather(host, lay.part_bytes, lay.in_off, N, lay.out_off, N, M, N, es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


# (H, group, M, N, elem bytes, tile, programs, pad_in, pad_out); each input is W*M x N
A2A_CASES = [
    (2, (0, 1, 2), 64, 256, 2, (8, 256), 4, 0, 0),
    (3, (0, 1, 3), 17, 40, 2, (4, 16), 5, 3, 5),
    (4, (0, 1, 4), 130, 300, 4, (32, 128), 7, 4, 12),
    (8, (1, 2, 4), 33, 264, 4, (8, 256), 16, 0, 0),
    (8, (0, 1, 8), 64, 1024, 2, (8, 256), 148, 0, 0),
    (5, (2, 1, 3), 1, 1, 4, (1, 1), 2, 0, 0),
    (1, (0, 1, 1), 9, 24, 2, (8, 8), 1, 0, 0),
    (64, (0, 1, 64), 2, 40, 2, (8, 16), 37, 0, 0),         # 64 members
    (40, (3, 1, 33), 3, 264, 4, (4, 64), 300, 0, 8),       # 33 members, more programs than SMs
]


def _a2a_setup(H, group, M, N, es, pi, po, seed):
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    lay = hi.make_layout(H, W, W * M, N, es, ld_in=N + pi, ld_out=N + po)
    host = hi.sentinel_heap(lay)
    for h in members:
        hi.put_block(host, lay, h, gg_inputs.index_coded(h * 17 + seed, W * M, N, es).numpy(),
                     lay.in_off, lay.ld_in)
    return lay, host, members


@pytest.mark.parametrize("mode", ["group", "ranks", "external"])
@pytest.mark.parametrize("path", ["auto", "tma", "vector"])
@pytest.mark.parametrize("case", A2A_CASES, ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}e{c[4]}t{c[5]}")
def test_all_to_all_matches_oracle(oracle, case, path, mode):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs, pi, po = case
    if path == "tma" and not _tma_ok(N, pi, po, es, tile):
        pytest.skip("tensor-map path needs 16-byte pitches and tile rows")
    W = group[2]
    lay, host, members = _a2a_setup(H, group, M, N, es, pi, po, 5)
    sh = device_heap(lay, host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if mode == "group":
        gg.all_to_all(sh.heap, -1, sh.ptr(members[0], lay.in_off), lay.ld_in,
                      sh.ptr(members[0], lay.out_off), lay.ld_out, M, N, DT[es], tile, programs,
                      group, status=status, path=path)
    else:
        for h in members:
            if mode == "ranks":
                src = sh.ptr(h, lay.in_off)
                ld = lay.ld_in
            else:
                src = torch.from_numpy(hi.get_block(host, lay, h, lay.in_off, W * M, lay.ld_in, N,
                                                    NPDT[es])).cuda()
                ld = N
            gg.all_to_all(sh.heap, h, src, ld, sh.ptr(h, lay.out_off), lay.ld_out, M, N, DT[es],
                          tile, programs, group, status=status, path=path)
            if mode == "external":
                torch.cuda.synchronize()
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_to_all(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


def test_all_to_all_twice_restores_inputs(oracle):
    """Exchanging the outputs again gives back every member's input blocks."""
    import gemm_gather_gb300 as gg
    H, group, M, N, es = 4, (0, 1, 4), 48, 512, 2
    lay, host, members = _a2a_setup(H, group, M, N, es, 0, 0, 6)
    sh = device_heap(lay, host)
    W = group[2]
    gg.all_to_all(sh.heap, -1, sh.ptr(0, lay.in_off), N, sh.ptr(0, lay.out_off), N, M, N,
                  torch.float16, (8, 256), 12, group)
    # a second exchange from the outputs into a fresh region past the output
    back_off = lay.out_off + W * M * N * es + 4096
    assert back_off + W * M * N * es <= lay.part_bytes
    gg.all_to_all(sh.heap, -1, sh.ptr(0, lay.out_off), N, sh.ptr(0, back_off), N, M, N,
                  torch.float16, (16, 128), 12, group)
    got = download(sh)
    for h in members:
        a = hi.get_block(host, lay, h, lay.in_off, W * M, N, N, np.int16)
        b = hi.get_block(got, lay, h, back_off, W * M, N, N, np.int16)
        assert np.array_equal(a, b), h
