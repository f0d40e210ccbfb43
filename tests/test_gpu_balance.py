"""Load-balanced launches (runs of tiles claimed from a workspace counter)
against the oracle, through the C ABI.

With a workspace, tensor-map all-gathers and all-to-alls can hand tiles out in
runs claimed from a per-launch counter instead of a fixed share per pipeline.
The result must not change: every case compares the WHOLE heap with the
oracle, byte for byte, with and without a workspace, for the all-gather (all
at once and grouped), the partitioned all-gather and the all-to-all, on the
tensor-map and bulk paths.  The cases have few programs and many tiles, so
that every pipeline claims several runs under the "always" policy; the
counters left in the workspace show which launches claimed.
"""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

pytestmark = pytest.mark.gpu

DT = {2: torch.float16, 4: torch.float32}
SLOT_WORDS = 128 // 8


@pytest.fixture(autouse=True)
def claim_always():
    """These cases are small: let every tensor-map launch claim runs."""
    import gemm_gather_gb300 as gg
    gg.set_claim_policy("always")
    yield
    gg.set_claim_policy("auto")


def _setup(H, group, rows_in, N, es, seed, slots, pad=(0, 0)):
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    lay = hi.make_layout(H, W, rows_in, N, es, ld_in=N + pad[0], ld_out=N + pad[1])
    host = hi.sentinel_heap(lay)
    for h in members:
        hi.put_block(host, lay, h, gg_inputs.index_coded(h * 313 + seed, rows_in, N, es).numpy(),
                     lay.in_off, lay.ld_in)
    return lay, host, members, device_heap(lay, host, workspace_slots=slots)


def _counter(sh, slot):
    return int(sh.workspace.view(torch.int64)[slot * SLOT_WORDS].item())


def _items(M, N, tile, sources):
    return -(-M // tile[0]) * -(-N // tile[1]) * sources


# (H, group, M, N, elem bytes, tile, programs, pads)
CASES = [
    (4, (0, 1, 4), 256, 1024, 2, (8, 256), 1, (0, 0)),
    (4, (0, 1, 4), 256, 1024, 2, (8, 256), 3, (0, 0)),
    (8, (0, 1, 8), 192, 520, 2, (8, 128), 5, (8, 24)),      # ragged columns, padded pitches
    (6, (1, 2, 3), 203, 264, 4, (16, 64), 2, (4, 0)),       # strided group, ragged rows
    (8, (0, 1, 8), 512, 2048, 4, (32, 128), 8, (0, 0)),
]
IDS = [f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}e{c[4]}t{c[5]}p{c[6]}" for c in CASES]


@pytest.mark.parametrize("slots", [64, 0], ids=["workspace", "none"])
@pytest.mark.parametrize("path", ["tma", "bulk"])
@pytest.mark.parametrize("dests_per_wait", [0, 3])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_all_gather_balanced(oracle, case, path, dests_per_wait, slots):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs, pad = case
    if path == "bulk" and ((N + pad[0]) * es % 16 or (N + pad[1]) * es % 16 or N * es % 16):
        pytest.skip("bulk copies need 16-byte rows and pitches")
    lay, host, members, sh = _setup(H, group, M, N, es, 1, slots, pad)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (sh.heap, -1, sh.ptr(members[0], lay.in_off), lay.ld_in,
            sh.ptr(members[0], lay.out_off), lay.ld_out, M, N, DT[es], tile, programs, group)
    if dests_per_wait:
        gg.all_gather_grouped(*args, dests_per_wait, status=status, path=path)
    else:
        gg.all_gather(*args, status=status, path=path)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)
    if slots:  # tensor maps claimed from slot 0; bulk copies keep fixed shares
        assert (_counter(sh, 0) > 0) == (path == "tma")


@pytest.mark.parametrize("slots", [64, 0], ids=["workspace", "none"])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_partitioned_balanced(oracle, case, slots):
    """The partitioned all-gather keeps fixed shares with or without a workspace."""
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs, pad = case
    W = group[2]
    programs = max(programs, W)  # at least one program per destination
    lay, host, members, sh = _setup(H, group, M, N, es, 2, slots, pad)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.all_gather_partitioned(sh.heap, -1, sh.ptr(members[0], lay.in_off), lay.ld_in,
                              sh.ptr(members[0], lay.out_off), lay.ld_out, M, N, DT[es], tile,
                              programs, group, status=status, path="tma")
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)
    if slots:
        assert _counter(sh, 0) == 0


@pytest.mark.parametrize("slots", [64, 0], ids=["workspace", "none"])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_all_to_all_balanced(oracle, case, slots):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs, pad = case
    W = group[2]
    Mb = max(M // W, 1)
    lay, host, members, sh = _setup(H, group, W * Mb, N, es, 3, slots, pad)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.all_to_all(sh.heap, -1, sh.ptr(members[0], lay.in_off), lay.ld_in,
                  sh.ptr(members[0], lay.out_off), lay.ld_out, Mb, N, DT[es], tile, programs, group,
                  status=status, path="tma")
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_to_all(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, Mb, N,
                      es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)
    if slots:
        assert _counter(sh, 0) > 0


def test_slot_use():
    """A claiming launch takes the next slot and leaves its counter above zero
    and below the number of tiles; launches that keep fixed shares (bulk
    path, partitioned all-gather) take no slot."""
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile = 4, (0, 1, 4), 512, 2048, 2, (8, 256)
    lay, host, members, sh = _setup(H, group, M, N, es, 4, 64)
    total = _items(M, N, tile, 4)
    args = (sh.heap, -1, sh.ptr(0, lay.in_off), N, sh.ptr(0, lay.out_off), N, M, N, DT[es], tile)
    gg.all_gather(*args, 2, group, path="tma")           # slot 0
    gg.all_gather(*args, 2, group, path="bulk")          # no slot
    gg.all_gather_partitioned(*args, 4, group, path="tma")  # no slot
    gg.all_gather(*args, 3, group, path="tma")           # slot 1
    torch.cuda.synchronize()
    assert 0 < _counter(sh, 0) < total
    assert 0 < _counter(sh, 1) < total
    assert _counter(sh, 2) == 0


def test_slots_are_reused_round_robin(oracle):
    """More launches than slots, back to back on one stream (each launch
    zeroes its slot first): every result equals the oracle's."""
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile = 4, (0, 1, 4), 128, 1024, 2, (8, 256)
    lay, host, members, sh = _setup(H, group, M, N, es, 5, 3)
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      es, group)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(10):
        sh.partition(0)[lay.out_off: lay.out_off + 4 * M * N * es].fill_(0)
        gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), N, sh.ptr(0, lay.out_off), N, M, N,
                      DT[es], tile, 1 + i % 3, group, status=status, path="tma")
        got = download(sh)
        assert int(status.item()) == 0
        assert np.array_equal(got, host), (i, first_diff(got, host, lay))


@pytest.mark.parametrize("policy", ["auto", "never"])
def test_policy_keeps_fixed_shares(oracle, policy):
    """A small launch over two programs: "auto" keeps fixed shares (too few
    bytes, too few SMs), so does "never"; the slot stays zero."""
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile = 4, (0, 1, 4), 512, 2048, 2, (8, 256)
    lay, host, members, sh = _setup(H, group, M, N, es, 6, 64)
    gg.set_claim_policy(policy)
    gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), N, sh.ptr(0, lay.out_off), N, M, N, DT[es],
                  tile, 2, group, path="tma")
    got = download(sh)
    assert _counter(sh, 0) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, N, lay.out_off, N, M, N, es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


def test_concurrent_launches_on_several_streams(oracle):
    """Five launches in flight at once on five streams, into disjoint output
    regions of one heap: two claiming tensor-map all-gathers (each takes its
    own workspace slot), a grouped bulk all-gather, a partitioned all-gather on
    the vector path and a claiming all-to-all; plus a fused matmul +
    all-gather on a sixth stream into a second heap.  Each region must hold
    the oracle's result and nothing else may change, as if the launches had
    run one after another; every status word stays 0."""
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile = 4, (0, 1, 4), 256, 2048, 2, (8, 256)
    W = group[2]
    base = hi.make_layout(H, W, W * M, N, es)            # inputs hold W*M rows (all-to-all)
    region = -(-(W * M * N * es + hi.GUARD) // 4096) * 4096   # one gathered output + guard
    part = base.out_off + 5 * region
    lay = hi.Layout(H, part, base.in_off, N, base.out_off, N, M, N, W, es)
    host = np.full(H * part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
    for h in range(H):
        hi.put_block(host, lay, h, gg_inputs.index_coded(h * 97 + 11, W * M, N, es).numpy(),
                     lay.in_off, N)
    sh = device_heap(lay, host, workspace_slots=8)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(5)]
    status = torch.zeros(5, dtype=torch.int32, device="cuda")
    out = [lay.out_off + j * region for j in range(5)]
    inp = sh.ptr(0, lay.in_off)
    calls = [
        lambda s, st: gg.all_gather(sh.heap, -1, inp, N, sh.ptr(0, out[0]), N, M, N, DT[es], tile,
                                    3, group, status=st, stream=s, path="tma"),
        lambda s, st: gg.all_gather(sh.heap, -1, inp, N, sh.ptr(0, out[1]), N, M, N, DT[es], tile,
                                    5, group, status=st, stream=s, path="tma"),
        lambda s, st: gg.all_gather_grouped(sh.heap, -1, inp, N, sh.ptr(0, out[2]), N, M, N,
                                            DT[es], tile, 4, group, 2, status=st, stream=s,
                                            path="bulk"),
        lambda s, st: gg.all_gather_partitioned(sh.heap, -1, inp, N, sh.ptr(0, out[3]), N, M, N,
                                                DT[es], (16, 128), 8, group, status=st, stream=s,
                                                path="vector"),
        lambda s, st: gg.all_to_all(sh.heap, -1, inp, N, sh.ptr(0, out[4]), N, M, N, DT[es],
                                    tile, 3, group, status=st, stream=s, path="tma"),
    ]
    # and a fused matmul + all-gather (integer operands: exact) on a sixth stream,
    # into a heap of its own
    fW, fM, fN, fK = 2, 256, 512, 128
    fl = hi.make_layout(fW, fW, fM, fN, 2, ld_in=fK)
    fhost = hi.sentinel_heap(fl)
    fgen = gg_inputs.generator(5)
    for h in range(fW):
        a = gg_inputs.integers((fM, fK), -2, 2, torch.float16, fgen)
        hi.put_block(fhost, fl, h, a.view(torch.int16).numpy().view(np.uint16), fl.in_off, fK)
    fB = gg_inputs.integers((fK, fN), -2, 2, torch.float16, fgen)
    fh = device_heap(fl, fhost)
    fB_dev = fB.to("cuda")
    fstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    fstream = torch.cuda.Stream()
    for s, call, st in zip(streams, calls, status):
        call(s, st)
    gg.matmul_all_gather(fh.heap, -1, fh.ptr(0, fl.in_off), fK, fB_dev, fN, fh.ptr(0, fl.out_off),
                         fN, fM, fN, fK, torch.float16, gg.FUSED_TILE_WIDE, 8, (0, 1, fW),
                         status=fstatus, stream=fstream)
    got = download(sh)
    fgot = download(fh)
    assert status.tolist() == [0] * 5 and int(fstatus.item()) == 0
    oracle.matmul_all_gather(fhost, fl.part_bytes, fl.in_off, fK,
                             fB.view(torch.int16).numpy().view(np.uint16), fl.out_off, fN, fM, fN,
                             fK, 0, (0, 1, fW))
    assert np.array_equal(fgot, fhost), first_diff(fgot, fhost, fl)
    for j in range(4):
        oracle.all_gather(host, part, lay.in_off, N, out[j], N, M, N, es, group)
    oracle.all_to_all(host, part, lay.in_off, N, out[4], N, M, N, es, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)
    assert _counter(sh, 0) > 0 and _counter(sh, 1) > 0 and _counter(sh, 2) > 0
