"""The checked build's device-side table check, on a planted fault of the
input (a wrong entry in the device heap-bases table), never of a kernel.

The planted entry always points inside the test's own heap allocation: at
another member's partition, at an unused partition, or a few bytes into the
member's own partition.  A launch that used the entry would therefore still
stay inside the allocation; the checked build must instead report
GG_ERR_NOT_IN_HEAP and reach the member at its partition's address, so that
the whole heap still matches the oracle byte for byte.

These tests need libgemm_gather_checked.so loaded (GEMM_GATHER_CHECKED=1 at
import); test_gpu_checked_build.py runs them in a child process that sets it.
In a run of the release build they are skipped."""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

import gemm_gather_gb300 as gg
from gemm_gather_gb300 import _lib

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not gg.checked_build(),
                       reason="needs the checked build (run by test_gpu_checked_build.py)"),
]

DT = {2: torch.float16, 4: torch.float32}
H, GROUP = 5, (0, 1, 4)   # members 0..3; partition 4 is in no group


def _plant(sh, kind):
    """Overwrite one device table entry; returns the heap index planted."""
    part = sh.part_bytes
    if kind == "unused_partition":
        sh.table[1] = sh.base + 4 * part
        return 1
    if kind == "other_member":
        sh.table[2] = sh.base + 0 * part
        return 2
    if kind == "shifted":
        sh.table[3] = sh.base + 3 * part + 256
        return 3
    raise ValueError(kind)


def _setup(kind_of_call, M, N, es, pi, po, seed):
    start, stride, W = GROUP
    members = [start + i * stride for i in range(W)]
    rows_in = W * M if kind_of_call == "all_to_all" else M
    lay = hi.make_layout(H, W, rows_in, N, es, ld_in=N + pi, ld_out=N + po)
    # the all-to-all output holds W blocks of M rows: the layout above is
    # sized for W * rows_in rows, which covers it
    host = hi.sentinel_heap(lay)
    for h in members:
        hi.put_block(host, lay, h, gg_inputs.index_coded(h * 71 + seed, rows_in, N, es).numpy(),
                     lay.in_off, lay.ld_in)
    return lay, host, members


CALLS = [
    # (collective, path, M, N, elem bytes, tile, programs, pad_in, pad_out)
    ("all_gather", "bulk", 40, 264, 2, (8, 256), 6, 0, 0),
    ("all_gather", "vector", 33, 100, 2, (8, 64), 5, 3, 1),
    ("all_gather", "tma", 64, 512, 4, (16, 128), 9, 0, 4),
    ("all_gather_partitioned", "vector", 17, 40, 2, (4, 16), 8, 0, 0),
    ("all_gather_partitioned", "tma", 64, 256, 2, (8, 256), 8, 0, 0),
    ("all_to_all", "vector", 9, 24, 4, (8, 8), 5, 1, 0),
    ("all_to_all", "tma", 16, 256, 2, (8, 128), 7, 0, 0),
]


@pytest.mark.parametrize("planted", ["unused_partition", "other_member", "shifted"])
@pytest.mark.parametrize("call", CALLS, ids=lambda c: f"{c[0]}_{c[1]}_{c[2]}x{c[3]}e{c[4]}")
def test_wrong_table_entry_is_reported_and_not_used(oracle, call, planted):
    coll, path, M, N, es, tile, programs, pi, po = call
    lay, host, members = _setup(coll, M, N, es, pi, po, 3)
    sh = device_heap(lay, host, workspace_slots=0)
    _plant(sh, planted)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = {"all_gather": gg.all_gather, "all_gather_partitioned": gg.all_gather_partitioned,
          "all_to_all": gg.all_to_all}[coll]
    fn(sh.heap, -1, sh.ptr(0, lay.in_off), lay.ld_in, sh.ptr(0, lay.out_off), lay.ld_out, M, N,
       DT[es], tile, programs, GROUP, status=status, path=path)
    got = download(sh)
    assert int(status.item()) == _lib.GG_ERR_NOT_IN_HEAP
    if coll == "all_to_all":
        oracle.all_to_all(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M,
                          N, es, GROUP)
    else:
        oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out,
                          M, N, es, GROUP)
    assert np.array_equal(got, host), first_diff(got, host, lay)


def test_correct_table_reports_nothing(oracle):
    lay, host, members = _setup("all_gather", 40, 264, 2, 0, 0, 4)
    sh = device_heap(lay, host, workspace_slots=0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), lay.ld_in, sh.ptr(0, lay.out_off),
                  lay.ld_out, 40, 264, torch.float16, (8, 256), 6, GROUP, status=status)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, 40,
                      264, 2, GROUP)
    assert np.array_equal(got, host), first_diff(got, host, lay)


def test_library_word_receives_the_report_without_a_status_word(oracle):
    lay, host, members = _setup("all_gather", 33, 100, 2, 3, 1, 5)
    sh = device_heap(lay, host, workspace_slots=0)
    _plant(sh, "shifted")
    gg.clear_device_status()
    gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), lay.ld_in, sh.ptr(0, lay.out_off),
                  lay.ld_out, 33, 100, torch.float16, (8, 64), 5, GROUP)
    assert gg.device_status() == _lib.GG_ERR_NOT_IN_HEAP
    gg.clear_device_status()
    assert gg.device_status() == 0
    got = download(sh)
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, 33,
                      100, 2, GROUP)
    assert np.array_equal(got, host), first_diff(got, host, lay)
