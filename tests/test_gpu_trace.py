"""Tracing (gg_set_trace / gg_trace_read): a traced launch records its first
CTA's start and end wall time and SM cycle counter, one record per kernel
family; launches after tracing is switched off leave the records alone; the
traced launch's result is still the oracle's."""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

pytestmark = pytest.mark.gpu


def _check(rec):
    assert rec["end_ns"] > rec["start_ns"] > 0
    assert rec["end_cycles"] > rec["start_cycles"]
    assert 100.0 < rec["sm_mhz"] < 3000.0, rec  # a GB300's SM clock range, with margin


def test_trace_records_each_family(oracle):
    import gemm_gather_gb300 as gg
    H, group, M, N = 4, (0, 1, 4), 512, 2048
    lay = hi.make_layout(H, 4, M, N, 2)
    host = hi.sentinel_heap(lay)
    for h in range(H):
        hi.put_block(host, lay, h, gg_inputs.index_coded(h, M, N, 2).numpy(), lay.in_off, N)
    sh = device_heap(lay, host)
    fl = hi.make_layout(2, 2, 256, 512, 2, ld_in=256)
    fh = device_heap(fl, hi.sentinel_heap(fl))
    B = torch.zeros((256, 512), dtype=torch.float16, device="cuda")
    try:
        gg.set_trace(True)
        for path in ("tma", "bulk", "vector"):
            gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), N, sh.ptr(0, lay.out_off), N, M, N,
                          torch.float16, (8, 256), 8, group, path=path)
            _check(gg.trace_read()["all_gather"])
        gg.matmul_all_gather(fh.heap, -1, fh.ptr(0, fl.in_off), 256, B, 512, fh.ptr(0, fl.out_off),
                             512, 256, 512, 256, torch.float16, gg.FUSED_TILE_WIDE, 4, (0, 1, 2))
        rec = gg.trace_read()
        _check(rec["matmul_all_gather"])
        gg.set_trace(False)
        gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), N, sh.ptr(0, lay.out_off), N, M, N,
                      torch.float16, (8, 256), 8, group)
        gg.matmul_all_gather(fh.heap, -1, fh.ptr(0, fl.in_off), 256, B, 512, fh.ptr(0, fl.out_off),
                             512, 256, 512, 256, torch.float16, gg.FUSED_TILE_WIDE, 4, (0, 1, 2))
        assert gg.trace_read() == rec  # untraced launches leave the records alone
    finally:
        gg.set_trace(False)
    got = download(sh)
    oracle.all_gather(host, lay.part_bytes, lay.in_off, N, lay.out_off, N, M, N, 2, group)
    assert np.array_equal(got, host), first_diff(got, host, lay)
