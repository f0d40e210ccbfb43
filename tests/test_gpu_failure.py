"""Bounded waits on the GPU.  With the stall hook on, program 0 of a launch
leaves one ring stage unarmed, so the wait on it is a wait on a flag that
nothing sets: it runs out after the (shortened) wait limit, the kernel stores
GG_ERR_TIMEOUT in the status word, drains its copies in flight and returns.
The context stays usable: a normal launch right after gives the oracle's
result.  Nothing here faults, traps or hangs the GPU."""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

pytestmark = pytest.mark.gpu

TIMEOUT = -6


@pytest.fixture
def short_waits():
    import gemm_gather_gb300 as gg
    gg.set_wait_limit_ns(20_000_000)
    gg.debug_inject_stall(True)
    yield
    gg.debug_inject_stall(False)
    gg.set_wait_limit_ns(0)  # back to the default


def _gather_heap():
    lay = hi.make_layout(4, 4, 512, 4096, 2)
    host = hi.sentinel_heap(lay)
    for h in range(4):
        hi.put_block(host, lay, h, gg_inputs.index_coded(h, 512, 4096, 2).numpy(), lay.in_off,
                     lay.ld_in)
    return lay, host


@pytest.mark.parametrize("path", ["bulk", "tma"])
def test_gather_wait_limit_reports_timeout(oracle, short_waits, path):
    import gemm_gather_gb300 as gg
    lay, host = _gather_heap()
    sh = device_heap(lay, host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.clear_device_status()
    gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), lay.ld_in, sh.ptr(0, lay.out_off),
                  lay.ld_out, lay.M, lay.N, torch.float16, (8, 256), 4, (0, 1, 4),
                  status=status, path=path)
    torch.cuda.synchronize()
    assert int(status.item()) == TIMEOUT
    assert gg.device_status() == 0  # the caller's word got it; the library's stays clear
    # the context is intact: a normal launch gives the oracle's heap
    gg.debug_inject_stall(False)
    gg.set_wait_limit_ns(0)
    status.zero_()
    gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), lay.ld_in, sh.ptr(0, lay.out_off),
                  lay.ld_out, lay.M, lay.N, torch.float16, (8, 256), 4, (0, 1, 4),
                  status=status, path=path)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out,
                      lay.M, lay.N, 2, (0, 1, 4))
    assert np.array_equal(got, host), first_diff(got, host, lay)


@pytest.mark.parametrize("path", ["1sm", "2sm", "wide"])
def test_fused_wait_limit_reports_timeout(oracle, short_waits, path):
    import gemm_gather_gb300 as gg
    from tests.test_gpu_fused import kernel_args
    path, tile = kernel_args(path)
    W, M, N, K = 2, 512, 1024, 2048
    lay = hi.make_layout(W, W, M, N, 2, ld_in=K)
    host = hi.sentinel_heap(lay)
    gen = gg_inputs.generator(1)
    for h in range(W):
        a = gg_inputs.integers((M, K), -2, 2, torch.float16, gen)
        hi.put_block(host, lay, h, a.view(torch.int16).numpy(), lay.in_off, K)
    B = gg_inputs.integers((K, N), -2, 2, torch.float16, gen)
    sh = device_heap(lay, host)
    Bd = B.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.clear_device_status()
    gg.matmul_all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), K, Bd, N, sh.ptr(0, lay.out_off), N,
                         M, N, K, torch.float16, tile, 8, (0, 1, W), status=status,
                         path=path)
    torch.cuda.synchronize()
    assert int(status.item()) == TIMEOUT
    assert gg.device_status() == 0  # the caller's word got it; the library's stays clear
    gg.debug_inject_stall(False)
    gg.set_wait_limit_ns(0)
    status.zero_()
    gg.matmul_all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), K, Bd, N, sh.ptr(0, lay.out_off), N,
                         M, N, K, torch.float16, tile, 8, (0, 1, W), status=status,
                         path=path)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.matmul_all_gather(host, lay.part_bytes, lay.in_off, K,
                             B.view(torch.int16).numpy().view(np.uint16), lay.out_off, N, M, N, K,
                             0, (0, 1, W))
    assert np.array_equal(got, host), first_diff(got, host, lay)


@pytest.mark.parametrize("kind", ["bulk", "tma", "1sm", "2sm", "wide"])
def test_timeout_without_status_word_is_reported(oracle, short_waits, kind):
    """A launch given no status word (NULL) reports a wait that gave up in the
    library's status word of the device: no early stop goes unreported.  After
    clearing it, the same launch runs normally, leaves the word at 0 and gives
    the oracle's heap."""
    import gemm_gather_gb300 as gg
    from tests.test_gpu_fused import kernel_args
    fused = kind in ("1sm", "2sm", "wide")
    path, tile = kernel_args(kind) if fused else (kind, None)
    if fused:
        W, M, N, K = 2, 512, 1024, 2048
        lay = hi.make_layout(W, W, M, N, 2, ld_in=K)
        host = hi.sentinel_heap(lay)
        gen = gg_inputs.generator(2)
        for h in range(W):
            a = gg_inputs.integers((M, K), -2, 2, torch.float16, gen)
            hi.put_block(host, lay, h, a.view(torch.int16).numpy(), lay.in_off, K)
        B = gg_inputs.integers((K, N), -2, 2, torch.float16, gen)
        Bd = B.to("cuda")
    else:
        lay, host = _gather_heap()
    sh = device_heap(lay, host)

    def launch():
        if fused:
            gg.matmul_all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), K, Bd, N,
                                 sh.ptr(0, lay.out_off), N, M, N, K, torch.float16,
                                 tile, 8, (0, 1, W), status=None, path=path)
        else:
            gg.all_gather(sh.heap, -1, sh.ptr(0, lay.in_off), lay.ld_in, sh.ptr(0, lay.out_off),
                          lay.ld_out, lay.M, lay.N, torch.float16, (8, 256), 4, (0, 1, 4),
                          status=None, path=path)

    gg.clear_device_status()
    assert gg.device_status() == 0
    launch()
    assert gg.device_status() == TIMEOUT
    gg.debug_inject_stall(False)
    gg.set_wait_limit_ns(0)
    gg.clear_device_status()
    assert gg.device_status() == 0
    launch()
    got = download(sh)
    assert gg.device_status() == 0
    if fused:
        oracle.matmul_all_gather(host, lay.part_bytes, lay.in_off, K,
                                 B.view(torch.int16).numpy().view(np.uint16), lay.out_off, N, M,
                                 N, K, 0, (0, 1, W))
    else:
        oracle.all_gather(host, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out,
                          lay.M, lay.N, 2, (0, 1, 4))
    assert np.array_equal(got, host), first_diff(got, host, lay)
