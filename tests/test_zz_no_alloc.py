"""The allocation-free all-gather (gg_all_gather_noalloc) against the
ordinary entry point and the oracle, through the C ABI.

gg_all_gather_noalloc exists for callers that cannot allocate device memory
once running (a plugin inside a framework that owns the device memory, a
real-time loop that may not synchronize on an allocation): when it claims
runs of tiles, its counter lives in a small static device array of the
library instead of a heap workspace the caller would have to allocate.

Each case gathers the same inputs twice in a row with the new call.  After
each call
* every member's output equals gg_all_gather's, byte for byte (a gather is a
  copy, so the bar is bit-exact);
* the whole heap equals the oracle's image (small cases): outputs, inputs,
  guard bands, padding and inactive heaps; at the benchmark's 4096x4096 size,
  every block equals its source on the GPU, every guard byte keeps its
  sentinel, and sampled rows match the oracle.
The second call starts from the counter the first one left behind in the
shared array: it only matches if the call clears it first.  That proves
something only if the launch claims runs, so every claiming case is sized
well above the claim threshold, and the ordinary call on the same arguments
(same claim rule, but counting in the heap's one-slot workspace) shows that
the launch claimed.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import download, first_diff

pytestmark = pytest.mark.gpu

DT = {2: torch.float16, 4: torch.float32}


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view({2: torch.int16, 4: torch.int32}[t.element_size()])


def _heap(H, part):
    import gemm_gather_gb300 as gg
    # one workspace slot: only the ordinary call uses it (the new call never does)
    return gg.SymmetricHeap(H, part, device="cuda", fill=gg_inputs.SENTINEL_BYTE,
                            workspace_slots=1)


def _counter(sh) -> int:
    return int(sh.workspace.view(torch.int64)[0].item())


# (H, group, M, N, elem bytes, tile, programs, claim policy, input misalignment
#  in elements, claims expected)
CASES = [
    (4, (0, 1, 4), 512, 2048, 2, (8, 256), 2, "always", 0, True),
    (3, (0, 1, 3), 1000, 520, 4, (16, 64), 5, "always", 0, True),    # ragged tiles
    (7, (1, 2, 3), 600, 1024, 2, (8, 128), 6, "always", 0, True),    # strided: inactive heaps
    (4, (0, 1, 4), 64, 256, 2, (8, 256), 4, "auto", 1, False),       # unaligned: vector path
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}_e{c[4]}_"
                         f"t{c[5][0]}x{c[5][1]}_p{c[6]}_{c[7]}_mis{c[8]}")
def test_noalloc_matches_all_gather_and_oracle_twice(oracle, case):
    import gemm_gather_gb300 as gg
    H, group, M, N, es, tile, programs, policy, mis, claims = case
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    dt = DT[es]
    # out_a: the ordinary call; out_b: the new one (same layout, further on)
    lay = hi.make_layout(H, W, M, N, es, extra_in=mis * es)
    out_b = lay.out_off + (lay.out_bytes + 2 * hi.GUARD) // 256 * 256 + 256
    part = (out_b + lay.out_bytes + hi.GUARD + 4095) // 4096 * 4096
    lay_b = hi.Layout(H, part, lay.in_off, N, out_b, N, M, N, W, es)
    lay_a = hi.Layout(H, part, lay.in_off, N, lay.out_off, N, M, N, W, es)
    host = np.full(H * part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
    for h in members:
        hi.put_block(host, lay_a, h, gg_inputs.index_coded(h * 131 + 7, M, N, es).numpy(),
                     lay.in_off, N)
    sh = _heap(H, part)
    sh.storage.copy_(torch.from_numpy(host).cuda())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.set_claim_policy(policy)
    try:
        gg.all_gather(sh.heap, -1, sh.ptr(start, lay.in_off), N, sh.ptr(start, lay.out_off), N,
                      M, N, dt, tile, programs, group, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # the ordinary call's claim decision (its counter in the one workspace
        # slot) is the new call's: same rule, same arguments
        assert (_counter(sh) > 0) == claims, _counter(sh)
        oracle.all_gather(host, part, lay.in_off, N, lay.out_off, N, M, N, es, group)
        oracle.all_gather(host, part, lay.in_off, N, out_b, N, M, N, es, group)
        for call in range(2):
            for h in members:  # the new call must write every byte of its output
                sh.partition(h)[out_b: out_b + lay_b.out_bytes].fill_(gg_inputs.SENTINEL_BYTE)
            ws_before = _counter(sh)
            gg.all_gather_noalloc(sh.heap, -1, sh.ptr(start, lay.in_off), N,
                                  sh.ptr(start, out_b), N, M, N, dt, tile, programs, group,
                                  status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert _counter(sh) == ws_before, "the new call used the heap's workspace"
            for h in members:
                want = _bits(sh.view(h, lay.out_off, W * M, N, N, dt))
                got = _bits(sh.view(h, out_b, W * M, N, N, dt))
                assert torch.equal(got, want), (call, h)
            got = download(sh)
            assert np.array_equal(got, host), (call, first_diff(got, host, lay_b))
    finally:
        gg.set_claim_policy("auto")


def test_noalloc_benchmark_size_twice(oracle):
    """W=8, 4096x4096 f16, tile 8x256, 148 programs, automatic claims: the
    benchmark's gather through the new call, twice in a row."""
    import gemm_gather_gb300 as gg
    from tests.test_gpu_fullsize import _assert_sentinel, _rows_sample
    W, M, N, dt, es = 8, 4096, 4096, torch.float16, 2
    guard = 1 << 16
    in_bytes, out_bytes = M * N * es, W * M * N * es
    in_off, out_off = guard, 2 * guard + in_bytes
    part = out_off + out_bytes + guard
    sh = _heap(W, part)
    gen = gg_inputs.generator(3, device="cuda")
    inputs = {}
    for h in range(W):
        x = gg_inputs.uniform_pm1((M, N), dt, gen)
        sh.view(h, in_off, M, N, N, dt).copy_(x)
        inputs[h] = x
    group = (0, 1, W)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the same launch through the ordinary call claims (automatic policy)
    gg.all_gather(sh.heap, -1, sh.ptr(0, in_off), N, sh.ptr(0, out_off), N, M, N, dt, (8, 256),
                  148, group, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and _counter(sh) > 0
    rows = _rows_sample(M, 6, seed=11)
    R = len(rows)
    host_part = R * N * es + W * R * N * es
    img = np.full(W * host_part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
    for h in range(W):
        blk = _bits(inputs[h][torch.from_numpy(rows).cuda()]).cpu().numpy()
        img[h * host_part: h * host_part + R * N * es] = blk.view(np.uint8).ravel()
    oracle.all_gather(img, host_part, 0, N, R * N * es, N, R, N, es, group)
    idx = torch.from_numpy(np.concatenate([i * M + rows for i in range(W)])).cuda()
    for call in range(2):
        for h in range(W):
            sh.view(h, out_off, W * M, N, N, dt).view(torch.int16).fill_(-1)
        gg.all_gather_noalloc(sh.heap, -1, sh.ptr(0, in_off), N, sh.ptr(0, out_off), N, M, N,
                              dt, (8, 256), 148, group, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for d in range(W):
            out = _bits(sh.view(d, out_off, W * M, N, N, dt))
            for i in range(W):
                assert torch.equal(out[i * M:(i + 1) * M], _bits(inputs[i])), (call, d, i)
            want = img[d * host_part + R * N * es: (d + 1) * host_part].view(np.int16)
            assert np.array_equal(out[idx].cpu().numpy().ravel(), want), (call, d)
        for h in range(W):
            p = sh.partition(h)
            _assert_sentinel(p[:in_off], f"heap {h} front guard")
            _assert_sentinel(p[in_off + in_bytes:out_off], f"heap {h} middle guard")
            _assert_sentinel(p[out_off + out_bytes:], f"heap {h} back guard")


def test_noalloc_rejects_like_all_gather():
    """Argument checks are the ordinary call's (nothing is launched)."""
    import gemm_gather_gb300 as gg
    sh = gg.SymmetricHeap(2, 1 << 20, device="cuda", workspace_slots=0)
    with pytest.raises(gg.GGError) as e:
        gg.all_gather_noalloc(sh.heap, -1, sh.ptr(0, 0), 64, sh.ptr(0, 4096), 32, 16, 64,
                              torch.float16, (8, 64), 2, (0, 1, 2))   # ld_out below N
    assert e.value.status == gg.GG_ERR_INVALID_ARG
