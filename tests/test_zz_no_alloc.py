"""The allocation-free all-gather (gg_all_gather_noalloc) against the
ordinary entry point, through the C ABI.

gg_all_gather_noalloc exists for callers that cannot allocate device memory
once running (a plugin inside a framework that owns the device memory, a
real-time loop that may not synchronize on an allocation): when it claims
runs of tiles, its counter lives in a small static device array of the
library instead of a heap workspace the caller would have to allocate.

Each case gathers the same inputs twice in a row with the new call and
compares every member's output, byte for byte, with gg_all_gather's (a gather
is a copy, so the bar is bit-exact).  The second call starts from the counter
the first one left behind in the shared array: it only matches if the call
clears it first.  The heap has no workspace, so the ordinary call keeps fixed
shares while the new one claims.  This file is collected last on purpose.
"""
import pytest
import torch

import gg_inputs

pytestmark = pytest.mark.gpu

GUARD = 1 << 16


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view({2: torch.int16, 4: torch.int32}[t.element_size()])


# (W, M, N, dtype, tile, programs, claim policy, input misalignment in elements)
CASES = [
    (4, 512, 2048, torch.float16, (8, 256), 2, "always", 0),     # claims from the static counter
    (8, 4096, 4096, torch.float16, (8, 256), 148, "auto", 0),   # the benchmark's gather: claims
    (3, 200, 520, torch.float32, (16, 64), 5, "always", 0),     # ragged tiles
    (4, 64, 256, torch.float16, (8, 256), 4, "auto", 1),        # unaligned: vector path, no scratch
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"W{c[0]}_{c[1]}x{c[2]}_{str(c[3])[6:]}_"
                         f"t{c[4][0]}x{c[4][1]}_p{c[5]}_{c[6]}_mis{c[7]}")
def test_noalloc_matches_all_gather_twice(case):
    import gemm_gather_gb300 as gg
    W, M, N, dtype, tile, programs, policy, mis = case
    es = torch.empty((), dtype=dtype).element_size()
    in_bytes, out_bytes = (M * N + mis) * es, W * M * N * es
    in_off = GUARD
    out_a = in_off + (in_bytes + GUARD) // 256 * 256 + 256
    out_b = out_a + (out_bytes + GUARD) // 256 * 256 + 256
    part = out_b + out_bytes + GUARD
    sh = gg.SymmetricHeap(W, part, device="cuda", fill=gg_inputs.SENTINEL_BYTE, workspace_slots=0)
    gen = gg_inputs.generator(7, device="cuda")
    src = in_off + mis * es
    for h in range(W):
        sh.view(h, src, M, N, N, dtype).copy_(gg_inputs.uniform_pm1((M, N), dtype, gen))
    group = (0, 1, W)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.set_claim_policy(policy)
    try:
        gg.all_gather(sh.heap, -1, sh.ptr(0, src), N, sh.ptr(0, out_a), N, M, N, dtype, tile,
                      programs, group, status=status)
        for call in range(2):
            for h in range(W):  # the new call must write every byte of its output
                sh.partition(h)[out_b: out_b + out_bytes].fill_(gg_inputs.SENTINEL_BYTE)
            gg.all_gather_noalloc(sh.heap, -1, sh.ptr(0, src), N, sh.ptr(0, out_b), N, M, N,
                                  dtype, tile, programs, group, status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            for h in range(W):
                want = _bits(sh.view(h, out_a, W * M, N, N, dtype))
                got = _bits(sh.view(h, out_b, W * M, N, N, dtype))
                assert torch.equal(got, want), (call, h)
    finally:
        gg.set_claim_policy("auto")


def test_noalloc_rejects_like_all_gather():
    """Argument checks are the ordinary call's (nothing is launched)."""
    import gemm_gather_gb300 as gg
    sh = gg.SymmetricHeap(2, 1 << 20, device="cuda", workspace_slots=0)
    with pytest.raises(gg.GGError) as e:
        gg.all_gather_noalloc(sh.heap, -1, sh.ptr(0, 0), 64, sh.ptr(0, 4096), 32, 16, 64,
                              torch.float16, (8, 64), 2, (0, 1, 2))   # ld_out below N
    assert e.value.status == gg.GG_ERR_INVALID_ARG
