"""CUDA graphs and randomized parity.

* The public calls enqueue only kernel launches on the caller's stream (and,
  for a launch that claims runs of tiles, one memset of its workspace
  counter); the host does its validation and tensor-map encoding before the
  launch.  So a whole step -- gather + fused -- can be captured into a CUDA
  graph and replayed; the replay must give the oracle's heap, with fixed
  shares and with claimed runs (the memset is replayed with the kernel).
* Seeded random configurations of the gather, the partitioned gather and the
  all-to-all (group, shape, tile, pitches, programs, path, dtype) must match
  the oracle over the whole heap, under the automatic claim policy and with
  claims forced on.
"""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy,M,N,programs,wide", [("auto", 48, 512, 16, True),
                                                      ("always", 256, 1024, 2, False)])
def test_step_captured_in_a_cuda_graph(oracle, policy, M, N, programs, wide):
    import gemm_gather_gb300 as gg
    fused_tile = gg.FUSED_TILE_WIDE if wide else gg.FUSED_TILE
    W = 4
    Mf, Nf, Kf = 256, 512, 192
    es = 2
    # one heap holding the gather's and the fused call's buffers
    in_off, out_off = 4096, 4096 + M * N * es + 4096
    a_off = out_off + W * M * N * es + 4096
    c_off = a_off + Mf * Kf * 2 + 4096
    part = c_off + W * Mf * Nf * 2 + 4096
    part = (part + 4095) // 4096 * 4096
    host = np.full(W * part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
    gen = gg_inputs.generator(21)
    for h in range(W):
        blk = gg_inputs.index_coded(h, M, N, es).numpy().view(np.uint8).ravel()
        host[h * part + in_off: h * part + in_off + blk.size] = blk
        a = gg_inputs.integers((Mf, Kf), -2, 2, torch.float16, gen)
        ab = a.view(torch.int16).numpy().view(np.uint8).ravel()
        host[h * part + a_off: h * part + a_off + ab.size] = ab
    B = gg_inputs.integers((Kf, Nf), -2, 2, torch.float16, gen)
    lay = hi.Layout(W, part, in_off, N, out_off, N, M, N, W, es)
    sh = device_heap(lay, host)
    Bd = B.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        gg.all_gather(sh.heap, -1, sh.ptr(0, in_off), N, sh.ptr(0, out_off), N, M, N,
                      torch.float16, (8, 256), programs, (0, 1, W), status=status, stream=stream)
        gg.matmul_all_gather(sh.heap, -1, sh.ptr(0, a_off), Kf, Bd, Nf, sh.ptr(0, c_off), Nf,
                             Mf, Nf, Kf, torch.float16, fused_tile, 8, (0, 1, W),
                             status=status, stream=stream)

    gg.set_claim_policy(policy)
    try:
        # warm once outside the graph (first-use set-up), then capture and replay
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        sh.storage.copy_(torch.from_numpy(host).cuda())
        sh.workspace.zero_()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    finally:
        gg.set_claim_policy("auto")
    assert int(status.item()) == 0
    # the captured gather used workspace slot 1 (the warm-up took slot 0)
    assert (int(sh.workspace.view(torch.int64)[16].item()) > 0) == (policy == "always")
    got = download(sh)
    oracle.all_gather(host, part, in_off, N, out_off, N, M, N, es, (0, 1, W))
    oracle.matmul_all_gather(host, part, a_off, Kf, B.view(torch.int16).numpy().view(np.uint16),
                             c_off, Nf, Mf, Nf, Kf, 0, (0, 1, W))
    assert np.array_equal(got, host), first_diff(got, host, lay)


def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        kind = rng.choice(["all_gather", "partitioned", "all_to_all"])
        W = int(rng.integers(1, 9))
        stride = int(rng.choice([1, 1, 2, 3]))
        start = int(rng.integers(0, 3))
        H = start + (W - 1) * stride + 1 + int(rng.integers(0, 2))
        es = int(rng.choice([2, 4]))
        M = int(rng.integers(1, 140))
        N = int(rng.choice([1, 3, 8, 40, 64, 256, 300, 520]))
        bm = int(rng.choice([1, 4, 8, 16, 32, 64]))
        bn = int(rng.choice([8, 16, 64, 128, 256]))
        if bm * bn * es > 32768:
            bn = 32768 // (bm * es)
        pi = int(rng.choice([0, 0, 1, 8]))
        po = int(rng.choice([0, 0, 3, 8]))
        programs = int(rng.integers(1, 200))
        if kind == "partitioned":
            programs = max(programs, W)
        path = str(rng.choice(["auto", "tma", "vector"]))
        cases.append((kind, H, (start, stride, W), M, N, es, (bm, bn), programs, pi, po, path))
    return cases


@pytest.mark.parametrize("policy", ["auto", "always"])
@pytest.mark.parametrize("case", _random_cases(40, 2026), ids=lambda c: f"{c[0]}_W{c[2][2]}_{c[3]}x{c[4]}e{c[5]}t{c[6]}p{c[7]}_{c[10]}")
def test_random_collective_matches_oracle(oracle, case, policy):
    """"always" makes every tensor-map all-gather / all-to-all with a few runs
    per pipeline claim them, so the claimed-run walk meets random shapes,
    tiles and budgets too."""
    import gemm_gather_gb300 as gg
    kind, H, group, M, N, es, tile, programs, pi, po, path = case
    W = group[2]
    ld_in, ld_out = N + pi, N + po
    tma_ok = (ld_in * es) % 16 == 0 and (ld_out * es) % 16 == 0 and (tile[1] * es) % 16 == 0 \
        and tile[1] <= 256
    if path == "tma" and not tma_ok:
        path = "auto"
    rows_in = W * M if kind == "all_to_all" else M
    lay = hi.make_layout(H, W, rows_in, N, es, ld_in=ld_in, ld_out=ld_out)
    host = hi.sentinel_heap(lay)
    members = [group[0] + i * group[1] for i in range(W)]
    for h in members:
        hi.put_block(host, lay, h, gg_inputs.index_coded(h * 3 + 1, rows_in, N, es).numpy(),
                     lay.in_off, ld_in)
    sh = device_heap(lay, host)
    dt = {2: torch.float16, 4: torch.float32}[es]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (sh.heap, -1, sh.ptr(members[0], lay.in_off), ld_in, sh.ptr(members[0], lay.out_off),
            ld_out, M, N, dt, tile, programs, group)
    fn = {"all_gather": gg.all_gather, "partitioned": gg.all_gather_partitioned,
          "all_to_all": gg.all_to_all}[kind]
    gg.set_claim_policy(policy)
    try:
        fn(*args, status=status, path=path)
    finally:
        gg.set_claim_policy("auto")
    got = download(sh)
    assert int(status.item()) == 0
    if kind == "all_to_all":
        oracle.all_to_all(host, lay.part_bytes, lay.in_off, ld_in, lay.out_off, ld_out, M, N, es,
                          group)
    else:
        oracle.all_gather(host, lay.part_bytes, lay.in_off, ld_in, lay.out_off, ld_out, M, N, es,
                          group)
    assert np.array_equal(got, host), first_diff(got, host, lay)
