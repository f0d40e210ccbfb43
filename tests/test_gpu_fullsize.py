"""Parity at the benchmark configurations' full sizes, in the launch
configuration bench.py times.

At these sizes the whole heap cannot be compared with a host oracle image, so
each case checks
* properties that hold at any size, on the GPU, for every byte: every member's
  row block i equals member i's input (a gather is a copy; fused: all W copies
  of each block are bit-identical), and every byte outside the outputs keeps
  its sentinel (guards, inactive heaps);
* rows against the oracle: the oracle gathers (or multiplies, in float64)
  sampled rows of every rank, and those rows of every member's output must
  match (bit-exact for the gather, the float64 tolerance for the fused
  product); the fused product at M_local=1024 is compared on every row, the
  larger fused shapes on 256 seeded rows per rank.
Inputs are drawn on the GPU from a seeded generator (same distributions as
the benchmark); the sampled rows are copied to the host for the oracle.
"""
import numpy as np
import pytest
import torch

import gg_inputs
from tests.test_gpu_fused import check_tolerance

pytestmark = pytest.mark.gpu

GUARD = 1 << 16


def _heap(H, part, fill=gg_inputs.SENTINEL_BYTE):
    import gemm_gather_gb300 as gg
    return gg.SymmetricHeap(H, part, device="cuda", fill=fill)


def _rows_sample(M, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    rows.update({0, M - 1})
    return np.array(sorted(rows), dtype=np.int64)


def _ints(t: torch.Tensor) -> torch.Tensor:
    """Raw bit view of a 16- or 32-bit tensor."""
    return t.view({2: torch.int16, 4: torch.int32}[t.element_size()])


def _assert_sentinel(t: torch.Tensor, what: str):
    bad = int((t != gg_inputs.SENTINEL_BYTE).sum().item())
    assert bad == 0, f"{bad} bytes changed in {what}"


GATHER_CASES = [
    # (W, group, M, N, dtype, tile, programs, path, values)
    (8, (0, 1, 8), 4096, 4096, torch.float16, (8, 256), 148, "auto", "uniform"),
    (8, (0, 1, 8), 4096, 4096, torch.float16, (8, 256), 148, "bulk", "uniform"),
    (8, (0, 1, 8), 4096, 4096, torch.float16, (8, 256), 8, "auto", "uniform"),
    (8, (0, 1, 8), 16384, 8192, torch.float32, (8, 256), 148, "auto", "normal"),
    (8, (0, 1, 8), 16384, 8192, torch.float32, (32, 128), 128, "auto", "normal"),
    (4, (0, 1, 4), 16384, 8192, torch.bfloat16, (16, 128), 64, "bulk", "normal"),
    (4, (1, 2, 4), 16384, 8192, torch.float16, (8, 256), 148, "auto", "normal"),
]


@pytest.mark.parametrize("case", GATHER_CASES,
                         ids=lambda c: f"W{c[0]}g{c[1]}_{c[2]}x{c[3]}_{str(c[4])[6:]}_t{c[5]}_p{c[6]}_{c[7]}")
def test_gather_full_size(oracle, case):
    import gemm_gather_gb300 as gg
    W, group, M, N, dtype, tile, programs, path, values = case
    start, stride, _ = group
    members = [start + i * stride for i in range(W)]
    H = members[-1] + 1 + (1 if stride > 1 else 0)
    es = torch.empty((), dtype=dtype).element_size()
    in_bytes, out_bytes = M * N * es, W * M * N * es
    in_off, out_off = GUARD, 2 * GUARD + in_bytes
    part = out_off + out_bytes + GUARD
    sh = _heap(H, part)
    gen = gg_inputs.generator(0, device="cuda")
    draw = gg_inputs.uniform_pm1 if values == "uniform" else gg_inputs.normal
    inputs = {}
    for h in members:
        x = draw((M, N), dtype, gen)
        sh.view(h, in_off, M, N, N, dtype).copy_(x)
        inputs[h] = x
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.all_gather(sh.heap, -1, sh.ptr(start, in_off), N, sh.ptr(start, out_off), N, M, N, dtype,
                  tile, programs, group, status=status, path=path)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the automatic claim policy: tensor maps over >= 3/4 of the SMs claim runs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    claimed = int(sh.workspace.view(torch.int64)[0].item()) > 0
    assert claimed == (path == "auto" and 4 * programs >= 3 * sms), claimed
    # every byte: block i of every member == member i's input
    for d in members:
        out = sh.view(d, out_off, W * M, N, N, dtype)
        for i, h in enumerate(members):
            assert torch.equal(_ints(out[i * M:(i + 1) * M]), _ints(inputs[h])), (d, i)
    # guards and inactive heaps keep their sentinel
    for h in range(H):
        p = sh.partition(h)
        _assert_sentinel(p[:in_off], f"heap {h} front guard")
        if h in members:
            _assert_sentinel(p[in_off + in_bytes:out_off], f"heap {h} middle guard")
            _assert_sentinel(p[out_off + out_bytes:], f"heap {h} back guard")
        else:
            _assert_sentinel(p, f"inactive heap {h}")
    # sampled rows against the oracle
    rows = _rows_sample(M, 6, seed=M + N)
    R = len(rows)
    npdt = {2: np.int16, 4: np.int32}[es]
    host_part = R * N * es + W * R * N * es
    img = np.full(H * host_part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
    for h in members:
        blk = _ints(inputs[h][torch.from_numpy(rows).cuda()]).cpu().numpy()
        img[h * host_part: h * host_part + R * N * es] = blk.view(np.uint8).ravel()
    oracle.all_gather(img, host_part, 0, N, R * N * es, N, R, N, es, group)
    for d in members:
        want = img[d * host_part + R * N * es: (d + 1) * host_part].view(npdt).reshape(W * R, N)
        out = _ints(sh.view(d, out_off, W * M, N, N, dtype))
        idx = torch.from_numpy(np.concatenate([i * M + rows for i in range(W)])).cuda()
        got = out[idx].cpu().numpy()
        assert np.array_equal(got, want), d


# Rows of every rank compared with the float64 oracle: all of them at
# M_local=1024 (481 GFLOP of oracle work), a seeded sample of 256 (plus the
# first and last row) at the larger shapes.
FUSED_ALL_ROWS_UP_TO = 1024
FUSED_SAMPLE_ROWS = 256

FUSED_CASES = [
    # (W, group, M, dtype, kernel: "wide" = the bench's 128 x 512 CTA tiles on CTA
    #  pairs, "2sm" / "1sm" = 128 x 256 CTA tiles on CTA pairs / one CTA)
    (8, (0, 1, 8), 1024, torch.float16, "wide"),
    (8, (0, 1, 8), 1024, torch.float16, "2sm"),
    (8, (0, 1, 8), 1024, torch.float16, "1sm"),
    (8, (0, 1, 8), 4096, torch.float16, "wide"),
    (8, (0, 1, 8), 4096, torch.float16, "2sm"),
    (8, (0, 1, 8), 4096, torch.bfloat16, "wide"),
    (8, (0, 1, 8), 16384, torch.float16, "wide"),
    (8, (0, 1, 8), 16384, torch.bfloat16, "wide"),
    (4, (0, 2, 4), 4096, torch.float16, "wide"),
    (4, (0, 2, 4), 16384, torch.float16, "wide"),
    (4, (0, 2, 4), 16384, torch.bfloat16, "wide"),
]


@pytest.mark.parametrize("case", FUSED_CASES,
                         ids=lambda c: f"W{c[0]}g{c[1]}_M{c[2]}_{str(c[3])[6:]}_{c[4]}")
def test_fused_full_size(oracle, case):
    import gemm_gather_gb300 as gg
    from tests.test_gpu_fused import kernel_args
    W, group, M, dtype, kernel = case
    path, tile = kernel_args(kernel)
    N, K = 3584, 8192
    start, stride, _ = group
    members = [start + i * stride for i in range(W)]
    H = members[-1] + 1 + (1 if stride > 1 else 0)
    a_bytes, out_bytes = M * K * 2, W * M * N * 2
    a_off, out_off = GUARD, 2 * GUARD + a_bytes
    part = out_off + out_bytes + GUARD
    sh = _heap(H, part)
    gen = gg_inputs.generator(0, device="cuda")
    A = {}
    for h in members:
        a = gg_inputs.normal((M, K), dtype, gen, scale=K ** -0.5)
        sh.view(h, a_off, M, K, K, dtype).copy_(a)
        A[h] = a
    B = gg_inputs.normal((K, N), dtype, gen, scale=K ** -0.5)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    gg.matmul_all_gather(sh.heap, -1, sh.ptr(start, a_off), K, B, N, sh.ptr(start, out_off), N,
                         M, N, K, dtype, tile, sms, group, status=status, path=path)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # every byte: the W copies of every block are identical
    ref_out = sh.view(members[0], out_off, W * M, N, N, dtype).view(torch.int16)
    for d in members[1:]:
        assert torch.equal(sh.view(d, out_off, W * M, N, N, dtype).view(torch.int16), ref_out), d
    for h in range(H):
        p = sh.partition(h)
        _assert_sentinel(p[:a_off], f"heap {h} front guard")
        if h in members:
            _assert_sentinel(p[a_off + a_bytes:out_off], f"heap {h} middle guard")
            _assert_sentinel(p[out_off + out_bytes:], f"heap {h} back guard")
        else:
            _assert_sentinel(p, f"inactive heap {h}")
    # rows of every rank (all of them, or a seeded sample) against the float64 oracle
    if M <= FUSED_ALL_ROWS_UP_TO:
        rows = np.arange(M, dtype=np.int64)
    else:
        rows = _rows_sample(M, FUSED_SAMPLE_ROWS, seed=M + 17 * W + int(dtype == torch.bfloat16))
    Bbits = B.view(torch.int16).cpu().numpy().view(np.uint16)
    fmt = 0 if dtype == torch.float16 else 1
    out = ref_out.view(dtype)
    for i, h in enumerate(members):
        a_rows = A[h][torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
        ref = oracle.matmul_f64(a_rows, Bbits, fmt)
        got = out[torch.from_numpy(i * M + rows).cuda()].to(torch.float64).cpu().numpy()
        check_tolerance(got, ref, dtype)


def test_all_to_all_full_size(oracle):
    """All-to-all, W=8, 4096x4096 f16 blocks (256 MB input per member), 148 programs."""
    import gemm_gather_gb300 as gg
    W, M, N, dtype = 8, 4096, 4096, torch.float16
    members = list(range(W))
    blk_bytes = M * N * 2
    in_off, out_off = GUARD, 2 * GUARD + W * blk_bytes
    part = out_off + W * blk_bytes + GUARD
    sh = _heap(W, part)
    gen = gg_inputs.generator(1, device="cuda")
    inputs = {}
    for h in members:
        x = gg_inputs.uniform_pm1((W * M, N), dtype, gen)
        sh.view(h, in_off, W * M, N, N, dtype).copy_(x)
        inputs[h] = x
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.all_to_all(sh.heap, -1, sh.ptr(0, in_off), N, sh.ptr(0, out_off), N, M, N, dtype, (8, 256),
                  148, (0, 1, W), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for d in members:
        out = _ints(sh.view(d, out_off, W * M, N, N, dtype))
        for i in members:
            assert torch.equal(out[i * M:(i + 1) * M], _ints(inputs[i][d * M:(d + 1) * M])), (d, i)
    for h in members:
        p = sh.partition(h)
        _assert_sentinel(p[:in_off], f"heap {h} front guard")
        _assert_sentinel(p[in_off + W * blk_bytes:out_off], f"heap {h} middle guard")
        _assert_sentinel(p[out_off + W * blk_bytes:], f"heap {h} back guard")
    # sampled rows of every block against the oracle
    rows = _rows_sample(M, 4, seed=7)
    R = len(rows)
    host_part = 2 * W * R * N * 2
    img = np.full(W * host_part, gg_inputs.SENTINEL_BYTE, dtype=np.uint8)
    idx_in = torch.from_numpy(np.concatenate([d * M + rows for d in range(W)])).cuda()
    for h in members:
        blk = _ints(inputs[h][idx_in]).cpu().numpy()
        img[h * host_part: h * host_part + W * R * N * 2] = blk.view(np.uint8).ravel()
    oracle.all_to_all(img, host_part, 0, N, W * R * N * 2, N, R, N, 2, (0, 1, W))
    for d in members:
        want = img[d * host_part + W * R * N * 2: (d + 1) * host_part].view(np.int16)
        got = _ints(sh.view(d, out_off, W * M, N, N, dtype))[idx_in].cpu().numpy()
        assert np.array_equal(got.ravel(), want), d
