"""Parity of the fused tcgen05 matmul + all-gather with the oracle, through
the C ABI.

* Integer-valued operands: every product and partial sum is an exact integer
  in float32, so the device result must equal the oracle's bit for bit, over
  the WHOLE heap (outputs, padding, guards, inputs, inactive heaps).
* Random operands (normal / sqrt(K)): every value within
  5e-3 * RMS(reference row) of the float64 reference, plus half an ulp of the
  output type for the final rounding; every byte outside the outputs
  untouched; the W copies of each block bit-identical.
"""
import numpy as np
import pytest
import torch

import gg_inputs
from tests import heap_image as hi
from tests.gpu_util import device_heap, download, first_diff

pytestmark = pytest.mark.gpu

FMT = {torch.float16: 0, torch.bfloat16: 1}
MANT = {torch.float16: 10, torch.bfloat16: 7}  # stored fraction bits
REL_TOL = 5e-3


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def half_ulp(x: np.ndarray, dtype) -> np.ndarray:
    """Half an ulp of the 16-bit type at |x| (normal range)."""
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    e = np.floor(np.log2(ax))
    return np.ldexp(1.0, (e - MANT[dtype] - 1).astype(np.int64))


def check_tolerance(gpu_vals: np.ndarray, ref: np.ndarray, dtype) -> None:
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    bound = REL_TOL * rms + np.maximum(half_ulp(ref, dtype), half_ulp(gpu_vals, dtype))
    err = np.abs(gpu_vals - ref)
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} values outside tolerance; worst "
                           f"{float((err / bound).max()):.3f} x bound")


def kernel_args(kernel):
    """(path, tile) of a kernel id: "1sm" / "2sm" run the 128 x 256 CTA tile on
    one CTA / CTA pairs; "wide" runs the 128 x 512 CTA tile (CTA pairs)."""
    import gemm_gather_gb300 as gg
    if kernel == "wide":
        return "auto", gg.FUSED_TILE_WIDE
    return kernel, gg.FUSED_TILE


def run_fused(oracle, H, group, M, N, K, dtype, programs, values="int", lda_pad=0,
              ld_out_pad=0, mode="group", seed=0, path="auto"):
    import gemm_gather_gb300 as gg
    path, tile = kernel_args(path)
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    lda = (K + 7) // 8 * 8 + lda_pad  # TMA needs 16-byte row pitches
    lay = hi.make_layout(H, W, M, N, 2, ld_in=lda, ld_out=N + ld_out_pad)
    host = hi.sentinel_heap(lay)
    gen = gg_inputs.generator(seed)
    A = {}
    for h in range(H):
        if values == "int":
            t = gg_inputs.integers((M, K), -2, 2, dtype, gen)
        else:
            t = gg_inputs.normal((M, K), dtype, gen, scale=K ** -0.5)
        if h in members:
            A[h] = t
            hi.put_block(host, lay, h, _bits(t), lay.in_off, lda)
    if values == "int":
        B = gg_inputs.integers((K, N), -2, 2, dtype, gen)
    else:
        B = gg_inputs.normal((K, N), dtype, gen, scale=K ** -0.5)
    sh = device_heap(lay, host)
    Bd = B.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if mode == "group":
        gg.matmul_all_gather(sh.heap, -1, sh.ptr(members[0], lay.in_off), lda, Bd, N,
                             sh.ptr(members[0], lay.out_off), lay.ld_out, M, N, K, dtype,
                             tile, programs, group, status=status, path=path)
    else:
        for h in members:
            gg.matmul_all_gather(sh.heap, h, sh.ptr(h, lay.in_off), lda, Bd, N,
                                 sh.ptr(h, lay.out_off), lay.ld_out, M, N, K, dtype,
                                 tile, programs, group, status=status, path=path)
    got = download(sh)
    assert int(status.item()) == 0, int(status.item())
    prods = oracle.matmul_all_gather(host, lay.part_bytes, lay.in_off, lda, _bits(B),
                                     lay.out_off, lay.ld_out, M, N, K, FMT[dtype], group)
    if values == "int":
        assert np.array_equal(got, host), first_diff(got, host, lay)
        return
    mask = hi.output_mask(lay, members)
    assert np.array_equal(got[~mask], host[~mask]), "bytes outside the outputs changed"
    outs = [hi.get_block(got, lay, d, lay.out_off, W * M, lay.ld_out, N, np.uint16)
            for d in members]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "destination copies differ"
    vals = torch.from_numpy(outs[0].view(np.int16)).view(dtype).to(torch.float64).numpy()
    for i in range(W):
        check_tolerance(vals[i * M:(i + 1) * M], prods[i], dtype)


# (H, group, M, N, K, programs, lda_pad, ld_out_pad)
INT_CASES = [
    (2, (0, 1, 2), 128, 256, 64, 2, 0, 0),        # one tile, one K block
    (2, (0, 1, 2), 128, 256, 192, 2, 0, 0),       # ring of 3 stages filled once
    (2, (0, 1, 2), 128, 256, 640, 1, 0, 0),       # ring wraps; one CTA
    (2, (0, 1, 2), 128, 256, 100, 2, 0, 0),       # ragged K
    (2, (0, 1, 2), 200, 264, 72, 4, 8, 16),       # ragged M, N, K; padded pitches
    (3, (0, 1, 3), 300, 520, 320, 5, 0, 8),       # several tiles per CTA
    (8, (0, 2, 4), 64, 512, 128, 3, 0, 0),        # strided subgroup, inactive heaps
    (8, (1, 2, 4), 129, 256, 64, 148, 0, 0),      # subgroup from heap 1, more CTAs than tiles
    (4, (0, 1, 4), 256, 768, 256, 1, 0, 0),       # one CTA walks 24 tiles (TMEM phases)
    (8, (0, 1, 8), 256, 1024, 1024, 2, 0, 0),     # one pair walks 32 tiles at W=8: every
                                                  # store slot of the paced epilogue
    (1, (0, 1, 1), 8, 8, 16, 1, 0, 0),            # tiny, W = 1
    (64, (0, 1, 64), 16, 256, 64, 40, 0, 0),      # 64 members: epilogue stores wrap the lanes
    (40, (3, 1, 33), 40, 264, 96, 400, 0, 8),     # 33 members from heap 3, more CTAs than SMs
]


PATHS = ["1sm", "2sm", "wide"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("case", INT_CASES, ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}x{c[4]}p{c[5]}")
def test_integer_operands_bit_exact(oracle, case, dtype, path):
    H, group, M, N, K, programs, lp, op = case
    if path != "1sm" and programs < 2:
        programs = 2
    run_fused(oracle, H, group, M, N, K, dtype, programs, "int", lp, op, path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("shape", [(256, 512, 1024), (130, 264, 520), (512, 1024, 2048)])
def test_random_operands_within_tolerance(oracle, shape, dtype, path):
    M, N, K = shape
    run_fused(oracle, 3, (0, 1, 3), M, N, K, dtype, 7, "normal", path=path)


# (H, group, M, N, K, programs): the 128 x 512 kernel's last wave is at most
# half full, so its pair tiles run as two 256 x 256 halves on twice as many pairs
TAIL_CASES = [
    (3, (0, 1, 3), 256, 1024, 256, 8),     # 6 tiles on 4 pairs: 2 split
    (5, (0, 1, 5), 300, 776, 200, 18),     # 20 tiles on 9 pairs: 2 split, ragged M, N, K
    (8, (1, 2, 3), 100, 520, 64, 10),      # 6 tiles on 5 pairs: 1 split, its half 1 empty
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("case", TAIL_CASES, ids=lambda c: f"H{c[0]}g{c[1]}_{c[2]}x{c[3]}x{c[4]}p{c[5]}")
def test_wide_tail_half_tiles_bit_exact(oracle, case, dtype):
    H, group, M, N, K, programs = case
    total = group[2] * -(-M // 256) * -(-N // 512)
    pairs = min(programs // 2, total)
    assert 0 < total % pairs and 2 * (total % pairs) <= pairs  # the tail is split
    run_fused(oracle, H, group, M, N, K, dtype, programs, "int", path="wide")
    run_fused(oracle, H, group, M, N, K, dtype, programs, "normal", path="wide", seed=1)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_single_rank_launches(oracle, dtype, path):
    run_fused(oracle, 4, (0, 1, 4), 160, 512, 192, dtype, 5, "int", mode="ranks", path=path)
    run_fused(oracle, 6, (1, 2, 3), 96, 256, 320, dtype, 3, "normal", mode="ranks", path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("mode", ["group", "ranks"])
def test_empty_contraction_gathers_zero_blocks(oracle, mode, dtype, path):
    """K == 0: C_r is the empty sum, the zero matrix; every member's gathered
    rows become zeros (padding columns untouched), exactly as the oracle's
    definition gives.  A and B are not read: B is passed as NULL."""
    import gemm_gather_gb300 as gg
    kpath, tile = kernel_args(path)
    H, group, M, N = 5, (1, 1, 3), 130, 264
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    lay = hi.make_layout(H, W, M, N, 2, ld_in=8, ld_out=N + 8)
    host = hi.sentinel_heap(lay)
    sh = device_heap(lay, host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    programs = 1 if path == "1sm" else 6
    if mode == "group":
        gg.matmul_all_gather(sh.heap, -1, sh.ptr(start, lay.in_off), 8, None, N,
                             sh.ptr(start, lay.out_off), lay.ld_out, M, N, 0, dtype, tile,
                             programs, group, status=status, path=kpath)
    else:
        for h in members:
            gg.matmul_all_gather(sh.heap, h, sh.ptr(h, lay.in_off), 8, None, N,
                                 sh.ptr(h, lay.out_off), lay.ld_out, M, N, 0, dtype, tile,
                                 programs, group, status=status, path=kpath)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.matmul_all_gather(host, lay.part_bytes, lay.in_off, 8, np.zeros((0, N), np.uint16),
                             lay.out_off, lay.ld_out, M, N, 0, FMT[dtype], group)
    assert np.array_equal(got, host), first_diff(got, host, lay)


def _fused_custom(oracle, A, B, dtype, path, group=(0, 1, 2)):
    """Run the group launch on the given operands (A: {member: M x K}, B: K x N)
    and return (device heap, oracle heap, layout, members)."""
    import gemm_gather_gb300 as gg
    kpath, tile = kernel_args(path)
    start, stride, W = group
    members = [start + i * stride for i in range(W)]
    M, K = A[members[0]].shape
    N = B.shape[1]
    H = members[-1] + 1
    lay = hi.make_layout(H, W, M, N, 2, ld_in=K, ld_out=N)
    host = hi.sentinel_heap(lay)
    for h in members:
        hi.put_block(host, lay, h, _bits(A[h]), lay.in_off, K)
    sh = device_heap(lay, host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gg.matmul_all_gather(sh.heap, -1, sh.ptr(start, lay.in_off), K, B.to("cuda"), N,
                         sh.ptr(start, lay.out_off), N, M, N, K, dtype, tile,
                         1 if path == "1sm" else 4, group, status=status, path=kpath)
    got = download(sh)
    assert int(status.item()) == 0
    oracle.matmul_all_gather(host, lay.part_bytes, lay.in_off, K, _bits(B), lay.out_off, N, M, N,
                             K, FMT[dtype], group)
    return got, host, lay, members


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_overflowing_sums_round_like_the_oracle(oracle, dtype, path):
    """A in {-256, 0, 256} and B in {-256, -1, 0, 1, 256}: every product is 0,
    +-256 or +-65536 and every f32 partial sum an exact multiple of 256 below
    2^24, so the products are exact whatever order the sums take.  Sums of
    65536 or more pass binary16's largest finite value (65504): the f16
    outputs hold +-inf there, as round-to-nearest-even gives; the whole heap
    must match the oracle bit for bit."""
    g = gg_inputs.generator(21)
    M, N, K = 160, 512, 64

    def draw(shape, vals):
        v = torch.tensor(vals)
        return v[torch.randint(0, len(vals), shape, generator=g)].to(dtype)

    A = {h: draw((M, K), [-256.0, 0.0, 256.0]) for h in (0, 1)}
    B = draw((K, N), [-256.0, -1.0, 0.0, 1.0, 256.0])
    got, host, lay, _ = _fused_custom(oracle, A, B, dtype, path)
    if dtype == torch.float16:
        out = hi.get_block(host, lay, 0, lay.out_off, 2 * M, N, N, np.uint16)
        assert ((out & 0x7FFF) == 0x7C00).sum() > 1000  # the case reaches overflow
    assert np.array_equal(got, host), first_diff(got, host, lay)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_non_finite_operands_propagate(oracle, dtype, path):
    """+-inf and NaN in A: inf * 0 and inf - inf give NaN, inf * x gives inf,
    NaN spreads along its row.  NaN has no unique encoding, so the test
    compares which outputs are NaN and every other output bit for bit (inf
    signs included); the W copies must be identical and nothing outside the
    outputs may change."""
    g = gg_inputs.generator(22)
    M, N, K = 128, 256, 64
    A = {}
    for h in (0, 1):
        a = gg_inputs.integers((M, K), -2, 2, dtype, g)
        a[3, 5] = float("inf")
        a[9, 0] = float("-inf")
        a[17, 2], a[17, 40] = float("inf"), float("-inf")
        a[33, 7] = float("nan")
        A[h] = a
    B = gg_inputs.integers((K, N), -2, 2, dtype, g)
    B[5, :8] = 0            # inf * 0 = NaN in row 3's first columns
    got, host, lay, members = _fused_custom(oracle, A, B, dtype, path)
    mask = hi.output_mask(lay, members)
    assert np.array_equal(got[~mask], host[~mask]), "bytes outside the outputs changed"
    outs = [hi.get_block(got, lay, d, lay.out_off, 2 * M, N, N, np.uint16) for d in members]
    assert np.array_equal(outs[0], outs[1]), "destination copies differ"
    ref = hi.get_block(host, lay, 0, lay.out_off, 2 * M, N, N, np.uint16)
    exp_mask, man_mask = (0x7C00, 0x03FF) if dtype == torch.float16 else (0x7F80, 0x007F)
    nan_got = ((outs[0] & exp_mask) == exp_mask) & ((outs[0] & man_mask) != 0)
    nan_ref = ((ref & exp_mask) == exp_mask) & ((ref & man_mask) != 0)
    assert nan_ref.sum() >= 2 * N and np.array_equal(nan_got, nan_ref)
    assert np.array_equal(outs[0][~nan_ref], ref[~nan_ref])
