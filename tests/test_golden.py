"""The oracle still produces the committed fixtures of tests/golden/ (written
by tests/golden/make_golden.py from the oracle only), and the fixtures obey
the definitions they freeze, checked here independently of the oracle."""
import json
import os

import numpy as np

from tests.golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def parse(text):
    lines = text.strip().splitlines()
    case = json.loads(lines[0])
    blocks, cur, key = {}, None, None
    for ln in lines[1:]:
        if ln.startswith(("input", "output")):
            kind, h = ln.split()
            key = (kind, int(h))
            blocks[key] = []
        else:
            blocks[key].append([int(v, 16) for v in ln.split()])
    return case, {k: np.array(v, dtype=np.uint16) for k, v in blocks.items()}


def test_fixtures_reproduce():
    for name, case in make_golden.CASES.items():
        ins, outs = make_golden.run(case)
        assert make_golden.render(case, ins, outs) == open(os.path.join(HERE, name)).read(), name


def test_fixtures_obey_their_definitions():
    for name in make_golden.CASES:
        case, blocks = parse(open(os.path.join(HERE, name)).read())
        start, stride, W = case["group"]
        M = case["M"]
        members = [start + i * stride for i in range(W)]
        for di, d in enumerate(members):
            out = blocks[("output", d)]
            for i, src in enumerate(members):
                inp = blocks[("input", src)]
                want = inp[di * M:(di + 1) * M] if case["kind"] == "all_to_all" else inp
                assert np.array_equal(out[i * M:(i + 1) * M], want), (name, d, i)


import pytest  # noqa: E402


@pytest.mark.gpu
def test_gpu_reproduces_fixtures():
    """The CUDA path gives the fixtures' outputs (values written by the oracle script)."""
    import torch

    import gemm_gather_gb300 as gg
    for name in make_golden.CASES:
        case, blocks = parse(open(os.path.join(HERE, name)).read())
        start, stride, W = case["group"]
        M, N = case["M"], case["N"]
        members = [start + i * stride for i in range(W)]
        rows = blocks[("input", members[0])].shape[0]
        in_off, out_off = 0, 4096
        sh = gg.SymmetricHeap(case["H"], 8192, device="cuda", fill=0)
        for h in members:
            sh.view(h, in_off, rows, N, N, torch.int16).copy_(
                torch.from_numpy(blocks[("input", h)].view(np.int16)).cuda())
        fn = gg.all_to_all if case["kind"] == "all_to_all" else gg.all_gather
        fn(sh.heap, -1, sh.ptr(start, in_off), N, sh.ptr(start, out_off), N, M, N,
           torch.float16, (1, 8), 3, tuple(case["group"]))
        torch.cuda.synchronize()
        for h in members:
            got = sh.view(h, out_off, W * M, N, N, torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, blocks[("output", h)]), (name, h)
