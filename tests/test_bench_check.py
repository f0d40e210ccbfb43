"""bench.py's per-point output check (check_point) on host tensors: it passes
on a correct gather / all-to-all / fused result and raises on a planted
mistake (a swapped block, one flipped element, a copy that differs, a value
outside the tolerance).  No GPU: the heap is a stand-in with the same view()
as gemm_gather_gb300.SymmetricHeap."""
import pytest
import torch

import bench
import gg_inputs


class HostHeap:
    def __init__(self, H, part):
        self.part = part
        self.storage = torch.zeros(H * part, dtype=torch.uint8)

    def view(self, h, offset, rows, cols, ld, dtype):
        es = torch.empty((), dtype=dtype).element_size()
        n = (rows - 1) * ld + cols
        flat = self.storage[h * self.part + offset: h * self.part + offset + n * es].view(dtype)
        return flat.as_strided((rows, cols), (ld, 1))


def _gather_heap(kind):
    g = bench.GatherCfg(W=3, M=16, N=24, dtype="f32", kind=kind)
    in_rows = g.W * g.M if kind == "all_to_all" else g.M
    offs = {"g_in": 0, "g_out": 4096}
    sh = HostHeap(3, 4096 + g.W * g.M * g.N * 4)
    gen = gg_inputs.generator(0)
    for h in g.members():
        sh.view(h, 0, in_rows, g.N, g.N, torch.float32).copy_(
            gg_inputs.normal((in_rows, g.N), torch.float32, gen))
    for d_idx, d in enumerate(g.members()):
        out = sh.view(d, 4096, g.W * g.M, g.N, g.N, torch.float32)
        for i, h in enumerate(g.members()):
            src = sh.view(h, 0, in_rows, g.N, g.N, torch.float32)
            blk = src[d_idx * g.M:(d_idx + 1) * g.M] if kind == "all_to_all" else src
            out[i * g.M:(i + 1) * g.M] = blk
    return g, sh, offs


@pytest.mark.parametrize("kind", ["all_gather", "all_to_all", "partitioned"])
def test_check_point_gather(kind):
    g, sh, offs = _gather_heap(kind)
    assert "bit-exact" in bench.check_point(g, None, sh, offs, None)
    out = sh.view(2, offs["g_out"], g.W * g.M, g.N, g.N, torch.float32)
    out[g.M + 3, 5] = out[g.M + 3, 5] + 1.0  # one element of block 1 of member 2
    with pytest.raises(RuntimeError, match="member 2 block 1"):
        bench.check_point(g, None, sh, offs, None)


def test_check_point_gather_swapped_blocks():
    g, sh, offs = _gather_heap("all_gather")
    out = sh.view(0, offs["g_out"], g.W * g.M, g.N, g.N, torch.float32)
    b0 = out[:g.M].clone()
    out[:g.M] = out[g.M:2 * g.M]
    out[g.M:2 * g.M] = b0
    with pytest.raises(RuntimeError, match="member 0 block 0"):
        bench.check_point(g, None, sh, offs, None)


def _fused_heap(dtype="f16"):
    f = bench.FusedCfg(W=2, M=8, N=16, K=32, dtype=dtype)
    dt = gg_inputs.DTYPES[dtype]
    offs = {"f_a": 0, "f_out": 1024}
    sh = HostHeap(2, 1024 + f.W * f.M * f.N * 2)
    gen = gg_inputs.generator(1)
    for h in f.members():
        sh.view(h, 0, f.M, f.K, f.K, dt).copy_(gg_inputs.normal((f.M, f.K), dt, gen,
                                                                scale=f.K ** -0.5))
    B = gg_inputs.normal((f.K, f.N), dt, gen, scale=f.K ** -0.5)
    for d in f.members():
        out = sh.view(d, 1024, f.W * f.M, f.N, f.N, dt)
        for i, h in enumerate(f.members()):
            a = sh.view(h, 0, f.M, f.K, f.K, dt).double()
            out[i * f.M:(i + 1) * f.M] = (a @ B.double()).to(dt)
    return f, sh, offs, B


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_check_point_fused(dtype):
    f, sh, offs, B = _fused_heap(dtype)
    assert "within tolerance" in bench.check_point(None, f, sh, offs, B)


def test_check_point_fused_copy_differs():
    f, sh, offs, B = _fused_heap()
    out = sh.view(1, offs["f_out"], f.W * f.M, f.N, f.N, torch.float16)
    out[5, 3] = -out[5, 3] if out[5, 3] != 0 else 1.0
    with pytest.raises(RuntimeError, match="copy differs"):
        bench.check_point(None, f, sh, offs, B)


def test_check_point_fused_value_outside_tolerance():
    f, sh, offs, B = _fused_heap()
    for d in f.members():  # same wrong value in every copy: only the oracle rows catch it
        out = sh.view(d, offs["f_out"], f.W * f.M, f.N, f.N, torch.float16)
        out[f.M + f.M // 2, 7] += 0.25
    with pytest.raises(RuntimeError, match="outside the tolerance"):
        bench.check_point(None, f, sh, offs, B)


@pytest.mark.parametrize("preset", ["largest", "small"])
def test_traffic_entries_cover_the_bench_workloads(preset):
    """bench.py reports each kernel's measured DRAM traffic by looking its
    workload string up in profiles/traffic.json; both presets' workloads must
    have entries (the source hash is checked at run time, not here)."""
    import json
    import os
    g, f = bench.PRESETS[preset]
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as fh:
        t = json.load(fh)
    gather = {e["bench_workload"] for e in t["ag_tma_kernel"]}
    fused = {e["bench_workload"] for e in t["mag2w_kernel" if f.bn == 512 else "mag2_kernel"]}
    assert g.describe() in gather, g.describe()
    assert f.describe() in fused, f.describe()


def test_bench_refuses_the_checked_build():
    """The checked build's bounds checks would make any timing meaningless:
    bench.py stops before loading it."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GEMM_GATHER_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--steps", "1"], cwd=root,
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "not for measurement" in r.stderr, r.stderr
