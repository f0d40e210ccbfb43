"""The oracle's all-gather against torch.distributed.all_gather_into_tensor on
W CPU processes over gloo (the library routine the pages' own tests compare
with: iris #594 "Multi-GPU CI" and "Local validation"), for a contiguous group
and a strided subgroup, and its all-to-all with all_to_all_single.  CPU only;
no GPU is touched."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import gg_inputs
from tests import heap_image as hi


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _block(h, M, N):
    g = gg_inputs.generator(100 + h)
    return gg_inputs.normal((M, N), torch.float32, g)


def _worker(rank, world, port, M, N, sub_ranks, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        x = _block(rank, M, N)
        out = torch.empty((world * M, N), dtype=torch.float32)
        dist.all_gather_into_tensor(out, x)
        np.save(os.path.join(out_dir, f"full_{rank}.npy"), out.numpy())
        # all_to_all_single with equal splits: rank r's input is W blocks
        xa = torch.cat([_block(100 * rank + j, M, N) for j in range(world)])
        oa = torch.empty_like(xa)
        dist.all_to_all_single(oa, xa)
        np.save(os.path.join(out_dir, f"a2a_{rank}.npy"), oa.numpy())
        grp = dist.new_group(ranks=sub_ranks)
        if rank in sub_ranks:
            o2 = torch.empty((len(sub_ranks) * M, N), dtype=torch.float32)
            dist.all_gather_into_tensor(o2, x, group=grp)
            np.save(os.path.join(out_dir, f"sub_{rank}.npy"), o2.numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,M,N,sub", [(4, 5, 7, (1, 2, 2)), (3, 3, 16, (0, 2, 2))])
def test_oracle_matches_gloo_all_gather(oracle, tmp_path, world, M, N, sub):
    start, stride, Wsub = sub
    sub_ranks = [start + i * stride for i in range(Wsub)]
    mp.start_processes(_worker, args=(world, _free_port(), M, N, sub_ranks, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    # full group
    lay = hi.make_layout(world, world, M, N, 4)
    heap = hi.sentinel_heap(lay)
    for h in range(world):
        hi.put_block(heap, lay, h, _block(h, M, N).numpy(), lay.in_off, lay.ld_in)
    oracle.all_gather(heap, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out,
                      M, N, 4, (0, 1, world))
    for h in range(world):
        ref = np.load(tmp_path / f"full_{h}.npy")
        got = hi.get_block(heap, lay, h, lay.out_off, world * M, lay.ld_out, N, np.float32)
        assert got.tobytes() == ref.tobytes()
    # all-to-all with equal splits
    lay = hi.make_layout(world, world, world * M, N, 4)
    heap = hi.sentinel_heap(lay)
    for h in range(world):
        xa = torch.cat([_block(100 * h + j, M, N) for j in range(world)]).numpy()
        hi.put_block(heap, lay, h, xa, lay.in_off, lay.ld_in)
    oracle.all_to_all(heap, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out, M, N,
                      4, (0, 1, world))
    for h in range(world):
        ref = np.load(tmp_path / f"a2a_{h}.npy")
        got = hi.get_block(heap, lay, h, lay.out_off, world * M, lay.ld_out, N, np.float32)
        assert got.tobytes() == ref.tobytes()
    # strided subgroup
    lay = hi.make_layout(world, Wsub, M, N, 4)
    heap = hi.sentinel_heap(lay)
    for h in range(world):
        hi.put_block(heap, lay, h, _block(h, M, N).numpy(), lay.in_off, lay.ld_in)
    oracle.all_gather(heap, lay.part_bytes, lay.in_off, lay.ld_in, lay.out_off, lay.ld_out,
                      M, N, 4, sub)
    for h in sub_ranks:
        ref = np.load(tmp_path / f"sub_{h}.npy")
        got = hi.get_block(heap, lay, h, lay.out_off, Wsub * M, lay.ld_out, N, np.float32)
        assert got.tobytes() == ref.tobytes()
