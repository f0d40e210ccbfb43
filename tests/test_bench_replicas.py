"""The benchmark's multi-GPU path is N independent replicas ("replicas only"):
each rank times its own step, the job takes the slowest rank's time, and the
value sums the replicas' work.  This checks that logic on 2 gloo CPU ranks
(no GPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        mine = 1.5 + rank  # rank 1 is the slow one
        worst = bench.max_over_ranks(mine)
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(repr(worst))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks(tmp_path):
    mp.start_processes(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"r{r}").read_text()) == 2.5


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_whole_job_value_sums_replicas():
    import bench
    one = bench.whole_job_value(0.5e-3, 1.0, 1)
    assert one == pytest.approx(50.0)
    assert bench.whole_job_value(0.5e-3, 1.0, 4) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the reference arm (the oracle on the host cores) runs on
    rank 0 alone; any other rank exits 0 at once without output."""
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 3, 3, 2

    peaks, src = bench.load_peaks()
    assert bench.run_reference(Args(), peaks, src, bench.GATHER, bench.FUSED) == 0
    assert capsys.readouterr().out == ""
