"""The multi-GPU bench path on CPU: two gloo ranks (127.0.0.1) stand for two
replicas.  The step time is the slowest rank's, the rate counts every rank's
cells, and the reference arm runs on rank 0 alone."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r took 10 + 5 r ms over 5 steps of 1,000 cells each
        ms_step, rate, w = bench.job_timing(10.0 + 5.0 * rank, 5, 1000)
        # the reference arm: rank 0 alone prints; the others return at once
        os.environ["RANK"], os.environ["WORLD_SIZE"] = str(rank), str(world)
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})())
        dist.barrier()
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{ms_step} {rate} {w} {len(buf.getvalue())}\n")
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_reference_arm(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        ms_step, rate, w, printed = open(tmp_path / f"r{r}.txt").read().split()
        assert float(ms_step) == pytest.approx(15.0 / 5)          # the slower rank's time
        assert float(rate) == pytest.approx(2 * 1000 / 3e-3)      # both ranks' cells
        assert int(w) == 2
        if r != 0:
            assert int(printed) == 0                               # reference arm: rank 0 only


def test_single_process_timing():
    sys.path.insert(0, ROOT)
    import bench
    ms_step, rate, w = bench.job_timing(20.0, 4, 500)
    assert (ms_step, w) == (5.0, 1)
    assert rate == pytest.approx(500 / 5e-3)
