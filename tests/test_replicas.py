"""The multi-GPU path of bench.py is replicas only: each rank runs its own copy of
the workload and rank 0 reports the units of all ranks over the slowest rank's
time. Its host side runs here on two gloo ranks on the CPU."""
import io
import contextlib
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        step_s = 0.010 + 0.005 * rank             # rank 1 is the slower replica
        slowest = bench.max_over_ranks(step_s)
        rate = bench.whole_job_rate(32, world, slowest)
        # the reference arm prints on rank 0 only; other ranks return without work
        os.environ["RANK"] = str(rank)
        buf = io.StringIO()
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                bench.run_reference(bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
        out[rank] = (slowest, rate, buf.getvalue())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_report_the_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()   # no fork of a multi-threaded process
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        slowest, rate, printed = out[r]
        assert slowest == pytest.approx(0.015)
        assert rate == pytest.approx(32 * 2 / 0.015)
    assert out[1][2] == ""


def test_single_process_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.whole_job_rate(1, 1, 0.5) == 2.0
