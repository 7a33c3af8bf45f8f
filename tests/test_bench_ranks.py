"""The benchmark's N > 1 logic on CPU: two gloo ranks, each with its own timed length, agree on the
slowest one, and the whole-job throughput counts every rank's full batch (weak scaling).  The
reference arm's other ranks do no work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        got = bench.max_over_ranks(ms, dist, "cpu")
        out[rank] = (got, bench.job_tokens_per_s(world, 32, 1, 4, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 15.0
    # 2 ranks x 32 tokens x 1 layer x 4 steps in 15 ms
    assert out[0][1] == pytest.approx(2 * 32 * 4 / 0.015)


def test_single_rank_is_its_own_time():
    import bench
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.job_tokens_per_s(1, 32, 4, 10, 20.0) == pytest.approx(32 * 4 * 10 / 0.02)


def test_reference_arm_other_ranks_do_nothing(capsys):
    import bench
    ns = type("A", (), dict(workload="reindex_decode_r2", steps=1, warmup=0))()
    assert bench.run_reference(ns, 1, 2) is None
    assert capsys.readouterr().out == ""
