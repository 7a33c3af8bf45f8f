"""The benchmark's N > 1 logic on CPU: two gloo ranks, each with its own timed length, agree on the
slowest one, and the whole-job throughput counts every rank's full batch (weak scaling).  The
reference arm's other ranks do no work, and its rank 0 prints one line of the benchmark contract."""
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


def test_reference_arm_prints_one_contract_line():
    """The reference arm (the oracle on the host cores) at N = 1: one JSON line carrying the keys the
    benchmark contract names, the throughput consistent with the step time, no transfers counted."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "reindex_decode_r2"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # tokens per step over the step time (the sample is one token of one layer)
    assert d["value"] == pytest.approx(1000.0 / d["ms_per_step"], rel=1e-6)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
