"""bench.py's multi-rank host logic on the CPU: two ranks over gloo.

With N GPUs the benchmark runs one replica of the workload per rank (no exchange
step in a GEMM), takes the slowest rank's elapsed time and reports the work of all
ranks over it.  Here each rank is a CPU process; the elapsed times are planted.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 25.0 * rank            # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, dist)
        e2e_s = bench.max_over_ranks(0.5 * (rank + 1), dist)
        dist.barrier()
        q.put((rank, job_ms, e2e_s))
    finally:
        dist.destroy_process_group()


def _run_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_ranks_take_the_slowest_time():
    out = _run_ranks(2)
    assert [r for r, _, _ in out] == [0, 1]
    for _, job_ms, e2e_s in out:
        assert job_ms == pytest.approx(125.0)     # every rank sees the slowest rank's time
        assert e2e_s == pytest.approx(1.0)


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # Four 8192^3 GEMMs per step, 10 steps per rank, 2 ranks, 125 ms for the slowest.
    flops_rank = 4 * 2.0 * 8192 ** 3 * 10
    assert bench.job_tflops(flops_rank, 2, 0.125) == pytest.approx(2 * flops_rank / 0.125 / 1e12)
    assert bench.max_over_ranks(7.5) == 7.5      # one rank: no collective


def test_rank_environment_and_config(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_info() == (1, 2, 1)
    assert bench.workload_config(2)["parallelism"] == "replicas2"


def test_reference_arm_other_ranks_do_no_work(capsys):
    """Only rank 0 times the oracle and prints; the other ranks return at once."""
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 2, 1

    bench.bench_reference(Args(), rank=1, world=2)
    assert capsys.readouterr().out == ""
