"""The N > 1 path of bench.py on CPU: world_size 2 over gloo, 127.0.0.1.

With several GPUs every rank runs its own replica of the step (the operations
have no data-path collective on one GPU each); the ranks meet only at the
barriers around the timed region and in the max-reduce of their step times.
These tests run that host logic in two processes: both ranks must see the
slower rank's time, the whole-job value must count every replica's work over
that time, and the reference arm must leave ranks other than 0 idle.
"""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        local_ms = 1.0 + 0.5 * rank             # rank 1 is the slower one
        slowest = bench.max_over_ranks(local_ms, world)
        value = bench.job_tflops(2.0e12, world, slowest)
        bench.barrier(world)
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_the_job_value():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in results] == [0, 1]
    for _, slowest, value in results:
        assert slowest == 1.5
        # two replicas of 2e12 FLOP each over 1.5 ms
        assert value == pytest.approx(2 * 2.0e12 / 1.5e-3 / 1e12)


def test_single_rank_value_and_max_are_local():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_tflops(1.0e12, 1, 2.0) == pytest.approx(500.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"])
    args = bench.parse_args()
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
