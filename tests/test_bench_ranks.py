"""bench.py's multi-rank path on the CPU: world_size 2 over gloo.  Each rank
times its own replica; the job's time is the max over ranks and its rate
counts every rank's tokens (replicas only: no exchange on the data path)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, ms_local, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.job_rate(ms_local[rank], world, 100, 2, device="cpu")
    finally:
        dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank_and_counts_all_tokens():
    world = 2
    ms_local = [700.0, 760.0]   # 100 steps each
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, _free_port(), ms_local, out), nprocs=world, join=True)
    for r in range(world):
        ms_per_step, value = out[r]
        assert ms_per_step == pytest.approx(7.6)
        assert value == pytest.approx(2 * world / 7.6e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms_per_step, value = bench.job_rate(50.0, 1, 10, 2)
    assert ms_per_step == 5.0 and value == pytest.approx(400.0)


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.main()                     # rank 1 of the reference arm: no work, no output
    assert capsys.readouterr().out == ""


def test_timing_plan_times_exactly_the_asked_steps():
    sys.path.insert(0, ROOT)
    import bench
    for steps, n_rot, passes in [(20, 3, 8), (30000, 3, 8), (2, 3, 8), (24, 3, 8), (25, 3, 8), (100, 64, 1),
                                 (7, 5, 1)]:
        per, reps, rem = bench.timing_plan(steps, n_rot, passes)
        assert reps * per + rem == steps and 0 <= rem < per and reps >= 1
        assert per <= n_rot * passes
        if per < steps:   # several replays: whole passes, so consecutive steps use different copies
            assert per % n_rot == 0
