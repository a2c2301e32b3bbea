"""bench.py's multi-GPU path is replicas only: N independent copies of the
step, a barrier around the timed region, the slowest rank's time, and the
whole job's units over it.  The aggregation runs here as two gloo ranks on
the CPU; the reference arm's extra ranks return without work."""
import argparse
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import bench
import replica_worker


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_slowest_rank_time_and_whole_job_rate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=replica_worker.run, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, (got, rate)) for r, got, rate in (q.get(timeout=180) for _ in procs))
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    want = [120.0, 400.0, 3.0]                 # each value's maximum over the two ranks
    for r in (0, 1):
        got, rate = res[r]
        assert got == want
        assert rate == 2 * 128 * 5 / 0.4       # both ranks' tokens over the slowest decode time


def test_single_rank_keeps_its_own_values():
    assert bench.max_over_ranks([1.0, 2.5, 3.0], 1, "cpu") == [1.0, 2.5, 3.0]
    assert bench.job_rate(1, 640, 1000.0) == 640.0


def test_reference_arm_runs_on_rank_zero_only():
    args = argparse.Namespace(workload="llama8b", steps=1, warmup=0)
    assert bench.run_reference(args, rank=1, world=2) is None


def test_gpus_n_outside_torchrun_starts_n_ranks():
    """bench.py --gpus N started without torchrun re-runs itself as N ranks
    under torchrun on 127.0.0.1: the launcher runs a gloo worker as two
    ranks, each sees WORLD_SIZE 2 and its own rank, and the arguments pass
    through."""
    here = os.path.dirname(os.path.abspath(__file__))
    cmd = bench.replica_command(2, ["--steps", "3"], os.path.join(here, "launcher_worker.py"), _free_port())
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=2" in cmd
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=240)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = sorted(l for l in out.stdout.splitlines() if l.startswith("rank "))
    assert lines == ["rank 0 of 2 local 0 sum 1 argv --steps 3", "rank 1 of 2 local 1 sum 1 argv --steps 3"]


def test_bench_main_launches_replicas_when_not_under_torchrun(monkeypatch):
    seen = {}

    def fake_launch(n, argv, script=None):
        seen["n"], seen["argv"] = n, list(argv)
        return 0
    monkeypatch.setattr(bench, "launch_replicas", fake_launch)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4", "--steps", "2"])
    try:
        bench.main()
    except SystemExit as e:
        assert e.code == 0
    assert seen == {"n": 4, "argv": ["--gpus", "4", "--steps", "2"]}
