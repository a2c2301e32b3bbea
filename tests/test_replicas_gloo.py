"""bench.py's multi-GPU path is replicas only: N independent copies of the
step, a barrier around the timed region, the slowest rank's time, and the
whole job's units over it.  The aggregation runs here as two gloo ranks on
the CPU; the reference arm's extra ranks return without work."""
import argparse
import multiprocessing as mp
import socket

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
