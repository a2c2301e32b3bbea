"""One rank of the world-size-2 gloo test of bench.py's replica aggregation
(run in a spawned process)."""
import os


def run(rank, world, port, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank prefill ms, decode ms, wall s: rank 1 is slower in two of them
        mine = [100.0 + 20.0 * rank, 400.0 - 50.0 * rank, 1.5 * (rank + 1)]
        got = bench.max_over_ranks(mine, world, "cpu")
        rate = bench.job_rate(world, 128 * 5, got[1])
        out_q.put((rank, got, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()
