"""A stand-in for bench.py under the replica launcher: each rank joins a
gloo group from the environment torchrun sets, sums its rank over the group
and prints one line (run as a script by tests/test_replicas_gloo.py)."""
import os
import sys

import torch
import torch.distributed as dist


def main():
    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    dist.init_process_group("gloo")
    t = torch.tensor([float(rank)])
    dist.all_reduce(t)
    line = f"rank {rank} of {world} local {os.environ['LOCAL_RANK']} sum {int(t.item())} argv {' '.join(sys.argv[1:])}\n"
    os.write(1, line.encode())        # one write, so the ranks' lines never interleave
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
