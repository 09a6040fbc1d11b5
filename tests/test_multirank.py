"""The bench's multi-process path on CPU: two gloo ranks on 127.0.0.1.

Each rank of a multi-GPU run owns its own replica of the workload (the path
has no exchange step); the only cross-rank operations are the barriers around
the timed region and the max-over-ranks of its duration, which are checked
here without a GPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    slowest = bench.max_over_ranks(10.0 * (rank + 1), world)
    bench.barrier(world)

    class Args:
        workload, steps, warmup, gpus = "decode", 1, 3, world
    ran = bench.run_reference(Args, world, rank) if rank != 0 else "rank0"
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{slowest} {ran}")
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        slowest, ran = open(tmp_path / f"r{r}.txt").read().split()
        assert float(slowest) == 20.0
        if r != 0:
            assert ran == "None"  # non-zero ranks print nothing for the reference arm
