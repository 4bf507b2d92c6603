"""The N > 1 launch of bench.py on CPU: two gloo ranks (127.0.0.1).  The layer
shards by sequence and head with no exchange, so N GPUs run N replicas; what
the ranks share is the barrier around the timed region, the slowest rank's
time, and the reference arm, which rank 0 alone runs and prints."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import importlib.util
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    bench._barrier(world)
    slowest = bench._max_over_ranks(10.0 * (rank + 1), world)

    class Args:
        steps, warmup = 1, 0

    ref = bench.run_reference(Args, rank, world) if rank != 0 else "rank 0 runs the oracle"
    out[rank] = (slowest, ref)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == 20.0 and res[1][0] == 20.0       # max over ranks
    assert res[1][1] is None                              # only rank 0 runs the reference arm
