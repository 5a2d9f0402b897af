"""The benchmark's multi-rank host logic with world_size 2 on the gloo backend (CPU): every
rank joins, the time reported is the maximum over ranks, barriers pass, and the reference
arm does no work on ranks other than 0."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import argparse
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    w, r, _ = bench.dist_setup(world, backend="gloo")
    assert (w, r) == (world, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w)
    if rank != 0:
        args = argparse.Namespace(gpus=world, steps=3, warmup=3, shape="prefill")
        out[10 + rank] = bench.run_reference(args)  # returns at once, no work
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 2.5
    assert out[11] == 0
