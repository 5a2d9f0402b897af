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


def _qb_worker(rank, world, port, out):
    """Each rank holds one part of a batch; the candidate exchange must let every rank see
    the whole batch's k-th largest logit per expert.  The candidates are made here with
    torch.topk (the library's own candidate kernel is checked on the GPU)."""
    import sys
    import torch
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from latent_compressed_expert_gb300 import lmoe
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    T_parts, E, K = [300, 724], 64, 8
    full = torch.randn(sum(T_parts), E, generator=torch.Generator().manual_seed(5))
    t0 = sum(T_parts[:rank])
    part = full[t0:t0 + T_parts[rank]]
    Tg = lmoe.global_token_count(part.shape[0], "cpu")
    k = lmoe.fair_share_rank(Tg, K, E)
    cand = torch.topk(part, k, dim=0).values
    stacked = lmoe.gather_candidates(cand)
    kth = torch.topk(stacked, k, dim=0).values[-1]
    ref = torch.topk(full, k, dim=0).values[-1]
    out[rank] = (Tg, k, tuple(stacked.shape), bool(torch.equal(kth, ref)),
                 bool(torch.equal(stacked[rank * k:(rank + 1) * k], cand)))
    dist.barrier()
    dist.destroy_process_group()


def test_threshold_candidate_exchange_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_qb_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        Tg, k, shape, same_kth, in_place = out[r]
        assert Tg == 1024 and k == 128 and shape == (2 * k, 64)
        assert same_kth and in_place
