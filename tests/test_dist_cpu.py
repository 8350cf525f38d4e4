"""The replicated (N > 1) benchmark path on the CPU with two gloo ranks: each
rank builds its own seeded batch (different from the other rank's), and the
whole-job figures are the slowest rank's time and the work of all ranks
together."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads
        from paged_kv_cache_143_gb300 import accounting
        assert bench.dist_env() == (rank, world, rank)
        w = workloads.make(2, device="cpu", sub=rank, num_requests=8)
        kv = accounting.decode_kv_bytes(w.seq_lens, w.Hkv, w.D, w.elt_bytes)
        times = (1.0 + rank, 5.0 - rank)  # rank 1 slower on the first, faster on the second
        (t0, t1), total = bench.combine_ranks(times, kv, world, "cpu")
        seqs = [None] * world
        dist.all_gather_object(seqs, w.seq_lens.tolist())
        kvs = [None] * world
        dist.all_gather_object(kvs, int(kv))
        out[rank] = dict(t=(t0, t1), total=total, kvs=kvs, seqs=seqs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_combine_max_time_and_summed_work():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    r0, r1 = out[0], out[1]
    assert r0["t"] == r1["t"] == (2.0, 5.0)                 # max over ranks, each time
    assert r0["total"] == r1["total"] == sum(r0["kvs"])      # summed over ranks
    assert r0["seqs"][0] != r0["seqs"][1]                    # each rank its own batch
    assert r0["kvs"][0] != r0["kvs"][1]


def test_single_rank_is_the_identity():
    import bench
    assert bench.combine_ranks((3.0, 4.0), 123, 1, "cpu") == ([3.0, 4.0], 123.0)
