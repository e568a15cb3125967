"""The N>1 bench path on CPU: two gloo ranks, each an independent replica
with its own seeded batch; whole-job time is the max over ranks and bytes are
summed over ranks.  No GPU and no data-path collective involved."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from paged_kv_cache_172_gb300 import workloads
        # each replica draws its own batch (seed 1 + rank), as bench.py does
        ctx = workloads.llama13b_context_lens(seed=1 + rank)
        step_bytes = bench.decode_bytes(ctx, 38, 40, 128, 16)
        timed = 1.0 + rank          # rank 1 is the slower one
        e2e = 2.0 + 0.5 * rank
        t, e, b = bench.aggregate_ranks(timed, e2e, step_bytes, world, "cpu")
        results[rank] = (t, e, b, step_bytes, int(ctx.sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                       start_method="spawn", join=True)
    r0, r1 = results[0], results[1]
    assert r0[0] == r1[0] == 2.0            # max of the timed regions
    assert r0[1] == r1[1] == 2.5            # max of the end-to-end times
    assert r0[2] == r1[2] == r0[3] + r1[3]  # bytes of both replicas
    assert r0[4] != r1[4]                   # independent batches


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate_ranks(1.5, 2.5, 1000, 1, "cpu") == (1.5, 2.5, 1000.0)
