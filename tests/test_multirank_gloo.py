"""Host-side multi-rank logic of bench.py, on CPU with the gloo backend.

Weak scaling: every rank builds its own full-size batch (same shapes, its own
seed), times its own steps, and rank 0 reports the max time over ranks; no
collective touches the attention data.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from paged_kv_cache_95_gb300 import workloads as W
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist = bench.init_dist(ws, "gloo")
    try:
        bench.barrier(dist)
        t = bench.max_over_ranks(1.0 + rank, dist)          # rank-local "elapsed time"
        wl = W.shard_for_rank("tiny", rank, world)
        results[rank] = (t, wl.decode.q.tobytes(), wl.decode.context_lens.tolist(), wl.k_cache.shape)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_weak_scaling_host_logic():
    world = 2
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn", join=True)
    (t0, q0, lens0, shape0), (t1, q1, lens1, shape1) = results[0], results[1]
    assert t0 == t1 == 2.0                 # max over ranks seen by every rank
    assert lens0 == lens1 and shape0 == shape1  # same shapes on every rank (weak scaling)
    assert q0 != q1                        # but each rank draws its own data


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5
    bench.barrier(None)
