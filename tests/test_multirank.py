"""Multi-rank host logic of bench.py on CPU: two gloo ranks (no GPU).

Each rank draws an independent batch (distinct input seeds) and the step time
is the maximum over ranks.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from workloads import WORKLOADS, row_tokens
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist_env()
        assert (ws, r, local) == (world, rank, rank)
        t = bench.max_over_ranks(10.0 * (rank + 1), dist)
        w = WORKLOADS["tiny"]
        q, _, _ = row_tokens(w, bench.rank_layer_seed(rank), 0, 0)
        out[rank] = (t, int(q[:4].astype("int64").sum()))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_independent_inputs():
    world = 2
    port = _free_port()
    mgr = tmp.get_context("spawn").Manager()
    out = mgr.dict()
    tmp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                        start_method="spawn")
    assert out[0][0] == out[1][0] == 20.0
    assert out[0][1] != out[1][1]


def test_single_rank_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
