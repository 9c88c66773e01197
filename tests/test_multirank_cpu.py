"""The multi-rank path of bench.py on CPU: two gloo ranks, each timing its own
replica, agree on the maximum (the only cross-rank exchange)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench

    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 5.0 - rank, float(rank)]
        out[rank] = bench.reduce_max(mine, world, "cpu")
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_rank_max_reduction():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    assert out[0] == out[1] == [11.0, 5.0, 1.0]


def test_single_rank_is_identity():
    import bench

    assert bench.reduce_max([1.0, 2.0], 1, "cpu") == [1.0, 2.0]
