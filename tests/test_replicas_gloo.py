"""The multi-process path of bench.py, on CPU with two gloo ranks: every
replica ends with the slowest rank's times (so the reported whole-job value is
all ranks' units over that time), and a single process passes its values
through."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.0 + rank, 10.0 - rank]          # rank 1 is slower on the first, faster on the second
        out[rank] = bench.max_over_ranks(torch, local, "cpu")
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        got = dict(out)
    assert got[0] == got[1] == [2.0, 10.0]


def test_max_over_ranks_single_process():
    assert not torch.distributed.is_initialized()
    assert bench.max_over_ranks(torch, [3.5, 1.25], "cpu") == [3.5, 1.25]
