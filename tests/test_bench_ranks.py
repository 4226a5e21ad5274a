"""The multi-rank path of bench.py on CPU: two gloo ranks, max of the elapsed
times and sum of the token counts (the only numbers ranks exchange)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, tokens = bench.reduce_over_ranks(10.0 + 5.0 * rank, 100.0 * (rank + 1),
                                         torch.device("cpu"))
    out[rank] = (ms, tokens)
    dist.destroy_process_group()


def test_two_ranks_max_time_sum_tokens():
    world, port = 2, _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        assert out[0] == out[1] == (15.0, 300.0)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    assert bench.reduce_over_ranks(3.5, 7, torch.device("cpu")) == (3.5, 7.0)
