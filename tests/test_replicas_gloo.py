"""The N > 1 path of bench.py runs independent replicas; its only cross-rank steps are the
barrier, the max of the timed region and the sum of processed tokens.  Checked here with
two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_setup()
    assert (ws, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(ws)
    t = bench.max_over_ranks(10.0 + rank, ws, torch.device("cpu"))
    n = bench.sum_over_ranks(100.0 * (rank + 1), ws, torch.device("cpu"))
    out[rank] = (t, n)
    dist.destroy_process_group()


def test_two_replicas_reduce_time_and_tokens():
    if torch.cuda.is_available():
        pytest.skip("CPU gloo test")
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()   # no fork of this (multi-threaded) process
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == (11.0, 300.0)
