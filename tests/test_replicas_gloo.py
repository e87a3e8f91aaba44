"""The benchmark's multi-process path on CPU: under torchrun every rank runs
an independent replica (decode attention has no cross-GPU exchange), and the
reported time is the slowest rank's. Two gloo ranks check that reduction."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        out = manager.dict()
        mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        result = dict(out)
    assert result == {0: 15.0, 1: 15.0}


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
