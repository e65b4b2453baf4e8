"""Multi-rank host logic on CPU: two gloo ranks reduce their step times to the
slowest one and agree on the weak-scaling aggregate."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_deltanet_prefill_gb300 import dist as gdist


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = gdist.rank_world()
    ms = 10.0 + 5.0 * r                       # rank 1 is the slower one
    slow = gdist.max_over_ranks(ms)
    val = gdist.aggregate_throughput(131072, w, slow)
    seeds = [None] * w
    dist.all_gather_object(seeds, gdist.rank_seed(5, r))
    out[rank] = (r, w, lr, slow, val, tuple(seeds))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert set(out.keys()) == {0, 1}
    for rank in (0, 1):
        r, w, lr, slow, val, seeds = out[rank]
        assert (r, w, lr) == (rank, 2, rank)
        assert slow == 15.0
        assert val == pytest.approx(2 * 131072 / 15e-3)
        assert len(set(seeds)) == 2


def test_single_process_identity():
    assert gdist.max_over_ranks(3.5) == 3.5
    assert gdist.rank_seed(5, 0) == 5
