"""The multi-GPU path shards requests across ranks with no collective on the
data path (weak scaling) and takes the maximum of the ranks' timed region.
Its host-side logic runs here as two gloo ranks on CPU."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ids = bench.shard_request_ids(8, rank)
    gathered = [None] * world
    dist.all_gather_object(gathered, ids)
    ms_local = [10.0 + 5.0 * rank, 20.0 - rank]  # rank 1 is slower on the first timer
    ms, value = bench.aggregate(ms_local, world, 2048, 100, dist, "cpu")
    out[rank] = (gathered, ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_aggregate():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    g0, ms0, v0 = out[0]
    g1, ms1, v1 = out[1]
    # request ids are disjoint and cover both replicas
    assert sorted(g0[0] + g0[1]) == list(range(16)) and not set(g0[0]) & set(g0[1])
    # max over ranks, identical on every rank
    assert ms0 == ms1 == [15.0, 20.0]
    # whole-job throughput counts both ranks' positions
    assert v0 == v1 == pytest.approx(2 * 2048 * 100 / 0.015)
