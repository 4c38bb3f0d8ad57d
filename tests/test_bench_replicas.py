"""The N>1 path of bench.py (independent replicas, one per rank) on CPU:
two gloo ranks, each with its own time and tokens; the whole-job value must
be all tokens over the slowest rank's time, identical on both ranks."""
import os
import socket

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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [100.0, 250.0][rank]
    value, ms, tokens = bench.aggregate_replicas(local_ms, 131072 * 5, world)
    out[rank] = (value, ms, tokens)
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    value, ms, tokens = out[0]
    assert ms == 250.0 and tokens == 2 * 131072 * 5
    assert value == pytest.approx(2 * 131072 * 5 / 0.25)


def test_replica_aggregation_single_rank_is_local():
    import bench
    assert bench.aggregate_replicas(200.0, 1000, 1) == (5000.0, 200.0, 1000)
