"""The N>1 path of bench.py: independent replicas, max over ranks, no data
collective.  Run as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    local_ms = [0.30, 0.45][rank]
    mean_ms, value = bench.aggregate_over_ranks(local_ms, 1_000_000_000, ws, device="cpu")
    results[rank] = (mean_ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(world, port, results), nprocs=world, start_method="spawn")
        res = dict(results)
    for rank in range(world):
        mean_ms, value = res[rank]
        assert mean_ms == pytest.approx(0.45)
        # two replicas each moved 1 GB in 0.45 ms
        assert value == pytest.approx(2 * 1e9 / 0.45e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    mean_ms, value = bench.aggregate_over_ranks(0.5, 2_000_000_000, 1)
    assert mean_ms == 0.5 and value == pytest.approx(4000.0)
