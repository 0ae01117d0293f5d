"""The multi-process path of bench.py on the CPU (gloo, two ranks).

One process per GPU runs its own replica of the workload; the job's timed span
is the maximum over ranks and its value sums every rank's tokens.  The GPU
kernels are not involved here: this covers the host-side rank handling.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, local_ms, units, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench  # noqa: E402
    w, r, _ = bench._dist()  # initialises the gloo group from the environment
    assert (w, r) == (world, rank)
    total_ms, value = bench.aggregate_ranks(local_ms[rank], units, world, torch.device("cpu"))
    out[rank] = (total_ms, value)
    # the reference arm runs on rank 0 only; the other ranks do no work
    if rank != 0:
        args = type("A", (), {"workload": "tiny", "steps": 1, "warmup": 0})()
        assert bench.run_reference(args, world, rank) is None
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_max_time_and_summed_value():
    world, units = 2, 1000
    local_ms = [2.0, 5.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), local_ms, units, out), nprocs=world, join=True)
        for rank in range(world):
            total_ms, value = out[rank]
            assert total_ms == pytest.approx(5.0)  # the slowest rank's span
            assert value == pytest.approx(world * units / 5e-3)


def test_single_rank_needs_no_group():
    import bench
    total_ms, value = bench.aggregate_ranks(4.0, 500, 1, torch.device("cpu"))
    assert total_ms == 4.0 and value == pytest.approx(500 / 4e-3)
