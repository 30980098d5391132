"""bench.py's multi-rank aggregation on CPU (gloo, world size 2): the job's
time is the slowest rank's, and throughput counts every rank's batch. The
hot path itself needs no collective (each rank runs its own batch), so this
host logic is all that N > 1 adds."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as tdist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [40.0, 55.5][rank]
        ms = bench.max_over_ranks(local_ms)
        out[rank] = (ms, bench.job_tokens_per_s(world, 2048, 20, ms))
        tdist.barrier()
    finally:
        tdist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    for rank in (0, 1):
        ms, tps = out[rank]
        assert ms == 55.5
        assert tps == pytest.approx(2 * 2048 * 20 / 55.5e-3)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_tokens_per_s(1, 100, 10, 1000.0) == pytest.approx(1000.0)
