"""The N > 1 host path of bench.py on CPU: two gloo ranks, each an independent
replica, joined only by the barrier and the max-over-ranks timing."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    ws, r, local, dist = bench.dist_setup(None, backend="gloo")
    try:
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(dist)
        local_ms = 1.0 + rank                       # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, dist)
        gbs = bench.aggregate_gbs(1e9, ms, ws)
        out[rank] = (ms, gbs)
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_work():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1]
    ms, gbs = out[0]
    assert ms == 2.0                                # the slowest rank bounds the step
    assert gbs == pytest.approx(world * 1e9 / 2e-3 / 1e9)


def test_single_process_has_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    ws, r, local, dist = bench.dist_setup(None)
    assert (ws, r, local, dist) == (1, 0, 0, None)
    assert bench.max_over_ranks(3.5, None) == 3.5
