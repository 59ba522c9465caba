"""The bench's N > 1 path: independent replicas, slowest-rank timing, whole-job value.

Runs two gloo ranks on the CPU (no GPU): each rank reports a different time per step and
the aggregate must use the maximum and count both ranks' work.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    flops = 2.0 * 4096 ** 3
    ms_local = [2.0, 3.0][rank]
    ms, value = bench.aggregate_ranks(ms_local, lambda sec: flops / sec / 1e12, world, dist,
                                      torch.device("cpu"))
    e2e = {"value": 0.0, "unit": "TFLOPS", "h2d_bytes_per_step": 100, "d2h_bytes_per_step": 10,
           "ms_per_step": round(ms_local * 2, 4), "_ms": ms_local * 2}
    e2e = bench.aggregate_e2e(e2e, lambda sec: flops / sec / 1e12, world, dist, torch.device("cpu"))
    out[rank] = (ms, value, e2e)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_uses_slowest_rank_and_total_work():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    flops = 2.0 * 4096 ** 3
    for r in range(world):
        ms, value, e2e = out[r]
        assert ms == 3.0
        assert value == pytest.approx(world * flops / 3e-3 / 1e12)
        # The e2e object is the whole job too: slowest rank's step, both ranks' work and copies.
        assert "_ms" not in e2e and e2e["ms_per_step"] == 6.0
        assert e2e["value"] == pytest.approx(world * flops / 6e-3 / 1e12, abs=1e-3)
        assert e2e["h2d_bytes_per_step"] == 200 and e2e["d2h_bytes_per_step"] == 20


def test_single_rank_aggregate_is_identity():
    import bench
    ms, value = bench.aggregate_ranks(2.5, lambda sec: 1.0 / sec, 1, None, None)
    assert ms == 2.5 and value == pytest.approx(400.0)
    e2e = bench.aggregate_e2e({"value": 1.0, "unit": "x", "h2d_bytes_per_step": 7,
                               "d2h_bytes_per_step": 3, "ms_per_step": 2.5, "_ms": 2.5},
                              lambda sec: 1.0 / sec, 1, None, None)
    assert e2e["value"] == pytest.approx(400.0) and e2e["ms_per_step"] == 2.5
    assert e2e["h2d_bytes_per_step"] == 7 and e2e["d2h_bytes_per_step"] == 3
    assert bench.aggregate_e2e(None, lambda sec: 1.0, 1, None, None) is None
