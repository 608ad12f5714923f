"""The multi-rank host logic of bench.py (one replica per GPU, no collective on
the data path): the max over ranks of the timings and the whole-job rate, run
as two gloo ranks on CPU."""
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


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank timed its own replica; the slowest decides
        step_s, other = 1.0 + rank, 5.0 - rank
        got = bench.reduce_max([step_s, other], torch.device("cpu"), dist)
        rate = bench.whole_job_rate(1000, world, 10, got[0])
        out[rank] = (got, rate)
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        got, rate = out[rank]
        assert got == [2.0, 5.0]                  # max over ranks, elementwise
        assert rate == pytest.approx(1000 * 2 * 10 / 2.0)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max([3.0, 4.0], torch.device("cpu"), None) == [3.0, 4.0]
    assert bench.whole_job_rate(16388, 1, 200, 0.0312) == pytest.approx(16388 * 200 / 0.0312)
    # byte models used for the roofline
    assert bench.prefill_bytes(4, 16, 4096, 128, 128) == 276889600
    assert bench.decode_bytes(256, 16, 128, 128) == 545259520
    # LA "固定大小的状态也可能不小": 32 layers x 16 heads of FP32 state at r = dv = 128
    assert 32 * 16 * 4 * (128 * 128 + 128) == 33816576
