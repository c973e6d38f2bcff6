"""The benchmark's multi-rank host logic on CPU: two gloo ranks, max-over-ranks
timing and whole-job throughput (the attention path itself needs no exchange
between GPUs; ranks are independent replicas)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [0.5, 0.8][rank]
        total = bench.aggregate_ranks(local, world, bench.make_reduce_max(dist, "cpu"))
        out[rank] = (total, bench.job_throughput(world, 10, 1e12, total))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of a multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(0.8) and res[1][0] == pytest.approx(0.8)
    # 2 ranks x 10 steps x 1 TFLOP in 0.8 s
    assert res[0][1] == pytest.approx(25.0)


def test_single_rank_is_identity():
    import bench

    assert bench.aggregate_ranks(1.25, 1, None) == 1.25
    assert bench.job_throughput(1, 4, 2.5e11, 1.0) == pytest.approx(1.0)
