"""The N>1 host path of bench.py on CPU: two gloo ranks, each with its own
heads (different seeds), agree on the slowest rank's time and on the
whole-job throughput. No GPU and no collective on the data path."""

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


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from exact_attention_64_gb300.workloads import make_inputs

        my_ms = 10.0 + 5.0 * rank
        ms = bench.slowest_rank_ms(my_ms, dist, "cpu")
        tf = bench.job_tflops(1e12, world, 4, ms)
        q, _, _, _ = make_inputs(1, 1, 8, 4, torch.float32, seed=rank)
        out[rank] = (ms, tf, float(q.sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    (ms0, tf0, q0), (ms1, tf1, q1) = out[0], out[1]
    assert ms0 == ms1 == 15.0
    assert tf0 == tf1 == pytest.approx(1e12 * 2 * 4 / 15e-3 / 1e12)
    assert q0 != q1  # each rank draws its own heads
