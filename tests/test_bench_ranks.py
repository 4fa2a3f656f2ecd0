"""bench.py's multi-process path (one process per GPU, replicas): the job's
time is the slowest rank's and the value counts every rank's work.  Checked
with two gloo ranks on CPU; the GPU measurement itself is not involved."""
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        q.put((rank, ms, bench.whole_job_tflops(1e12, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_both():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), q), nprocs=world, join=True, start_method="spawn")
    got = sorted(q.get() for _ in range(world))
    for rank, ms, tflops in got:
        assert ms == 5.0
        assert tflops == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(7.0, 1, "cpu") == 7.0
    assert bench.whole_job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)
