"""Host logic of bench.py's multi-process path on CPU: two gloo ranks take the
max of their step times and report one whole-job µs/call.  The matmul itself
has no cross-GPU exchange (replicas), so this is the only N>1 logic."""
import os
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        got = bench.max_over_ranks(ms)
        out[rank] = got
        out[world + rank] = bench.job_value_us(got, world, steps=4, ncalls=14)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world = 2
    out = mp.get_context("spawn").Array("d", 2 * world)
    ctx = mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert list(out[:world]) == [15.0, 15.0]
    assert out[world] == pytest.approx(15.0 * 1e3 / (2 * 4 * 14))
    assert out[world] == out[world + 1]


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value_us(28.0, 1, 2, 14) == pytest.approx(1000.0)
