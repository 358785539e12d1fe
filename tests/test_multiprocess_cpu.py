"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each with its own replica.

Each rank reports its own step time; the job's time is the slowest rank's and the job's
throughput counts the tokens of every rank (weak scaling: no data-path collective, the
only collective is the timing reduction).
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [1.5, 2.25][rank]
        slow = bench.slowest_ms(my_ms, world, torch.device("cpu"))
        val = bench.job_tokens_per_s(1000, world, slow)
        out[rank] = (slow, val)
        tdist.barrier()
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_tokens():
    world, port = 2, _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        slow, val = res[rank]
        assert slow == 2.25
        assert val == pytest.approx(2 * 1000 / 2.25e-3)


def test_single_process_is_its_own_slowest():
    assert bench.slowest_ms(3.0, 1, None) == 3.0
    assert bench.job_tokens_per_s(10, 1, 2.0) == pytest.approx(5000.0)
