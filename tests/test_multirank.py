"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with its
own step time, agree on the slowest rank's time and on the whole-job
throughput (every rank's tokens over that time).  The data path has no
collective: only the timing is reduced."""
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


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    step_ms = [0.100, 0.130][rank]
    slow = bench.slowest_rank_ms(step_ms, world, torch.device("cpu"))
    value = bench.job_tokens_per_s(world, 32768, slow)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slow, value))


def test_two_gloo_ranks_agree_on_slowest_time_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, value in out:
        assert slow == pytest.approx(0.130)
        assert value == pytest.approx(2 * 32768 / 0.130e-3)


def test_single_rank_is_the_identity():
    import bench
    assert bench.slowest_rank_ms(0.25, 1, torch.device("cpu")) == 0.25
    assert bench.job_tokens_per_s(1, 1000, 1.0) == pytest.approx(1e6)
