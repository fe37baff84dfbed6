"""The multi-GPU path is replicas only: every rank runs the whole per-GPU workload on its
own tokens, and the job's time is the slowest rank's.  The host logic of that path
(max over ranks, whole-job tokens/s) runs here on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_ms, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total = bench.max_over_ranks(local_ms[rank], world, torch.device("cpu"))
    q.put((rank, total, bench.job_tokens_per_s(world, 16384, 20, total)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    world, local_ms = 2, [812.5, 840.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, local_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value in got:
        assert total == max(local_ms)
        assert value == pytest.approx(world * 16384 * 20 / (max(local_ms) / 1e3))


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_tokens_per_s(1, 100, 10, 1000.0) == pytest.approx(1000.0)
