"""The multi-GPU path of the bench is independent replicas (one per rank, no
collective on the data path); its host side — the slowest rank's time and the
whole-job throughput — runs here as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    env = bench.dist_env()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 130.0][rank]  # rank 1 is the slower one
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        q.put((rank, env, ms, bench.job_tokens_per_s(world, 16384, 10, ms)))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_time_and_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, ms, tps in out:
        assert env == (world, rank, rank)
        assert ms == 130.0  # every rank reports the slowest rank's time
        assert tps == pytest.approx(world * 16384 * 10 / 0.130)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(42.0, 1, "cpu") == 42.0
    assert bench.job_tokens_per_s(1, 1000, 5, 500.0) == pytest.approx(10000.0)
