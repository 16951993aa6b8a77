"""The benchmark's multi-rank path on CPU: two gloo ranks, each a replica of the layer (the MoE
forward shards over tokens with no data-path exchange), the job timed by its slowest rank."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow replica
    ms = bench.max_over_ranks(local_ms, world, "cpu")
    rate = bench.whole_job_rate(world, 8192, 20, ms * 20 / 1e3)
    # replicas: every rank holds the same token count; nothing but the timing crosses ranks
    dist.barrier()
    q.put((rank, ms, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, rate in res:
        assert ms == 15.0
        assert abs(rate - 2 * 8192 / 0.015) < 1e-6 * rate


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(1, 100, 10, 2.0) == 500.0
